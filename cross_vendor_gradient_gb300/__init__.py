"""GB300-native reduce-bridge-broadcast gradient all_reduce (libgb).

The C ABI is ``include/gb.h``; ``binding`` mirrors it one function per entry
point, and ``api`` offers the same calls on torch tensors.
"""
from .api import (CODECS, OPS, Context, GbError, bucket_plan, island_payload_bytes, kernel_launch_count,
                  payload_bytes, payload_scales_offset)

__all__ = ["CODECS", "OPS", "Context", "GbError", "bucket_plan", "island_payload_bytes", "kernel_launch_count",
           "payload_bytes", "payload_scales_offset"]
