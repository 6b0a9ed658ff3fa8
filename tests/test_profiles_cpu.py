"""The committed ncu summaries belong to the kernel sources as they stand:
every summary under profiles/ names the hash of the sources' code (comments
left out) it was captured from,
and the recorded DRAM traffic that bench.py reports is keyed by the same
hash.  A kernel change without a new capture fails here (and bench.py would
report no traffic)."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_profile_summaries_match_the_kernel_sources():
    import bench
    sha = bench.kernel_source_sha()
    summaries = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert summaries
    for path in summaries:
        text = open(path).read()
        found = re.findall(r"sha256\[:16\] \(bench\.kernel_source_sha\): ([0-9a-f]{16})", text)
        assert found == [sha], "%s was captured from other kernel sources" % os.path.basename(path)
        assert "--clock-control none" in text, "%s: every ncu command keeps the clocks" % os.path.basename(path)


def test_recorded_traffic_is_for_the_current_kernels():
    import bench
    for kernel in ("k_decode_bcast", "k_reduce_encode"):
        t = bench.traffic_from_profiles(kernel)
        assert t is not None and t > 0, kernel


def test_the_capture_key_ignores_comments_only():
    import bench
    code = "int f(int x) {\n    return x + 1;  // one more\n}\n/* a note\n   over lines */\n"
    assert bench._code_only(code) == bench._code_only(code.replace("one more", "plus one").replace("note", "remark"))
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))
