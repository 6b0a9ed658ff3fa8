// The exact path (sm_103a): MAX / MIN for every dtype, and SUM / AVG for the
// float16, float64 and integer dtypes (gpubridge README, API table and
// supported-dtype list; "Bridge compression": MAX/MIN and integer dtypes
// stay exact).  Same reduce-bridge-broadcast shape as the codec path:
//   k_exact_reduce   island fold (ascending rank) -> payload
//   k_exact_combine  fold of the I payloads (island order), AVG, -> ranks
// Arithmetic: float16 / bfloat16 / float32 fold in float32 (payload float32
// for SUM / AVG, the dtype itself for MAX / MIN, whose result is always one
// of the inputs); float64 in float64; integers wrap modulo 2^bits for SUM.
// MAX keeps the earlier value unless a later one is strictly greater (MIN:
// strictly less).  Threads move 16-byte vectors: two per step, with every
// operand's load issued before the first fold, when the rank (payload)
// count is a compile-time 1, 2 or 4 (1 or 2); one per step otherwise.
#include <cstring>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gb_device.cuh"
#include "gb_kernels.cuh"

namespace gb {

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------- dtype traits
template <typename T> struct Ex;  // A: fold arithmetic type
template <> struct Ex<float> {
    using A = float;
    __device__ static A widen(float x) { return x; }
    __device__ static float narrow(A a) { return a; }
};
template <> struct Ex<bf16> {
    using A = float;
    __device__ static A widen(bf16 x) { return __bfloat162float(x); }
    __device__ static bf16 narrow(A a) { return __float2bfloat16_rn(a); }
};
template <> struct Ex<__half> {
    using A = float;
    __device__ static A widen(__half x) { return __half2float(x); }
    __device__ static __half narrow(A a) { return __float2half_rn(a); }
};
template <> struct Ex<double> {
    using A = double;
    __device__ static A widen(double x) { return x; }
    __device__ static double narrow(A a) { return a; }
};
template <typename I> struct ExInt {
    using A = I;
    __device__ static A widen(I x) { return x; }
    __device__ static I narrow(A a) { return a; }
};
template <> struct Ex<int8_t> : ExInt<int8_t> {};
template <> struct Ex<uint8_t> : ExInt<uint8_t> {};
template <> struct Ex<int32_t> : ExInt<int32_t> {};
template <> struct Ex<int64_t> : ExInt<int64_t> {};

template <typename A>
__device__ __forceinline__ A add_(A a, A b) {
    if constexpr (std::is_same<A, float>::value) return __fadd_rn(a, b);
    else if constexpr (std::is_same<A, double>::value) return __dadd_rn(a, b);
    else {  // integers: two's complement wrap-around
        using U = typename std::make_unsigned<A>::type;
        return (A)(U)((U)a + (U)b);
    }
}

template <int OP, typename A>
__device__ __forceinline__ A fold(A a, A b) {
    if constexpr (OP == GB_MAX) return b > a ? b : a;
    else if constexpr (OP == GB_MIN) return b < a ? b : a;
    else return add_(a, b);
}

// Payload element: float32 island sums for 16-bit floats (SUM / AVG), the
// dtype itself otherwise.
template <typename T, int OP>
using PayloadT = typename std::conditional<(OP == GB_SUM || OP == GB_AVG) && sizeof(T) == 2 &&
                                               !std::is_integral<T>::value,
                                           float, T>::type;

template <typename T, int OP>
__device__ __forceinline__ typename Ex<T>::A to_acc(PayloadT<T, OP> p) {
    if constexpr (std::is_same<PayloadT<T, OP>, float>::value && !std::is_same<T, float>::value) return p;
    else return Ex<T>::widen(p);
}
template <typename T, int OP>
__device__ __forceinline__ PayloadT<T, OP> to_payload(typename Ex<T>::A a) {
    if constexpr (std::is_same<PayloadT<T, OP>, float>::value && !std::is_same<T, float>::value) return a;
    else return Ex<T>::narrow(a);
}

// 8-bit integers: four lanes per 32-bit word with the per-byte SIMD
// intrinsics.  MAX / MIN of integers have no tie to break (equal values are
// equal bits) and __vadd4 wraps each byte modulo 256, so a word-wise fold
// gives the same bytes as the element-wise one.
template <typename T>
constexpr bool kByteSimd = sizeof(T) == 1 && std::is_integral<T>::value;

template <typename T, int OP>
__device__ __forceinline__ uint32_t fold4(uint32_t a, uint32_t b) {
    if constexpr (OP == GB_MAX) return std::is_signed<T>::value ? __vmaxs4(a, b) : __vmaxu4(a, b);
    else if constexpr (OP == GB_MIN) return std::is_signed<T>::value ? __vmins4(a, b) : __vminu4(a, b);
    else return __vadd4(a, b);
}

// 16 bytes of T per thread step.
template <typename T> struct V16 {
    static constexpr int N = 16 / sizeof(T);
    T v[N];
};

template <typename T>
__device__ __forceinline__ V16<T> load16(const T *p) {
    const uint4 u = ld_u4(p);
    V16<T> r;
    memcpy(&r, &u, 16);
    return r;
}

// --------------------------------------------------------------- kernels
// The fold of KT rank vectors (16 bytes of T each, ascending rank) into the
// payload vector out (NPO 16-byte words of P).
template <typename T, int OP, int KT, int NPO>
__device__ __forceinline__ void fold_ranks_raw(const uint4 (&raw)[KT], uint4 (&out)[NPO]) {
    using A = typename Ex<T>::A;
    using P = PayloadT<T, OP>;
    constexpr int N = V16<T>::N;
    if constexpr (kByteSimd<T>) {
        uint4 acc = raw[0];
#pragma unroll
        for (int q = 1; q < KT; ++q)
            acc = make_uint4(fold4<T, OP>(acc.x, raw[q].x), fold4<T, OP>(acc.y, raw[q].y),
                             fold4<T, OP>(acc.z, raw[q].z), fold4<T, OP>(acc.w, raw[q].w));
        out[0] = acc;
    } else {
        A s[N];
#pragma unroll
        for (int q = 0; q < KT; ++q) {
            T x[N];
            memcpy(x, &raw[q], 16);
#pragma unroll
            for (int k = 0; k < N; ++k) s[k] = q == 0 ? Ex<T>::widen(x[k]) : fold<OP>(s[k], Ex<T>::widen(x[k]));
        }
        P o[N];
#pragma unroll
        for (int k = 0; k < N; ++k) o[k] = to_payload<T, OP>(s[k]);
        memcpy(out, o, sizeof o);
    }
}

// KT > 0: every island has KT ranks.  Then a thread takes kFoldU full
// vectors per step, spaced a grid apart, and issues all KT * kFoldU rank
// loads before the first fold; the rest, and KT == 0, take the loop below.
constexpr int kFoldU = 2;

template <typename T, int OP, int KT>
__global__ void __launch_bounds__(256) k_exact_reduce(const __grid_constant__ ReduceEncodeArgs a) {
    using A = typename Ex<T>::A;
    using P = PayloadT<T, OP>;
    constexpr int N = V16<T>::N;
    const int isl = blockIdx.y;
    const int r0 = a.first[isl];
    const int K = a.first[isl + 1] - r0;
    P *out = (P *)a.payload[isl];
    const uint64_t nvec = (a.n + N - 1) / N;
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    uint64_t vi = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x + wait_prior_grid();
    if constexpr (KT > 0) {
        constexpr int NPO = (int)(sizeof(P) * N / 16);
        const uint64_t nfull = a.n / N;
        for (; vi + (kFoldU - 1) * nth < nfull; vi += kFoldU * nth) {
            uint4 raw[kFoldU][KT];
#pragma unroll
            for (int v = 0; v < kFoldU; ++v)
#pragma unroll
                for (int q = 0; q < KT; ++q) raw[v][q] = ld_u4((const T *)a.src[r0 + q] + (vi + v * nth) * N);
#pragma unroll
            for (int v = 0; v < kFoldU; ++v) {
                uint4 o[NPO];
                fold_ranks_raw<T, OP, KT, NPO>(raw[v], o);
#pragma unroll
                for (int i = 0; i < NPO; ++i) st_u4((unsigned char *)(out + (vi + v * nth) * N) + 16 * i, o[i]);
            }
        }
    }
    for (; vi < nvec; vi += nth) {
        const uint64_t j0 = vi * N;
        const int cnt = (a.n - j0) < (uint64_t)N ? (int)(a.n - j0) : N;
        if constexpr (kByteSimd<T>) {
            if (cnt == N) {
                uint4 acc = ld_u4((const T *)a.src[r0] + j0);
                for (int q = 1; q < K; ++q) {
                    const uint4 y = ld_u4((const T *)a.src[r0 + q] + j0);
                    acc = make_uint4(fold4<T, OP>(acc.x, y.x), fold4<T, OP>(acc.y, y.y), fold4<T, OP>(acc.z, y.z),
                                     fold4<T, OP>(acc.w, y.w));
                }
                st_u4(out + j0, acc);
                continue;
            }
        }
        A s[N];
        if (cnt == N) {
            const V16<T> x = load16((const T *)a.src[r0] + j0);
            if constexpr (sizeof(T) == 2 && !std::is_integral<T>::value) {
                // 16-bit floats: widening takes conversions, so the next
                // rank's load is issued before the current one is folded
                // (f16 AVG fold 20.6 -> 17.4 us on 4 x 13 MB; for 32-bit types
                // the same change measured slower)
                V16<T> y = x;
                if (K > 1) y = load16((const T *)a.src[r0 + 1] + j0);
#pragma unroll
                for (int k = 0; k < N; ++k) s[k] = Ex<T>::widen(x.v[k]);
                for (int q = 1; q < K; ++q) {
                    V16<T> nx = y;
                    if (q + 1 < K) nx = load16((const T *)a.src[r0 + q + 1] + j0);
#pragma unroll
                    for (int k = 0; k < N; ++k) s[k] = fold<OP>(s[k], Ex<T>::widen(y.v[k]));
                    y = nx;
                }
            } else {
#pragma unroll
                for (int k = 0; k < N; ++k) s[k] = Ex<T>::widen(x.v[k]);
                for (int q = 1; q < K; ++q) {
                    const V16<T> y = load16((const T *)a.src[r0 + q] + j0);
#pragma unroll
                    for (int k = 0; k < N; ++k) s[k] = fold<OP>(s[k], Ex<T>::widen(y.v[k]));
                }
            }
            P o[N];
#pragma unroll
            for (int k = 0; k < N; ++k) o[k] = to_payload<T, OP>(s[k]);
            uint4 w[sizeof(P) * N / 16];
            memcpy(w, o, sizeof o);
#pragma unroll
            for (int i = 0; i < (int)(sizeof(P) * N / 16); ++i) st_u4((unsigned char *)(out + j0) + 16 * i, w[i]);
        } else {
            for (int k = 0; k < cnt; ++k) {
                A v = Ex<T>::widen(((const T *)a.src[r0])[j0 + k]);
                for (int q = 1; q < K; ++q) v = fold<OP>(v, Ex<T>::widen(((const T *)a.src[r0 + q])[j0 + k]));
                out[j0 + k] = to_payload<T, OP>(v);
            }
        }
    }
}

// The fold of NS payload vectors (raw bits of N payload elements each, NP
// 16-byte words, island order), AVG applied, narrowed to 16 bytes of T.
template <typename T, int OP, int NS, int NP>
__device__ __forceinline__ uint4 combine_raw(const uint4 (&raw)[NS][NP], const DecodeBcastArgs &a) {
    using A = typename Ex<T>::A;
    using P = PayloadT<T, OP>;
    constexpr int N = V16<T>::N;
    if constexpr (kByteSimd<T> && OP != GB_AVG) {
        uint4 acc = raw[0][0];
#pragma unroll
        for (int q = 1; q < NS; ++q)
            acc = make_uint4(fold4<T, OP>(acc.x, raw[q][0].x), fold4<T, OP>(acc.y, raw[q][0].y),
                             fold4<T, OP>(acc.z, raw[q][0].z), fold4<T, OP>(acc.w, raw[q][0].w));
        return acc;
    } else {
        A t[N];
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            P x[N];
            memcpy(x, raw[q], sizeof x);
#pragma unroll
            for (int k = 0; k < N; ++k) {
                const A v = to_acc<T, OP>(x[k]);
                t[k] = (q == 0) ? v : fold<OP>(t[k], v);
            }
        }
        if constexpr (OP == GB_AVG) {
#pragma unroll
            for (int k = 0; k < N; ++k) {
                if constexpr (sizeof(A) == 8)
                    t[k] = __ddiv_rn(t[k], (double)a.world);
                else
                    t[k] = a.world_pow2 ? __fmul_rn(t[k], a.inv_world) : __fdiv_rn(t[k], a.world);
            }
        }
        T o[N];
#pragma unroll
        for (int k = 0; k < N; ++k) o[k] = Ex<T>::narrow(t[k]);
        uint4 w;
        memcpy(&w, o, 16);
        return w;
    }
}

// NS > 0: exactly NS payloads.  Then a thread takes kCombineU full vectors
// per step, spaced a grid apart, and issues all their payload loads before
// the first fold (the codec decode keeps as many bytes in flight per lane);
// the rest, and NS == 0, take the element-wise-capable loop below.
constexpr int kCombineU = 2;

template <typename T, int OP, int NS>
__global__ void __launch_bounds__(256) k_exact_combine(const __grid_constant__ DecodeBcastArgs a) {
    using A = typename Ex<T>::A;
    using P = PayloadT<T, OP>;
    constexpr int N = V16<T>::N;
    const int u = blockIdx.y;
    int g, r_lo, r_hi;
    uint64_t gofs, limit;
    if (a.rs) {
        g = a.group_of_rank[u];
        r_lo = u;
        r_hi = u + 1;
        gofs = a.rs_src[u];
        limit = a.rs_len[u];
    } else {
        g = u;
        r_lo = a.first[g];
        r_hi = a.first[g + 1];
        gofs = 0;
        limit = a.n;
    }
    const uint64_t nvec = (limit + N - 1) / N;
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    uint64_t vi = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x + wait_prior_grid();
    if constexpr (NS > 0) {
        constexpr int NP = (int)(sizeof(P) * N / 16);
        const uint64_t nfull = a.vec ? limit / N : 0;
        for (; vi + (kCombineU - 1) * nth < nfull; vi += kCombineU * nth) {
            uint4 raw[kCombineU][NS][NP];
#pragma unroll
            for (int v = 0; v < kCombineU; ++v)
#pragma unroll
                for (int q = 0; q < NS; ++q)
#pragma unroll
                    for (int i = 0; i < NP; ++i)
                        raw[v][q][i] = ld_u4((const unsigned char *)((const P *)a.payload[g][q] + gofs +
                                                                   (vi + v * nth) * N) + 16 * i);
#pragma unroll
            for (int v = 0; v < kCombineU; ++v) {
                const uint4 w = combine_raw<T, OP, NS, NP>(raw[v], a);
                for (int r = r_lo; r < r_hi; ++r) st_stream_u4((T *)a.dst[r] + (vi + v * nth) * N, w);
            }
        }
    }
    for (; vi < nvec; vi += nth) {
        const uint64_t l0 = vi * N;
        const int cnt = (limit - l0) < (uint64_t)N ? (int)(limit - l0) : N;
        const bool full = a.vec && cnt == N;
        if constexpr (kByteSimd<T> && OP != GB_AVG) {
            if (full) {
                uint4 acc = ld_u4((const T *)a.payload[g][0] + gofs + l0);
                for (int j = 1; j < a.n_src; ++j) {
                    const uint4 y = ld_u4((const T *)a.payload[g][j] + gofs + l0);
                    acc = make_uint4(fold4<T, OP>(acc.x, y.x), fold4<T, OP>(acc.y, y.y), fold4<T, OP>(acc.z, y.z),
                                     fold4<T, OP>(acc.w, y.w));
                }
                for (int r = r_lo; r < r_hi; ++r) st_stream_u4((T *)a.dst[r] + l0, acc);
                continue;
            }
        }
        A t[N];
        for (int j = 0; j < a.n_src; ++j) {
            const P *p = (const P *)a.payload[g][j] + gofs + l0;
            P x[N];
            if (full) {
                uint4 w[sizeof(P) * N / 16];
#pragma unroll
                for (int i = 0; i < (int)(sizeof(P) * N / 16); ++i) w[i] = ld_u4((const unsigned char *)p + 16 * i);
                memcpy(x, w, sizeof x);
            } else {
                for (int k = 0; k < cnt; ++k) x[k] = p[k];
            }
#pragma unroll
            for (int k = 0; k < N; ++k) {
                const A v = to_acc<T, OP>(x[k]);
                t[k] = (j == 0) ? v : fold<OP>(t[k], v);
            }
        }
        if constexpr (OP == GB_AVG) {
#pragma unroll
            for (int k = 0; k < N; ++k) {
                if constexpr (sizeof(A) == 8)
                    t[k] = __ddiv_rn(t[k], (double)a.world);
                else
                    t[k] = a.world_pow2 ? __fmul_rn(t[k], a.inv_world) : __fdiv_rn(t[k], a.world);
            }
        }
        T o[N];
#pragma unroll
        for (int k = 0; k < N; ++k) o[k] = Ex<T>::narrow(t[k]);
        for (int r = r_lo; r < r_hi; ++r) {
            T *d = (T *)a.dst[r] + l0;
            if (full) {
                uint4 w;
                memcpy(&w, o, 16);
                st_stream_u4(d, w);
            } else {
                for (int k = 0; k < cnt; ++k) d[k] = o[k];
            }
        }
    }
}

// ------------------------------------------------------------------ launch
template <auto Kern, typename Args>
static cudaError_t launch_vec(uint64_t vec_items, unsigned units, const Args &a, cudaStream_t s) {
    // launch_grid sizes in units of 8 warps per block: one vector per thread
    return launch_grid<Kern>((vec_items + 31) / 32, units, a, s);
}

template <typename T, int OP>
static cudaError_t launch_pair(bool combine, const void *args, cudaStream_t s) {
    constexpr int N = V16<T>::N;
    if (!combine) {
        const ReduceEncodeArgs &a = *(const ReduceEncodeArgs *)args;
        int K = a.first[1] - a.first[0];
        for (int i = 1; i < a.n_islands; ++i)
            if (a.first[i + 1] - a.first[i] != K) K = 0;
        const uint64_t vecs = (a.n + N - 1) / N, per_u = (vecs + kFoldU - 1) / kFoldU;
        switch (K) {
        case 1: return launch_vec<k_exact_reduce<T, OP, 1>>(per_u, (unsigned)a.n_islands, a, s);
        case 2: return launch_vec<k_exact_reduce<T, OP, 2>>(per_u, (unsigned)a.n_islands, a, s);
        case 4: return launch_vec<k_exact_reduce<T, OP, 4>>(per_u, (unsigned)a.n_islands, a, s);
        default: return launch_vec<k_exact_reduce<T, OP, 0>>(vecs, (unsigned)a.n_islands, a, s);
        }
    }
    const DecodeBcastArgs &a = *(const DecodeBcastArgs *)args;
    const unsigned units = a.rs ? (unsigned)a.first[a.n_groups] : (unsigned)a.n_groups;
    uint64_t limit = a.n;
    if (a.rs) {  // the longest unit
        limit = 0;
        for (unsigned u = 0; u < units; ++u)
            if (a.rs_len[u] > limit) limit = a.rs_len[u];
    }
    // one thread per kCombineU vectors when the payload count is unrolled
    const uint64_t vecs = (limit + N - 1) / N;
    switch (a.n_src) {
    case 1: return launch_vec<k_exact_combine<T, OP, 1>>((vecs + kCombineU - 1) / kCombineU, units, a, s);
    case 2: return launch_vec<k_exact_combine<T, OP, 2>>((vecs + kCombineU - 1) / kCombineU, units, a, s);
    default: return launch_vec<k_exact_combine<T, OP, 0>>(vecs, units, a, s);
    }
}

template <typename T>
static cudaError_t by_op(int op, bool combine, const void *args, cudaStream_t s) {
    switch (op) {
    case GB_SUM: return launch_pair<T, GB_SUM>(combine, args, s);
    case GB_MAX: return launch_pair<T, GB_MAX>(combine, args, s);
    case GB_MIN: return launch_pair<T, GB_MIN>(combine, args, s);
    case GB_AVG:
        if constexpr (std::is_integral<T>::value) return cudaErrorInvalidValue;
        else return launch_pair<T, GB_AVG>(combine, args, s);
    default: return cudaErrorInvalidValue;
    }
}

static cudaError_t by_dtype(int dtype, int op, bool combine, const void *args, cudaStream_t s) {
    switch (dtype) {
    case GB_F32: return by_op<float>(op, combine, args, s);
    case GB_BF16: return by_op<bf16>(op, combine, args, s);
    case GB_F16: return by_op<__half>(op, combine, args, s);
    case GB_F64: return by_op<double>(op, combine, args, s);
    case GB_I8: return by_op<int8_t>(op, combine, args, s);
    case GB_U8: return by_op<uint8_t>(op, combine, args, s);
    case GB_I32: return by_op<int32_t>(op, combine, args, s);
    case GB_I64: return by_op<int64_t>(op, combine, args, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_exact_reduce(const ReduceEncodeArgs &a, int dtype, int op, cudaStream_t s) {
    return by_dtype(dtype, op, false, &a, s);
}

cudaError_t launch_exact_combine(const DecodeBcastArgs &a, int dtype, int op, cudaStream_t s) {
    return by_dtype(dtype, op, true, &a, s);
}

size_t exact_payload_elem_bytes(int dtype, int op) {
    const bool small_float = dtype == GB_BF16 || dtype == GB_F16;
    if (small_float && (op == GB_SUM || op == GB_AVG)) return 4;
    switch (dtype) {
    case GB_F32: case GB_I32: return 4;
    case GB_BF16: case GB_F16: return 2;
    case GB_F64: case GB_I64: return 8;
    default: return 1;
    }
}

}  // namespace gb
