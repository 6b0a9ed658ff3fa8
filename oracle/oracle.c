/*
 * Oracle for the reduce-bridge-broadcast gradient all_reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded CPU
 * statement of what the collectives compute.  It shares no code, header,
 * table or constant with the CUDA library and must never be called from the
 * product path: only the tests, the smoke check and the benchmark's CPU
 * baseline load it.
 *
 * Sources (gpubridge README, the project page this library follows):
 *   - "all_reduce uses reduce-bridge-broadcast": reduce within each island
 *     onto its leader, leaders exchange the island sums over the bridge, each
 *     leader broadcasts the total to its island.
 *   - Island / leader paragraph: an island is every rank of one vendor, its
 *     leader is its lowest global rank.
 *   - API table, all_reduce row: SUM or AVG; AVG is the SUM divided by the
 *     world size, the same way on every rank.
 *   - API table, all_gather_into_tensor / reduce_scatter_tensor / broadcast
 *     rows.
 *   - "Bridge compression": leaders quantize the island sum before the bridge
 *     (bf16, or OCP E4M3 with a power-of-two scale per 256 values), exchange
 *     the payloads, dequantize and add them in float32; every rank ends with
 *     the same bits; broadcast and all_gather stay exact.
 *   - "If the cluster has only one vendor there is no bridge": one island is
 *     a native collective, so no codec is applied.
 *
 * Readings where the page is silent (each is listed in the design notes):
 *   - island sums: float32, ascending global rank order; bridge total:
 *     float32, ascending island order, every island's term decoded (its own
 *     included) so that every island ends with the same bits;
 *   - the block scale is 2^k with k the smallest integer such that
 *     absmax * 2^-k <= the format's largest finite value, clamped to
 *     k >= -126; an all-zero block has k = 0;
 *   - codes are rounded to nearest, ties to even, and saturate to the largest
 *     finite value;
 *   - scales are stored as float32 values, one per block; blocks start at
 *     element 0 of the buffer and the last one may be short;
 *   - E5M2 uses the same scale rule as E4M3;
 *   - reduce_scatter compresses the full island sum, then takes slice r.
 *
 * Floating point: every float operation below is a single IEEE binary32
 * operation rounded to nearest even (the file is built without fast-math and
 * without contraction, and FLT_EVAL_METHOD must be 0).  Encodings are
 * computed from the values' definitions in double precision, where every
 * intermediate used is exact.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

/* identifiers used by the Python wrapper */
enum { ORC_DT_F32 = 0, ORC_DT_BF16 = 1 };
enum { ORC_OP_SUM = 0, ORC_OP_AVG = 1 };
enum { ORC_CODEC_NONE = 0, ORC_CODEC_BF16 = 1, ORC_CODEC_E4M3 = 2, ORC_CODEC_E5M2 = 3 };

/* ------------------------------------------------------------------------ */
/* bfloat16: the top 16 bits of an IEEE binary32                             */
/* ------------------------------------------------------------------------ */

float orc_bf16_to_f32(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float x;
    memcpy(&x, &bits, sizeof x);
    return x;
}

/* Round a binary32 to bfloat16, to nearest, ties to even.  Adding
 * 0x7FFF + (bit 16) to the pattern and dropping the low half rounds the
 * magnitude to nearest with ties going to an even bit 16; a carry into the
 * exponent is the correct next binade, and a carry out of the largest finite
 * binade gives infinity, as IEEE rounding does.  NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    if ((bits & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((bits >> 16) | 0x0040u);
    uint32_t lsb = (bits >> 16) & 1u;
    bits += 0x7FFFu + lsb;
    return (uint16_t)(bits >> 16);
}

/* ------------------------------------------------------------------------ */
/* OCP 8-bit floating point (OFP8): E4M3 and E5M2                            */
/*   E4M3: 4 exponent bits, bias 7, 3 mantissa bits, no infinities,          */
/*         S.1111.111 is NaN, largest finite 448 = 1.75 * 2^8.               */
/*   E5M2: 5 exponent bits, bias 15, 2 mantissa bits, IEEE-style inf/NaN,    */
/*         largest finite 57344 = 1.75 * 2^15.                               */
/* ------------------------------------------------------------------------ */

static int fp8_exp_bits(int fmt) { return fmt == ORC_CODEC_E4M3 ? 4 : 5; }
static int fp8_man_bits(int fmt) { return fmt == ORC_CODEC_E4M3 ? 3 : 2; }
static int fp8_bias(int fmt) { return fmt == ORC_CODEC_E4M3 ? 7 : 15; }

double orc_fp8_max(int fmt) { return fmt == ORC_CODEC_E4M3 ? 448.0 : 57344.0; }

/* Value of an 8-bit code, from the field definitions. */
double orc_fp8_value(uint8_t code, int fmt)
{
    int man = fp8_man_bits(fmt);
    int emax_field = (1 << fp8_exp_bits(fmt)) - 1;
    int s = code >> 7;
    int e = (code >> man) & emax_field;
    int m = code & ((1 << man) - 1);
    double v;
    if (fmt == ORC_CODEC_E4M3 && e == emax_field && m == (1 << man) - 1)
        return NAN;
    if (fmt == ORC_CODEC_E5M2 && e == emax_field)
        v = (m == 0) ? INFINITY : NAN;
    else if (e == 0)
        v = ldexp((double)m, 1 - fp8_bias(fmt) - man);            /* subnormal */
    else
        v = ldexp((double)((1 << man) + m), e - fp8_bias(fmt) - man); /* normal */
    return s ? -v : v;
}

/* Code of an exact value v that lies on the format's finite grid, v >= 0. */
static uint8_t fp8_code_of_grid_value(double v, int fmt)
{
    int man = fp8_man_bits(fmt);
    int emin = 1 - fp8_bias(fmt); /* exponent of the smallest normal */
    if (v == 0.0)
        return 0;
    int e2;
    (void)frexp(v, &e2); /* v = f * 2^e2, f in [0.5, 1) */
    int ex = e2 - 1;     /* v in [2^ex, 2^(ex+1)) */
    if (ex < emin) {
        int m = (int)ldexp(v, man - emin);
        return (uint8_t)m;
    }
    int m = (int)(ldexp(v, man - ex) - (double)(1 << man));
    return (uint8_t)(((ex + fp8_bias(fmt)) << man) | m);
}

/* Round y to the 8-bit grid: to nearest, ties to even, values beyond the
 * largest finite magnitude (and infinities) saturate to it.  NaN gives the
 * format's NaN code. */
uint8_t orc_fp8_encode(double y, int fmt)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    int man = fp8_man_bits(fmt);
    int emin = 1 - fp8_bias(fmt);
    double maxv = orc_fp8_max(fmt);
    if (isnan(y))
        return (uint8_t)(sign | 0x7F);
    double a = fabs(y);
    if (a >= maxv)
        return (uint8_t)(sign | fp8_code_of_grid_value(maxv, fmt));
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);
    int ex = e2 - 1;            /* binade of a */
    if (ex < emin)
        ex = emin;              /* subnormals share the smallest normal's spacing */
    double quantum = ldexp(1.0, ex - man);
    double q = a / quantum;     /* exact: division by a power of two */
    double r = nearbyint(q);    /* default rounding mode: half to even */
    double v = r * quantum;     /* on the grid, <= maxv because maxv is on it */
    return (uint8_t)(sign | fp8_code_of_grid_value(v, fmt));
}

/* The same rounding by exhaustive search over every finite code: the nearest
 * value, ties to the even code.  Slow; kept as an independent check. */
uint8_t orc_fp8_encode_bruteforce(double y, int fmt)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    if (isnan(y))
        return (uint8_t)(sign | 0x7F);
    int best = -1;
    double best_d = 0.0;
    for (int c = 0; c < 128; ++c) {
        double v = orc_fp8_value((uint8_t)c, fmt);
        if (!isfinite(v))
            continue;
        double d = fabs(v - a);
        if (a > orc_fp8_max(fmt))
            d = orc_fp8_max(fmt) - v; /* saturate: the largest finite code wins */
        if (best < 0 || d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Block scale exponent: the smallest k with absmax * 2^-k <= largest finite
 * value M, so that the block's largest magnitude lands in (M/2, M]; clamped
 * to k >= -126 so that 2^k and 2^-k are normal binary32 numbers; 0 for an
 * all-zero block.  With absmax = f * 2^e, f in [0.5, 1), and M = 0.875 * 2^E
 * (E = 9 for E4M3, 16 for E5M2): k = e - E when f <= 0.875, else e - E + 1. */
int orc_block_scale_exponent(float absmax, int fmt)
{
    if (absmax == 0.0f)
        return 0;
    int E = (fmt == ORC_CODEC_E4M3) ? 9 : 16;
    int e;
    double f = frexp((double)absmax, &e);
    int k = (f <= 0.875) ? e - E : e - E + 1;
    if (k < -126)
        k = -126;
    return k;
}

/* ------------------------------------------------------------------------ */
/* Collective steps                                                         */
/* ------------------------------------------------------------------------ */

static float load_elem(const void *buf, int dtype, size_t j)
{
    if (dtype == ORC_DT_F32)
        return ((const float *)buf)[j];
    return orc_bf16_to_f32(((const uint16_t *)buf)[j]);
}

static void store_elem(void *buf, int dtype, size_t j, float v)
{
    if (dtype == ORC_DT_F32)
        ((float *)buf)[j] = v;
    else
        ((uint16_t *)buf)[j] = orc_f32_to_bf16(v);
}

/* Island reduce onto the leader: s[j] = ((x0[j] + x1[j]) + ...) + x_{K-1}[j]
 * in float32, ranks in ascending global order, each input widened exactly. */
void orc_island_sum(int K, const void *const *ranks, int dtype, size_t n, float *s)
{
    for (size_t j = 0; j < n; ++j) {
        float acc = load_elem(ranks[0], dtype, j);
        for (int q = 1; q < K; ++q)
            acc = acc + load_elem(ranks[q], dtype, j);
        s[j] = acc;
    }
}

size_t orc_n_blocks(size_t n, int block) { return (n + (size_t)block - 1) / (size_t)block; }

/* Bridge encode of an island sum.
 *   none: codes = the float32 sums (float array of n);
 *   bf16: codes = bf16 patterns (uint16 array of n);
 *   e4m3/e5m2: codes = uint8 array of n, scales = float array of
 *              ceil(n / block), scale b = 2^k_b. */
void orc_encode(const float *s, size_t n, int codec, int block, void *codes, float *scales)
{
    if (codec == ORC_CODEC_NONE) {
        for (size_t j = 0; j < n; ++j)
            ((float *)codes)[j] = s[j];
        return;
    }
    if (codec == ORC_CODEC_BF16) {
        for (size_t j = 0; j < n; ++j)
            ((uint16_t *)codes)[j] = orc_f32_to_bf16(s[j]);
        return;
    }
    size_t nb = orc_n_blocks(n, block);
    for (size_t b = 0; b < nb; ++b) {
        size_t lo = b * (size_t)block;
        size_t hi = lo + (size_t)block < n ? lo + (size_t)block : n;
        float m = 0.0f;
        for (size_t j = lo; j < hi; ++j)
            if (fabsf(s[j]) > m)
                m = fabsf(s[j]);
        int k = orc_block_scale_exponent(m, codec);
        for (size_t j = lo; j < hi; ++j)
            ((uint8_t *)codes)[j] = orc_fp8_encode(ldexp((double)s[j], -k), codec);
        scales[b] = (float)ldexp(1.0, k);
    }
}

/* Decoded value of element j of a payload (exact in float32). */
static float decode_elem(const void *codes, const float *scales, size_t j, int codec, int block)
{
    if (codec == ORC_CODEC_NONE)
        return ((const float *)codes)[j];
    if (codec == ORC_CODEC_BF16)
        return orc_bf16_to_f32(((const uint16_t *)codes)[j]);
    double v = orc_fp8_value(((const uint8_t *)codes)[j], codec) * (double)scales[j / (size_t)block];
    return (float)v;
}

void orc_decode(const void *codes, const float *scales, size_t n, int codec, int block, float *out)
{
    for (size_t j = 0; j < n; ++j)
        out[j] = decode_elem(codes, scales, j, codec, block);
}

/* Bridge total: t = dec(p_0); t = t + dec(p_i) for i = 1..I-1 (float32);
 * AVG divides once by the world size W (float32 division). */
void orc_bridge_total(int I, const void *const *codes, const float *const *scales, size_t n,
                      int codec, int block, int op, int W, float *t)
{
    for (size_t j = 0; j < n; ++j) {
        float acc = decode_elem(codes[0], scales[0], j, codec, block);
        for (int i = 1; i < I; ++i)
            acc = acc + decode_elem(codes[i], scales[i], j, codec, block);
        if (op == ORC_OP_AVG)
            acc = acc / (float)W;
        t[j] = acc;
    }
}

static size_t code_bytes(int codec)
{
    switch (codec) {
    case ORC_CODEC_NONE: return 4;
    case ORC_CODEC_BF16: return 2;
    default: return 1;
    }
}

/* Reduce-bridge-broadcast total over W = sum(island_sizes) ranks, islands
 * contiguous in global rank order.  t receives the float32 total (after the
 * AVG division).  If island_sums / codes_out / scales_out are non-NULL they
 * receive the intermediate island sums [I][n], codes [I][n * code bytes] and
 * scales [I][ceil(n / block)].  With one island there is no bridge: the codec
 * is not applied. */
int orc_rbb_total(int I, const int *island_sizes, const void *const *ranks, size_t n, int dtype,
                  int op, int codec, int block, float *t, float *island_sums, void *codes_out,
                  float *scales_out)
{
    int W = 0;
    for (int i = 0; i < I; ++i)
        W += island_sizes[i];
    if (I == 1)
        codec = ORC_CODEC_NONE;
    size_t nb = (codec == ORC_CODEC_E4M3 || codec == ORC_CODEC_E5M2) ? orc_n_blocks(n, block) : 0;
    size_t cb = code_bytes(codec);
    float *s = malloc((n ? n : 1) * sizeof(float) * (size_t)I);
    uint8_t *codes = malloc((n ? n : 1) * cb * (size_t)I);
    float *scales = malloc((nb ? nb : 1) * sizeof(float) * (size_t)I);
    const void **cptr = malloc(sizeof(void *) * (size_t)I);
    const float **sptr = malloc(sizeof(float *) * (size_t)I);
    if (!s || !codes || !scales || !cptr || !sptr) {
        free(s); free(codes); free(scales); free(cptr); free(sptr);
        return -1;
    }
    int first = 0;
    for (int i = 0; i < I; ++i) {
        /* step 1: island reduce onto the leader */
        orc_island_sum(island_sizes[i], ranks + first, dtype, n, s + (size_t)i * n);
        /* step 2: the leader encodes its island sum for the bridge */
        orc_encode(s + (size_t)i * n, n, codec, block, codes + (size_t)i * n * cb, scales + (size_t)i * nb);
        cptr[i] = codes + (size_t)i * n * cb;
        sptr[i] = scales + (size_t)i * nb;
        first += island_sizes[i];
    }
    /* steps 3-4: every leader holds all I payloads after the exchange and
     * decodes and adds them in island order (the same bits on every leader) */
    orc_bridge_total(I, cptr, sptr, n, codec, block, op, W, t);
    if (island_sums)
        memcpy(island_sums, s, n * sizeof(float) * (size_t)I);
    if (codes_out)
        memcpy(codes_out, codes, n * cb * (size_t)I);
    if (scales_out && nb)
        memcpy(scales_out, scales, nb * sizeof(float) * (size_t)I);
    free(s); free(codes); free(scales); free(cptr); free(sptr);
    return 0;
}

/* all_reduce: every rank buffer receives the total rounded to its dtype.
 * Inputs and outputs are separate arrays here (the library works in place). */
int orc_all_reduce(int I, const int *island_sizes, const void *const *in, void *const *out,
                   size_t n, int dtype, int op, int codec, int block)
{
    int W = 0;
    for (int i = 0; i < I; ++i)
        W += island_sizes[i];
    float *t = malloc((n ? n : 1) * sizeof(float));
    if (!t)
        return -1;
    if (orc_rbb_total(I, island_sizes, in, n, dtype, op, codec, block, t, NULL, NULL, NULL)) {
        free(t);
        return -1;
    }
    /* step 5: the leaders broadcast the total to their islands */
    for (int r = 0; r < W; ++r)
        for (size_t j = 0; j < n; ++j)
            store_elem(out[r], dtype, j, t[j]);
    free(t);
    return 0;
}

/* reduce_scatter: rank r receives elements [r*n/W, (r+1)*n/W) of the total;
 * n must be a multiple of W. */
int orc_reduce_scatter(int I, const int *island_sizes, const void *const *in, void *const *out,
                       size_t n, int dtype, int op, int codec, int block)
{
    int W = 0;
    for (int i = 0; i < I; ++i)
        W += island_sizes[i];
    if (n % (size_t)W)
        return -2;
    size_t m = n / (size_t)W;
    float *t = malloc((n ? n : 1) * sizeof(float));
    if (!t)
        return -1;
    if (orc_rbb_total(I, island_sizes, in, n, dtype, op, codec, block, t, NULL, NULL, NULL)) {
        free(t);
        return -1;
    }
    for (int r = 0; r < W; ++r)
        for (size_t j = 0; j < m; ++j)
            store_elem(out[r], dtype, j, t[(size_t)r * m + j]);
    free(t);
    return 0;
}

/* all_gather: out_r = in_0 | in_1 | ... | in_{W-1} for every r (bytes). */
void orc_all_gather(int W, const void *const *in, void *const *out, size_t bytes_per_rank)
{
    for (int r = 0; r < W; ++r)
        for (int q = 0; q < W; ++q)
            memcpy((uint8_t *)out[r] + (size_t)q * bytes_per_rank, in[q], bytes_per_rank);
}

/* broadcast: every rank buffer receives rank src's bytes. */
void orc_broadcast(int W, const void *const *in, void *const *out, size_t bytes, int src)
{
    for (int r = 0; r < W; ++r)
        memcpy(out[r], in[src], bytes);
}

/* Gradient bucket plan: walk the tensors in the order given and append each
 * to the open bucket unless the bucket already holds something and the
 * tensor would take it past cap_bytes; then close it and open a new one.  A
 * tensor larger than the cap therefore sits alone.  Tensors are packed with
 * no gap; a bucket's element count is then rounded up to a multiple of
 * pad_elems (pad_elems <= 1: no rounding).  Returns the bucket count, or -1
 * if more than max_buckets would be needed. */
int orc_bucket_plan(const size_t *numel, int n_tensors, size_t elem_bytes, size_t cap_bytes,
                    size_t pad_elems, int *bucket_of, size_t *offset, size_t *bucket_numel,
                    int max_buckets)
{
    int nbk = 0;
    size_t cur = 0; /* elements in the open bucket */
    for (int t = 0; t < n_tensors; ++t) {
        if (nbk == 0 || (cur > 0 && (cur + numel[t]) * elem_bytes > cap_bytes)) {
            if (nbk > 0)
                bucket_numel[nbk - 1] = cur;
            if (nbk == max_buckets)
                return -1;
            ++nbk;
            cur = 0;
        }
        bucket_of[t] = nbk - 1;
        offset[t] = cur;
        cur += numel[t];
    }
    if (nbk > 0)
        bucket_numel[nbk - 1] = cur;
    if (pad_elems > 1)
        for (int b = 0; b < nbk; ++b)
            bucket_numel[b] = (bucket_numel[b] + pad_elems - 1) / pad_elems * pad_elems;
    return nbk;
}

/* Array forms of the conversions, for the exhaustive conversion checks. */
void orc_fp8_encode_f32_array(const float *y, size_t n, int fmt, uint8_t *out)
{
    for (size_t j = 0; j < n; ++j)
        out[j] = orc_fp8_encode((double)y[j], fmt);
}

void orc_f32_to_bf16_array(const float *x, size_t n, uint16_t *out)
{
    for (size_t j = 0; j < n; ++j)
        out[j] = orc_f32_to_bf16(x[j]);
}

/* ------------------------------------------------------------------------ */
/* Error feedback (gpubridge README, "Bridge compression": each bridge      */
/* member keeps an error-feedback residual per buffer, so rounding error    */
/* carries into the next step instead of accumulating).                      */
/* Reading: the leader encodes s' = s + r (float32) and keeps                */
/* r <- s' - dec(enc(s')) (float32) for the next call on the same buffer.    */
/* ------------------------------------------------------------------------ */

void orc_encode_ef(const float *s, size_t n, int codec, int block, float *residual, void *codes,
                   float *scales)
{
    float *sp = calloc(n ? n : 1, sizeof(float));
    float *dec = calloc(n ? n : 1, sizeof(float));
    if (!sp || !dec) {
        free(sp);
        free(dec);
        return;
    }
    for (size_t j = 0; j < n; ++j)
        sp[j] = s[j] + residual[j];
    orc_encode(sp, n, codec, block, codes, scales);
    orc_decode(codes, scales, n, codec, block, dec);
    for (size_t j = 0; j < n; ++j)
        residual[j] = sp[j] - dec[j];
    free(sp);
    free(dec);
}

/* all_reduce with error feedback: residuals[i] (n floats, in/out) belongs to
 * island i's leader.  With one island there is no bridge and the residuals
 * are left as they are. */
int orc_all_reduce_ef(int I, const int *island_sizes, const void *const *in, void *const *out, size_t n,
                      int dtype, int op, int codec, int block, float *const *residuals)
{
    int W = 0;
    for (int i = 0; i < I; ++i)
        W += island_sizes[i];
    if (I == 1)
        return orc_all_reduce(I, island_sizes, in, out, n, dtype, op, codec, block);
    size_t nb = (codec == ORC_CODEC_E4M3 || codec == ORC_CODEC_E5M2) ? orc_n_blocks(n, block) : 0;
    size_t cb = code_bytes(codec);
    float *s = malloc((n ? n : 1) * sizeof(float));
    uint8_t *codes = malloc((n ? n : 1) * cb * (size_t)I);
    float *scales = malloc((nb ? nb : 1) * sizeof(float) * (size_t)I);
    float *t = malloc((n ? n : 1) * sizeof(float));
    const void **cptr = malloc(sizeof(void *) * (size_t)I);
    const float **sptr = malloc(sizeof(float *) * (size_t)I);
    if (!s || !codes || !scales || !t || !cptr || !sptr) {
        free(s); free(codes); free(scales); free(t); free(cptr); free(sptr);
        return -1;
    }
    int first = 0;
    for (int i = 0; i < I; ++i) {
        orc_island_sum(island_sizes[i], in + first, dtype, n, s);
        orc_encode_ef(s, n, codec, block, residuals[i], codes + (size_t)i * n * cb, scales + (size_t)i * nb);
        cptr[i] = codes + (size_t)i * n * cb;
        sptr[i] = scales + (size_t)i * nb;
        first += island_sizes[i];
    }
    orc_bridge_total(I, cptr, sptr, n, codec, block, op, W, t);
    for (int r = 0; r < W; ++r)
        for (size_t j = 0; j < n; ++j)
            store_elem(out[r], dtype, j, t[j]);
    free(s); free(codes); free(scales); free(t); free(cptr); free(sptr);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Exact path: MAX / MIN, and the float16, float64 and integer dtypes        */
/* (gpubridge README, API table: SUM, AVG, MAX, MIN; supported dtypes        */
/* float16, bfloat16, float32, float64, int8, uint8, int32, int64; "Bridge   */
/* compression": MAX/MIN and integer dtypes stay exact).                     */
/* Readings: integer SUM wraps modulo 2^bits (two's complement); float16    */
/* and bfloat16 accumulate in float32 and round once; float64 in float64;   */
/* MAX keeps the earlier value unless a later one is strictly greater (MIN: */
/* strictly less), so among equal values (+0 / -0) the lower rank's wins.   */
/* ------------------------------------------------------------------------ */

enum { ORC_DT_F16 = 2, ORC_DT_F64 = 3, ORC_DT_I8 = 4, ORC_DT_U8 = 5, ORC_DT_I32 = 6, ORC_DT_I64 = 7 };
enum { ORC_OP_MAX = 2, ORC_OP_MIN = 3 };

/* IEEE binary16 value of a pattern (exact in float). */
float orc_f16_to_f32(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp((double)(1024 + m), e - 25);
    return (float)(s ? -v : v);
}

/* Round a float to binary16, to nearest, ties to even; beyond the largest
 * finite value (65504) the IEEE result is an infinity. */
uint16_t orc_f32_to_f16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00);
    double a = fabs((double)x);
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);
    int ex = e2 - 1;
    if (ex < -14)
        ex = -14;                       /* subnormals share 2^-24 spacing */
    double q = ldexp(1.0, ex - 10);
    double v = nearbyint(a / q) * q;    /* exact quotient, half to even */
    if (v >= 65520.0)                   /* rounds past 65504: infinity */
        return (uint16_t)(sign | 0x7C00);
    if (v == 0.0)
        return sign;
    (void)frexp(v, &e2);
    int ev = e2 - 1;
    if (ev < -14)
        return (uint16_t)(sign | (int)ldexp(v, 24));
    return (uint16_t)(sign | ((ev + 15) << 10) | ((int)ldexp(v, 10 - ev) - 1024));
}

static int is_float_dt(int dt) { return dt == ORC_DT_F32 || dt == ORC_DT_BF16 || dt == ORC_DT_F16 || dt == ORC_DT_F64; }

size_t orc_dtype_bytes(int dt)
{
    switch (dt) {
    case ORC_DT_F32: case ORC_DT_I32: return 4;
    case ORC_DT_BF16: case ORC_DT_F16: return 2;
    case ORC_DT_F64: case ORC_DT_I64: return 8;
    default: return 1;
    }
}

/* One element as the accumulator value: float widening for the floats
 * (float64 stays double), the two's complement integer for the integers. */
typedef struct { double f; int64_t i; } acc_t;

static acc_t load_acc(const void *buf, int dt, size_t j)
{
    acc_t a = {0.0, 0};
    switch (dt) {
    case ORC_DT_F32: a.f = ((const float *)buf)[j]; break;
    case ORC_DT_BF16: a.f = orc_bf16_to_f32(((const uint16_t *)buf)[j]); break;
    case ORC_DT_F16: a.f = orc_f16_to_f32(((const uint16_t *)buf)[j]); break;
    case ORC_DT_F64: a.f = ((const double *)buf)[j]; break;
    case ORC_DT_I8: a.i = ((const int8_t *)buf)[j]; break;
    case ORC_DT_U8: a.i = ((const uint8_t *)buf)[j]; break;
    case ORC_DT_I32: a.i = ((const int32_t *)buf)[j]; break;
    case ORC_DT_I64: a.i = ((const int64_t *)buf)[j]; break;
    }
    return a;
}

/* a (op) b in the dtype's accumulator arithmetic. */
static acc_t combine(acc_t a, acc_t b, int dt, int op)
{
    acc_t r = a;
    if (is_float_dt(dt)) {
        if (op == ORC_OP_MAX) {
            if (b.f > a.f) r = b;
        } else if (op == ORC_OP_MIN) {
            if (b.f < a.f) r = b;
        } else if (dt == ORC_DT_F64) {
            r.f = a.f + b.f;                       /* binary64 */
        } else {
            r.f = (double)((float)a.f + (float)b.f); /* binary32 */
        }
    } else {
        if (op == ORC_OP_MAX) {
            if (b.i > a.i) r = b;
        } else if (op == ORC_OP_MIN) {
            if (b.i < a.i) r = b;
        } else {
            r.i = (int64_t)((uint64_t)a.i + (uint64_t)b.i); /* wraps; truncated on store */
        }
    }
    return r;
}

static void store_acc(void *buf, int dt, size_t j, acc_t a)
{
    switch (dt) {
    case ORC_DT_F32: ((float *)buf)[j] = (float)a.f; break;
    case ORC_DT_BF16: ((uint16_t *)buf)[j] = orc_f32_to_bf16((float)a.f); break;
    case ORC_DT_F16: ((uint16_t *)buf)[j] = orc_f32_to_f16((float)a.f); break;
    case ORC_DT_F64: ((double *)buf)[j] = a.f; break;
    case ORC_DT_I8: ((int8_t *)buf)[j] = (int8_t)(uint8_t)(uint64_t)a.i; break;
    case ORC_DT_U8: ((uint8_t *)buf)[j] = (uint8_t)(uint64_t)a.i; break;
    case ORC_DT_I32: ((int32_t *)buf)[j] = (int32_t)(uint32_t)(uint64_t)a.i; break;
    case ORC_DT_I64: ((int64_t *)buf)[j] = a.i; break;
    }
}

/* Exact reduce-bridge-broadcast total of element j: island folds in rank
 * order, then the fold over islands in island order, then AVG's division
 * (float32 for the 16- and 32-bit floats, float64 for float64). */
static acc_t exact_total(int I, const int *island_sizes, const void *const *in, int dt, int op, size_t j)
{
    int W = 0;
    for (int i = 0; i < I; ++i)
        W += island_sizes[i];
    acc_t t = {0.0, 0};
    int first = 0;
    for (int i = 0; i < I; ++i) {
        acc_t s = load_acc(in[first], dt, j);
        for (int q = 1; q < island_sizes[i]; ++q)
            s = combine(s, load_acc(in[first + q], dt, j), dt, op == ORC_OP_AVG ? ORC_OP_SUM : op);
        t = (i == 0) ? s : combine(t, s, dt, op == ORC_OP_AVG ? ORC_OP_SUM : op);
        first += island_sizes[i];
    }
    if (op == ORC_OP_AVG) {
        if (dt == ORC_DT_F64)
            t.f = t.f / (double)W;
        else
            t.f = (double)((float)t.f / (float)W);
    }
    return t;
}

int orc_all_reduce_exact(int I, const int *island_sizes, const void *const *in, void *const *out, size_t n,
                         int dtype, int op)
{
    int W = 0;
    for (int i = 0; i < I; ++i)
        W += island_sizes[i];
    if (op == ORC_OP_AVG && !is_float_dt(dtype))
        return -2;
    for (size_t j = 0; j < n; ++j) {
        acc_t t = exact_total(I, island_sizes, in, dtype, op, j);
        for (int r = 0; r < W; ++r)
            store_acc(out[r], dtype, j, t);
    }
    return 0;
}

int orc_reduce_scatter_exact(int I, const int *island_sizes, const void *const *in, void *const *out,
                             size_t n, int dtype, int op)
{
    int W = 0;
    for (int i = 0; i < I; ++i)
        W += island_sizes[i];
    if (n % (size_t)W || (op == ORC_OP_AVG && !is_float_dt(dtype)))
        return -2;
    size_t m = n / (size_t)W;
    for (int r = 0; r < W; ++r)
        for (size_t j = 0; j < m; ++j)
            store_acc(out[r], dtype, j, exact_total(I, island_sizes, in, dtype, op, (size_t)r * m + j));
    return 0;
}

void orc_f32_to_f16_array(const float *x, size_t n, uint16_t *out)
{
    for (size_t j = 0; j < n; ++j)
        out[j] = orc_f32_to_f16(x[j]);
}

/* ------------------------------------------------------------------------ */
/* sharded-bridge                                                           */
/* ------------------------------------------------------------------------ */

/* all_reduce under the sharded-bridge policy (gpubridge README, policy table,
 * sharded-bridge row).  k is the size of the smallest island.  Each island
 * reduce_scatters its sum onto its first k ranks, so that rank j of the
 * island holds the island sum of segment j; rank j of every island then
 * all_reduces segment j over its own bridge link (encode, exchange, decode
 * and add in island order, AVG); each island finally all_gathers the
 * segments to all its ranks.  With one island, or an island of one rank
 * (k == 1), it is reduce-bridge-broadcast.
 *
 * Reading (the page does not say where the tensor is cut): segment j is
 * [j * seg, (j + 1) * seg) with seg = ceil(n / k) rounded up to a multiple of
 * 256 elements, so that every codec block lies inside one segment; trailing
 * segments may be short or empty.  The codec blocks of a segment count from
 * its first element.  *seg_out (if not NULL) receives seg (n for k == 1).
 * dtype float32 or bf16. */
int orc_all_reduce_sharded(int I, const int *island_sizes, const void *const *in, void *const *out,
                           size_t n, int dtype, int op, int codec, int block, size_t *seg_out)
{
    int W = 0, k = island_sizes[0];
    for (int i = 0; i < I; ++i) {
        W += island_sizes[i];
        if (island_sizes[i] < k)
            k = island_sizes[i];
    }
    if (I == 1 || k == 1) {
        if (seg_out)
            *seg_out = n;
        return orc_all_reduce(I, island_sizes, in, out, n, dtype, op, codec, block);
    }
    size_t seg = (n + (size_t)k - 1) / (size_t)k;
    seg = (seg + 255) / 256 * 256;
    if (seg_out)
        *seg_out = seg;
    const size_t eb = orc_dtype_bytes(dtype);
    float *t = malloc((n ? n : 1) * sizeof(float));
    const void **part = malloc(sizeof(void *) * (size_t)W);
    if (!t || !part) {
        free(t); free(part);
        return -1;
    }
    for (int j = 0; j < k; ++j) {
        const size_t e0 = (size_t)j * seg;
        if (e0 >= n)
            break;
        const size_t m = (n - e0) < seg ? (n - e0) : seg;
        for (int r = 0; r < W; ++r)
            part[r] = (const uint8_t *)in[r] + e0 * eb;
        /* rank j of each island: the island sum of segment j (the island
         * reduce_scatter), encoded, exchanged over link j, decoded and added
         * in island order */
        if (orc_rbb_total(I, island_sizes, part, m, dtype, op, codec, block, t + e0, NULL, NULL, NULL)) {
            free(t); free(part);
            return -1;
        }
    }
    /* island all_gather: every rank receives every segment */
    for (int r = 0; r < W; ++r)
        for (size_t j = 0; j < n; ++j)
            store_elem(out[r], dtype, j, t[j]);
    free(t); free(part);
    return 0;
}
