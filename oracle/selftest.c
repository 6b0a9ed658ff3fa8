/* The oracle's self-test in C, with no GPU and no Python: it links
 * liboracle.so and checks the oracle against what the source pages and the
 * OCP 8-bit floating point definition fix, read from the golden fixtures
 * (the text files under tests/golden, paths given on the command line in
 * this order: demo_four_ranks.txt codec_sizes.txt ofp8_values.txt), plus
 * closed forms of
 * the block-scale rule.  Test infrastructure only.  Prints one line per
 * check ("ok <check>" or "FAIL <check>") and exits non-zero if any fails. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

enum { DT_F32 = 0, OP_SUM = 0, CODEC_NONE = 0, CODEC_BF16 = 1, CODEC_E4M3 = 2, CODEC_E5M2 = 3 };

/* the oracle's entry points (oracle/oracle.c) */
int orc_all_reduce(int I, const int *island_sizes, const void *const *in, void *const *out, size_t n,
                   int dtype, int op, int codec, int block);
void orc_decode(const void *codes, const float *scales, size_t n, int codec, int block, float *out);
int orc_block_scale_exponent(float absmax, int fmt);
size_t orc_n_blocks(size_t n, int block);

static int fails = 0;

static void check(int ok, const char *what)
{
    if (ok) {
        printf("ok %s\n", what);
    } else {
        printf("FAIL %s\n", what);
        ++fails;
    }
}

/* next non-comment line of f into buf; 0 at end of file */
static int next_line(FILE *f, char *buf, size_t size)
{
    while (fgets(buf, (int)size, f)) {
        if (buf[0] == '#' || buf[0] == '\n')
            continue;
        return 1;
    }
    return 0;
}

/* The four-rank demo: islands [0, 1] and [2, 3], every element of rank r is
 * r + 1, every rank ends with 10.0 -- for every codec (the island sums 3 and
 * 7 and the total 10 are exact in bf16, E4M3 and E5M2 with a power-of-two
 * scale). */
static void demo(const char *path)
{
    FILE *f = fopen(path, "r");
    char line[512];
    int sizes[2] = {0, 0};
    size_t n = 0;
    float in[4][16];
    float expect[16];
    int got_expect = 0;
    if (!f) {
        check(0, "demo fixture opens");
        return;
    }
    while (next_line(f, line, sizeof line)) {
        if (sscanf(line, "island_sizes %d %d", &sizes[0], &sizes[1]) == 2)
            continue;
        if (sscanf(line, "n %zu", &n) == 1)
            continue;
        int r;
        int pos = 0;
        if (sscanf(line, "input %d%n", &r, &pos) == 1 && r >= 0 && r < 4) {
            char *p = line + pos;
            for (size_t j = 0; j < n && j < 16; ++j)
                in[r][j] = strtof(p, &p);
            continue;
        }
        if (strncmp(line, "expected_sum", 12) == 0) {
            char *p = line + 12;
            for (size_t j = 0; j < n && j < 16; ++j)
                expect[j] = strtof(p, &p);
            got_expect = 1;
        }
    }
    fclose(f);
    check(sizes[0] == 2 && sizes[1] == 2 && n == 4 && got_expect, "demo fixture parsed");
    const int codecs[4] = {CODEC_NONE, CODEC_BF16, CODEC_E4M3, CODEC_E5M2};
    const char *names[4] = {"demo total, codec none", "demo total, codec bf16", "demo total, codec e4m3",
                            "demo total, codec e5m2"};
    for (int c = 0; c < 4; ++c) {
        float out[4][16];
        const void *ins[4] = {in[0], in[1], in[2], in[3]};
        void *outs[4] = {out[0], out[1], out[2], out[3]};
        int ok = orc_all_reduce(2, sizes, ins, outs, n, DT_F32, OP_SUM, codecs[c], 256) == 0;
        for (int r = 0; r < 4; ++r)
            for (size_t j = 0; j < n; ++j)
                ok = ok && out[r][j] == expect[j];
        check(ok, names[c]);
    }
}

/* The codec size ratios: float32 bytes over payload bytes for whole blocks,
 * to one decimal -- fp8 codes plus one float32 scale per block, bf16 codes. */
static void sizes_check(const char *path)
{
    FILE *f = fopen(path, "r");
    char line[512];
    int block = 0;
    double fp8_ratio = 0, bf16_ratio = 0;
    if (!f) {
        check(0, "codec size fixture opens");
        return;
    }
    while (next_line(f, line, sizeof line)) {
        if (sscanf(line, "fp8_e4m3_block %d", &block) == 1)
            continue;
        if (sscanf(line, "fp8_ratio_one_decimal %lf", &fp8_ratio) == 1)
            continue;
        sscanf(line, "bf16_ratio %lf", &bf16_ratio);
    }
    fclose(f);
    const size_t n = (size_t)block * 4096;
    const double fp8 = (double)(4 * n) / (double)(n + 4 * orc_n_blocks(n, block));
    const double bf16 = (double)(4 * n) / (double)(2 * n);
    check(block == 256 && fabs(round(fp8 * 10) / 10 - fp8_ratio) < 1e-9, "fp8 payload ratio 3.9");
    check(fabs(bf16 - bf16_ratio) < 1e-9, "bf16 payload ratio 2");
}

/* The OFP8 table: each listed code decodes (scale 1) to the listed value. */
static void ofp8(const char *path)
{
    FILE *f = fopen(path, "r");
    char line[512];
    int rows = 0, ok = 1;
    if (!f) {
        check(0, "OFP8 fixture opens");
        return;
    }
    while (next_line(f, line, sizeof line)) {
        char fmt[16], val[64];
        unsigned code;
        if (sscanf(line, "%15s %x %63s", fmt, &code, val) != 3)
            continue;
        const int codec = strcmp(fmt, "e4m3") == 0 ? CODEC_E4M3 : CODEC_E5M2;
        const uint8_t c8 = (uint8_t)code;
        const float one = 1.0f;
        float got;
        orc_decode(&c8, &one, 1, codec, 256, &got);
        if (strcmp(val, "nan") == 0)
            ok = ok && isnan(got);
        else if (strcmp(val, "inf") == 0)
            ok = ok && isinf(got) && got > 0;
        else if (strcmp(val, "-inf") == 0)
            ok = ok && isinf(got) && got < 0;
        else
            ok = ok && got == strtof(val, NULL);
        ++rows;
    }
    fclose(f);
    check(rows >= 10 && ok, "OFP8 table values decode");
}

/* The block-scale rule in closed form: the smallest k with absmax * 2^-k <=
 * M puts absmax into (M/2, M]. */
static void scale_rule(void)
{
    const float M4 = 448.0f, M5 = 57344.0f;
    check(orc_block_scale_exponent(M4, CODEC_E4M3) == 0, "scale: absmax = M (E4M3) gives k = 0");
    check(orc_block_scale_exponent(nextafterf(M4, INFINITY), CODEC_E4M3) == 1, "scale: just above M gives k = 1");
    check(orc_block_scale_exponent(M4 / 2, CODEC_E4M3) == -1, "scale: M / 2 gives k = -1");
    check(orc_block_scale_exponent(nextafterf(M4 / 2, INFINITY), CODEC_E4M3) == 0, "scale: just above M / 2 gives k = 0");
    check(orc_block_scale_exponent(M5 * 1024.0f, CODEC_E5M2) == 10, "scale: M * 2^10 (E5M2) gives k = 10");
    check(orc_block_scale_exponent(0.0f, CODEC_E4M3) == 0, "scale: an all-zero block gives k = 0");
    check(orc_block_scale_exponent(1e-44f, CODEC_E4M3) == -126, "scale: a subnormal absmax clamps to k = -126");
    int ok = 1;
    for (int e = -100; e <= 100; ++e) {
        const float a = ldexpf(1.0f, e) * 1.3f;
        const int k = orc_block_scale_exponent(a, CODEC_E4M3);
        const double y = ldexp((double)a, -k);
        ok = ok && (k == -126 || (y <= M4 && y > M4 / 2));
    }
    check(ok, "scale: absmax * 2^-k lands in (M/2, M] over 200 binades");
}

int main(int argc, char **argv)
{
    if (argc != 4) {
        fprintf(stderr, "usage: %s demo_four_ranks.txt codec_sizes.txt ofp8_values.txt\n", argv[0]);
        return 2;
    }
    demo(argv[1]);
    sizes_check(argv[2]);
    ofp8(argv[3]);
    scale_rule();
    return fails ? 1 : 0;
}
