/*
 * fp8bs_oracle.c -- plain, slow CPU oracle for the fine-grained FP8 linear layer.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline may load this file's library. It shares no code, header, table or
 * constant with the CUDA library; each side is written from the sources below.
 *
 * What it computes, and where each step is stated:
 *   - E4M3 number format: OCP 8-bit Floating Point Specification (OFP8), E4M3
 *     encoding (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
 *     subnormals at exponent 0, no infinities, only S.1111.111 is NaN).
 *     The pages fix the largest finite value 448 (TransformerEngine PR #3573,
 *     "Changes": the E4M3 bound is 448 unless 4over6 asks for 256) and the two
 *     zero payloads +0 = 0x00, -0 = 0x80 (prime-rl PR #4073, conventions
 *     table, row "Negative zero").
 *   - Fine-grained dynamic scaling: "FP8 动态量化里的 partial sum 漂移", section 3,
 *     table row (a): tiles of N_c = 128, a dynamic scale per tile from the
 *     tile's absmax, values rounded to FP8 inside the tile.
 *   - Tile shapes 1x128 (activations, gradients), 128x128 (weights) and the
 *     128x1 re-tiling of saved operands for Wgrad: "scratch: the backward pass,
 *     unrolled", "What is asserted, and from where", bullets 1 and 2.
 *   - Per-128 promotion: same partial-sum page, section 3 row (b) and section 5:
 *     the partial over 128 elements of K is flushed into an FP32 accumulator
 *     after being multiplied by s_x * s_w.
 *   - Unpromoted accumulation (drift model): same page, section 4,
 *     s_hat_t = round(s_hat_{t-1} + round(p_t)).
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes of the repository):
 *   - s = amax / 448 is a true IEEE fp32 division, and q = E4M3_RN(fp32(v / s))
 *     (the quotient is rounded to fp32 first, then to E4M3).
 *   - E4M3 rounding is round-to-nearest, ties to the even code, saturating to
 *     +-448, and a result of zero keeps the sign of its input.
 *   - An all-zero tile stores s = 1 and signed zeros.
 *   - Partial tiles at a ragged edge take the absmax over their valid elements.
 *   - The per-block partial sum P_b is exact (accumulated in fp64, which holds
 *     every sum of 128 E4M3 products exactly), rounded once to fp32, multiplied
 *     by the fp32 product s_a * s_b, and added to the fp32 accumulator in block
 *     order. Compile with -ffp-contract=off so that no FMA fuses these steps.
 *
 * Build: gcc -std=c99 -O2 -fPIC -shared -ffp-contract=off [-fopenmp]
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

/* ------------------------------------------------------------------------- */
/* E4M3 table (OCP OFP8 E4M3 definition).                                     */
/* ------------------------------------------------------------------------- */

static float g_dec[256];
static int g_dec_ready = 0;

/* Planted-mistake switch, used only by the negative-control tests: each value
 * makes one plausible implementation error on purpose so that the tests can
 * show that the pins catch it. 0 (the default) is the correct oracle. */
enum {
    FAULT_NONE = 0,
    FAULT_DROP_LAST_BLOCK = 1,   /* promoted sum skips the last K-block */
    FAULT_SCALE_NEXT_BLOCK = 2,  /* B scale taken from the next K-block */
    FAULT_TIES_AWAY = 3,         /* E4M3 ties round away from zero */
    FAULT_SIGNED_AMAX = 4,       /* tile scale from max(v) instead of max|v| */
    FAULT_TRANSPOSED_W = 5,      /* fprop reads W transposed */
    FAULT_DROP_NEG_ZERO = 6,     /* -0 results encoded as 0x00 */
    FAULT_RECIPROCAL = 7,        /* v * (1/s) instead of v / s */
    FAULT_SIGN_FLIP_TERM = 8,    /* one K-block's term subtracted */
    FAULT_UE8M0_DOWN = 9,        /* UE8M0 scale rounded down, not up */
    FAULT_FLOOR_AFTER = 10,      /* amax floor applied to s instead of amax */
    FAULT_SR_WORD = 11,          /* SR takes the next Philox output word */
    FAULT_SR_NEAREST = 12,       /* SR rounds to nearest instead */
    FAULT_SR_BLOCK_INDEX = 13,   /* 128x128 SR numbers elements inside each block, not in the tensor */
    FAULT_REQUANT_TILE_SCALE = 14  /* E4M3-source requant decodes every token of a tile with
                                      the source scale of the tile's first token */
};
static int g_fault = FAULT_NONE;

void oracle_set_fault(int f) { g_fault = f; }

static void build_table(void)
{
    if (g_dec_ready) return;
    for (int c = 0; c < 256; ++c) {
        int sign = (c >> 7) & 1;
        int e = (c >> 3) & 0xF;
        int m = c & 0x7;
        double mag;
        if (e == 0xF && m == 0x7) {      /* S.1111.111 is the only NaN */
            g_dec[c] = NAN;
            continue;
        }
        if (e == 0)
            mag = ldexp((double)m, -9);  /* subnormal: (m/8) * 2^(1-7) */
        else
            mag = ldexp(8.0 + m, e - 10); /* (1 + m/8) * 2^(e-7) */
        g_dec[c] = (float)(sign ? -mag : mag);
    }
    g_dec_ready = 1;
}

void oracle_e4m3_table(float out[256])
{
    build_table();
    memcpy(out, g_dec, sizeof(g_dec));
}

/* Nearest finite E4M3 by search over the table: the positive codes
 * 0x00..0x7E are ascending in value, so bisect for the largest code not above
 * |v| and compare |v| with the midpoint to the next one. Ties take the even
 * code (mantissa LSB 0). |v| >= 448 saturates to 448. Zero keeps v's sign. */
uint8_t oracle_e4m3_encode(float v)
{
    build_table();
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E;               /* g_dec[lo] <= a < g_dec[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if ((double)g_dec[mid] <= a) lo = mid; else hi = mid;
    }
    /* midpoint comparison done exactly: both sides are exact in double */
    double twice = 2.0 * a;
    double msum = (double)g_dec[lo] + (double)g_dec[lo + 1];
    int c;
    if (twice < msum) c = lo;
    else if (twice > msum) c = lo + 1;
    else if (g_fault == FAULT_TIES_AWAY) c = lo + 1;
    else c = (lo % 2 == 0) ? lo : lo + 1;
    if (c == 0 && g_fault == FAULT_DROP_NEG_ZERO) sign = 0;
    return (uint8_t)(sign | c);
}

void oracle_e4m3_encode_array(const float* v, i64 n, uint8_t* out)
{
    for (i64 i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

float oracle_e4m3_decode(uint8_t c)
{
    build_table();
    return g_dec[c];
}

/* bf16 bits -> fp32 (exact). */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs; NaN -> quiet NaN). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_f32_to_bf16_array(const float* in, i64 n, uint16_t* out)
{
    for (i64 i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------- */
/* Stochastic rounding to E4M3.                                               */
/* ------------------------------------------------------------------------- */

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 * as 1, 2, 3", SC 2011): ten rounds on a 4-word counter with a 2-word key;
 * each round multiplies words 0 and 2 by the round multipliers, keeps both
 * halves of the 64-bit products and mixes them with words 1 and 3 and the
 * key; the key grows by the Weyl constants between rounds. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The random word of element `idx` (its linear index in the quantized
 * tensor) under (seed, salt): Philox4x32-10 with key (seed low word, seed
 * high word) and counter (low and high words of idx / 4, salt, 0); element
 * idx takes output word idx % 4. Stateless: the word depends on nothing else
 * (tile shape, launch, thread). This contract is this repository's reading;
 * the pages name a stateless seed / salt / counter scheme without its
 * layout. */
uint32_t oracle_sr_word(uint64_t seed, uint32_t salt, uint64_t idx)
{
    uint64_t blk = idx / 4;
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), salt, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    int w = (int)(idx % 4);
    if (g_fault == FAULT_SR_WORD) w = (w + 1) % 4;
    return out[w];
}

/* Stochastic rounding of an fp32 quotient x to E4M3 with the random word r:
 * with L the largest E4M3 magnitude <= |x| and U the next one, the fraction
 * f = (|x| - L) / (U - L) in [0, 1) is cut to 20 bits, F = floor(f * 2^20),
 * and the result is U when F > (r >> 12), else L (so P(U) = F / 2^20). The
 * sign is x's (a zero result keeps it); |x| >= 448 gives 448. */
uint8_t oracle_e4m3_encode_sr(float x, uint32_t r)
{
    build_table();
    if (g_fault == FAULT_SR_NEAREST) return oracle_e4m3_encode(x);
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E;               /* g_dec[lo] <= a < g_dec[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if ((double)g_dec[mid] <= a) lo = mid; else hi = mid;
    }
    double L = g_dec[lo], U = g_dec[lo + 1];
    double f = (a - L) / (U - L);        /* exact: a, L, U are short dyadic numbers */
    uint32_t F = (uint32_t)floor(f * 1048576.0);
    int c = (F > (r >> 12)) ? lo + 1 : lo;
    return (uint8_t)(sign | c);
}

/* ------------------------------------------------------------------------- */
/* One quantization tile: amax, scale, codes.                                 */
/* ------------------------------------------------------------------------- */

/* Scale rule options (prime-rl PR #4073, conventions table, rows "Weight
 * floors", "Two-stage weights", "Activation floors", "Compact formats"): an
 * amax floor applied before the division, a scale floor applied after it,
 * and power-of-two (UE8M0) scales. The table names these conventions without
 * fixing their order; the reading used here (also stated in the design
 * notes): a = max(amax, amax_floor); s = a / 448, or 1 when a == 0 and no
 * scale floor is set; s = max(s, scale_floor); UE8M0: s = the smallest power
 * of two >= s. Defaults (rule 0, no floors) give the plain rule. */
static int g_ue8m0 = 0;
static float g_amax_floor = 0.0f;
static float g_scale_floor = 0.0f;

void oracle_set_scale_rule(int ue8m0, float amax_floor, float scale_floor)
{
    g_ue8m0 = ue8m0;
    g_amax_floor = amax_floor;
    g_scale_floor = scale_floor;
}

/* Smallest power of two that is >= s (s > 0), from frexp's decomposition
 * s = m * 2^e with m in [0.5, 1): s itself when m == 0.5, else 2^e. */
static float pow2_at_least(float s)
{
    int e;
    float m = frexpf(s, &e);
    return (m == 0.5f) ? s : ldexpf(1.0f, e);
}

/* Scale of a tile whose values are v[0..n) under the current scale rule
 * (default: amax / 448 in fp32, or 1 for an all-zero tile). */
static float tile_scale(const float* v, int n)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = (g_fault == FAULT_SIGNED_AMAX) ? v[i] : fabsf(v[i]);
        if (a > amax) amax = a;
    }
    if (g_fault != FAULT_FLOOR_AFTER && amax < g_amax_floor) amax = g_amax_floor;
    float s;
    if (amax == 0.0f && g_scale_floor == 0.0f && (g_fault != FAULT_FLOOR_AFTER || g_amax_floor == 0.0f))
        s = 1.0f;
    else
        s = amax / 448.0f;
    if (g_fault == FAULT_FLOOR_AFTER && s < g_amax_floor) s = g_amax_floor;
    if (s < g_scale_floor) s = g_scale_floor;
    if (g_ue8m0) {
        s = pow2_at_least(s);
        if (g_fault == FAULT_UE8M0_DOWN && amax != 0.0f) s = 0.5f * s;
    }
    return s;
}

static void tile_encode(const float* v, int n, float s, uint8_t* out, i64 out_step)
{
    for (int i = 0; i < n; ++i) {
        float quot = (g_fault == FAULT_RECIPROCAL) ? v[i] * (1.0f / s) : v[i] / s;
        out[i * out_step] = oracle_e4m3_encode(quot);
    }
}

/* tile_encode with stochastic rounding: element i's linear index in the
 * tensor is idx0 + i * idx_step. */
static void tile_encode_sr(const float* v, int n, float s, uint8_t* out, i64 out_step,
                           uint64_t seed, uint32_t salt, i64 idx0, i64 idx_step)
{
    for (int i = 0; i < n; ++i) {
        float quot = v[i] / s;
        uint32_t r = oracle_sr_word(seed, salt, (uint64_t)(idx0 + (i64)i * idx_step));
        out[i * out_step] = oracle_e4m3_encode_sr(quot, r);
    }
}

/* S1 with stochastic rounding (element index r * cols + c). */
void oracle_quant_1x128_sr(const uint16_t* x, i64 rows, i64 cols, i64 ldx,
                           uint8_t* q, i64 ldq, float* sc, i64 sc_rs, i64 sc_ts,
                           uint64_t seed, uint32_t salt)
{
    i64 ntiles = (cols + 127) / 128;
#pragma omp parallel for schedule(static)
    for (i64 r = 0; r < rows; ++r) {
        float v[128];
        for (i64 t = 0; t < ntiles; ++t) {
            i64 c0 = t * 128;
            int n = (int)((cols - c0) < 128 ? (cols - c0) : 128);
            for (int i = 0; i < n; ++i) v[i] = bf16_to_f32(x[r * ldx + c0 + i]);
            float s = tile_scale(v, n);
            sc[r * sc_rs + t * sc_ts] = s;
            tile_encode_sr(v, n, s, q + r * ldq + c0, 1, seed, salt, r * cols + c0, 1);
        }
    }
}

/* S2 with stochastic rounding (element index idx_base + r * cols + c). */
void oracle_quant_128x128_sr(const uint16_t* x, i64 rows, i64 cols, i64 ldx,
                             uint8_t* q, i64 ldq, float* sc, i64 ldsc,
                             uint64_t seed, uint32_t salt, i64 idx_base)
{
    i64 nbr = (rows + 127) / 128, nbc = (cols + 127) / 128;
#pragma omp parallel for schedule(static)
    for (i64 blk = 0; blk < nbr * nbc; ++blk) {
        i64 bi = blk / nbc, bj = blk % nbc;
        i64 r0 = bi * 128, c0 = bj * 128;
        int nr = (int)((rows - r0) < 128 ? (rows - r0) : 128);
        int nc = (int)((cols - c0) < 128 ? (cols - c0) : 128);
        float v[128 * 128];
        for (int i = 0; i < nr; ++i)
            for (int j = 0; j < nc; ++j)
                v[i * nc + j] = bf16_to_f32(x[(r0 + i) * ldx + c0 + j]);
        float s = tile_scale(v, nr * nc);
        sc[bi * ldsc + bj] = s;
        for (int i = 0; i < nr; ++i) {
            i64 idx0 = idx_base + (r0 + i) * cols + c0;
            if (g_fault == FAULT_SR_BLOCK_INDEX) idx0 = idx_base + blk * 128 * 128 + (i64)i * nc;
            tile_encode_sr(v + i * nc, nc, s, q + (r0 + i) * ldq + c0, 1, seed, salt, idx0, 1);
        }
    }
}

/* S1: 1x128 tiles along each row.
 * x: bf16 [rows x cols], row stride ldx (elements).
 * q: E4M3 [rows x cols], row stride ldq.
 * scale of (row r, tile t) is written to sc[r * sc_rs + t * sc_ts]. */
void oracle_quant_1x128(const uint16_t* x, i64 rows, i64 cols, i64 ldx,
                        uint8_t* q, i64 ldq, float* sc, i64 sc_rs, i64 sc_ts)
{
    i64 ntiles = (cols + 127) / 128;
#pragma omp parallel for schedule(static)
    for (i64 r = 0; r < rows; ++r) {
        float v[128];
        for (i64 t = 0; t < ntiles; ++t) {
            i64 c0 = t * 128;
            int n = (int)((cols - c0) < 128 ? (cols - c0) : 128);
            for (int i = 0; i < n; ++i) v[i] = bf16_to_f32(x[r * ldx + c0 + i]);
            float s = tile_scale(v, n);
            sc[r * sc_rs + t * sc_ts] = s;
            tile_encode(v, n, s, q + r * ldq + c0, 1);
        }
    }
}

/* S2: 128x128 blocks. Scale of block (bi, bj) goes to sc[bi * ldsc + bj]. */
void oracle_quant_128x128(const uint16_t* x, i64 rows, i64 cols, i64 ldx,
                          uint8_t* q, i64 ldq, float* sc, i64 ldsc)
{
    i64 nbr = (rows + 127) / 128, nbc = (cols + 127) / 128;
#pragma omp parallel for schedule(static)
    for (i64 blk = 0; blk < nbr * nbc; ++blk) {
        i64 bi = blk / nbc, bj = blk % nbc;
        i64 r0 = bi * 128, c0 = bj * 128;
        int nr = (int)((rows - r0) < 128 ? (rows - r0) : 128);
        int nc = (int)((cols - c0) < 128 ? (cols - c0) : 128);
        float v[128 * 128];
        for (int i = 0; i < nr; ++i)
            for (int j = 0; j < nc; ++j)
                v[i * nc + j] = bf16_to_f32(x[(r0 + i) * ldx + c0 + j]);
        float s = tile_scale(v, nr * nc);
        sc[bi * ldsc + bj] = s;
        for (int i = 0; i < nr; ++i)
            tile_encode(v + i * nc, nc, s, q + (r0 + i) * ldq + c0, 1);
    }
}

/* ------------------------------------------------------------------------- */
/* MXFP8: 1x32 blocks with power-of-two (UE8M0) scales.              */
/* ------------------------------------------------------------------------- */

/* OCP Microscaling Formats (MX) v1.0: a block of 32 consecutive elements
 * along K shares one 8-bit exponent scale X = 2^(E - 127); elements are E4M3.
 * Scale choice (this repository's reading, the same power-of-two rule as the
 * UE8M0 option of the 1x128 casts; the MX spec's own floor(log2 amax) - 8
 * rule can saturate the block maximum): X = the smallest power of two
 * >= fp32(amax / 448), X = 1 for an all-zero block; q = E4M3_RN(v / X), exact
 * division. Scales are returned as exponent bytes E, row-major
 * [rows x cols/32]. */
static uint8_t mx_scale_byte(float amax)
{
    if (amax == 0.0f) return 127;
    float s = pow2_at_least(amax / 448.0f);
    int e;
    frexpf(s, &e);                        /* s = 0.5 * 2^e = 2^(e - 1) */
    int E = (e - 1) + 127;
    if (E < 0) E = 0;
    if (E > 254) E = 254;
    return (uint8_t)E;
}

void oracle_mx_quant_1x32(const uint16_t* x, i64 rows, i64 cols, uint8_t* q, uint8_t* sc)
{
    build_table();
    i64 nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (i64 r = 0; r < rows; ++r) {
        for (i64 b = 0; b < nb; ++b) {
            float v[32], amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                v[i] = bf16_to_f32(x[r * cols + b * 32 + i]);
                if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
            }
            uint8_t E = mx_scale_byte(amax);
            sc[r * nb + b] = E;
            float s = ldexpf(1.0f, (int)E - 127);
            for (int i = 0; i < 32; ++i) q[r * cols + b * 32 + i] = oracle_e4m3_encode(v[i] / s);
        }
    }
}

/* MXFP8 GEMM: out[i, j] = sum_k dec(a[i, k]) 2^(Ea[i, k/32] - 127) *
 * dec(b[j, k]) 2^(Eb[j, k/32] - 127), with A [M x K] and B [N x K] both
 * blocked along K; accumulated in fp64 (every product is exact; the sum is
 * rounded once, to fp32, at the end). If ii/jj are given, only those n
 * elements are computed (out[e] for (ii[e], jj[e])); else all M x N. */
void oracle_mx_gemm(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                    i64 M, i64 N, i64 K, float* out, const i64* ii, const i64* jj, i64 n)
{
    build_table();
    i64 nb = K / 32;
    i64 total = ii ? n : M * N;
#pragma omp parallel for schedule(static)
    for (i64 e = 0; e < total; ++e) {
        i64 i = ii ? ii[e] : e / N;
        i64 j = ii ? jj[e] : e % N;
        double acc = 0.0;
        for (i64 blk = 0; blk < nb; ++blk) {
            double part = 0.0;
            for (int t = 0; t < 32; ++t) {
                i64 k = blk * 32 + t;
                part += (double)g_dec[a[i * K + k]] * (double)g_dec[b[j * K + k]];
            }
            acc += part * ldexp(1.0, (int)sa[i * nb + blk] - 127) * ldexp(1.0, (int)sb[j * nb + blk] - 127);
        }
        out[e] = (float)acc;
    }
}

/* Number of token columns the transposed output holds: each group's token
 * count rounded up to a whole number of 128-token tiles. */
i64 oracle_padded_tokens(const int32_t* offsets, int groups, i64 rows)
{
    if (!offsets || groups <= 0) return ((rows + 127) / 128) * 128;
    i64 tot = 0;
    for (int g = 0; g < groups; ++g) {
        i64 n = (i64)offsets[g + 1] - (i64)offsets[g];
        tot += ((n + 127) / 128) * 128;
    }
    return tot;
}

/* S3: 128x1 tiles along the token (row) axis, transposed output.
 *   mode 0 (B): src is bf16 [rows x cols] with row stride ld_src.
 *   mode 1 (Q): src is E4M3 [rows x cols] with row stride ld_src and 1x128
 *               scales src_sc[r * src_rs + t * src_ts]; an element is
 *               decoded as fp32(dec(q) * s) before requantization.
 * groups > 0 splits the rows at offsets[0..groups] (offsets[0] = 0); each
 * group's tiles start at its own first row and the group's segment in the
 * output starts at a multiple of 128 (padded token index).
 * qT: E4M3 [cols x Mpad], row stride ldqT; padding bytes are 0x00.
 * scT: fp32 [Mpad/128 x cols], row stride ldscT. */
/* S3 body: with sr != 0 the codes are stochastically rounded, the element
 * (row r, column c) of the source taking the word of index r * cols + c. */
static void requant_impl(int mode, const void* src, i64 ld_src,
                         const float* src_sc, i64 src_rs, i64 src_ts,
                         i64 rows, i64 cols, const int32_t* offsets, int groups,
                         uint8_t* qT, i64 ldqT, float* scT, i64 ldscT,
                         int sr, uint64_t seed, uint32_t salt)
{
    build_table();
    int ng = (offsets && groups > 0) ? groups : 1;
    i64 pstart = 0;
    for (int g = 0; g < ng; ++g) {
        i64 r_begin = (offsets && groups > 0) ? offsets[g] : 0;
        i64 r_end = (offsets && groups > 0) ? offsets[g + 1] : rows;
        i64 n = r_end - r_begin;
        i64 ntiles = (n + 127) / 128;
#pragma omp parallel for schedule(static)
        for (i64 c = 0; c < cols; ++c) {
            float v[128];
            for (i64 t = 0; t < ntiles; ++t) {
                i64 r0 = r_begin + t * 128;
                int len = (int)((r_end - r0) < 128 ? (r_end - r0) : 128);
                for (int i = 0; i < len; ++i) {
                    i64 r = r0 + i;
                    if (mode == 0) {
                        v[i] = bf16_to_f32(((const uint16_t*)src)[r * ld_src + c]);
                    } else {
                        uint8_t code = ((const uint8_t*)src)[r * ld_src + c];
                        i64 rs = (g_fault == FAULT_REQUANT_TILE_SCALE) ? r0 : r;
                        float s1 = src_sc[rs * src_rs + (c / 128) * src_ts];
                        v[i] = g_dec[code] * s1;
                    }
                }
                float s = tile_scale(v, len);
                scT[(pstart / 128 + t) * ldscT + c] = s;
                uint8_t* dst = qT + c * ldqT + pstart + t * 128;
                if (sr)
                    tile_encode_sr(v, len, s, dst, 1, seed, salt, r0 * cols + c, cols);
                else
                    tile_encode(v, len, s, dst, 1);
                for (int i = len; i < 128; ++i) dst[i] = 0x00;
            }
        }
        pstart += ntiles * 128;
    }
}

void oracle_requant_128x1_T(int mode, const void* src, i64 ld_src,
                            const float* src_sc, i64 src_rs, i64 src_ts,
                            i64 rows, i64 cols, const int32_t* offsets, int groups,
                            uint8_t* qT, i64 ldqT, float* scT, i64 ldscT)
{
    requant_impl(mode, src, ld_src, src_sc, src_rs, src_ts, rows, cols, offsets, groups, qT, ldqT, scT, ldscT,
                 0, 0, 0);
}

/* S3 with stochastic rounding (element index r * cols + c of the source). */
void oracle_requant_128x1_T_sr(int mode, const void* src, i64 ld_src,
                               const float* src_sc, i64 src_rs, i64 src_ts,
                               i64 rows, i64 cols, const int32_t* offsets, int groups,
                               uint8_t* qT, i64 ldqT, float* scT, i64 ldscT,
                               uint64_t seed, uint32_t salt)
{
    requant_impl(mode, src, ld_src, src_sc, src_rs, src_ts, rows, cols, offsets, groups, qT, ldqT, scT, ldscT,
                 1, seed, salt);
}

/* ------------------------------------------------------------------------- */
/* Promoted block-scaled GEMM.                                               */
/* ------------------------------------------------------------------------- */

/* Exact partial sum of one K-block: sum of dec(a[k]) * dec(b[k]) for k in
 * [k0, k1), accumulated in fp64 (exact for at most 128 E4M3 products). */
static double block_partial(const uint8_t* a, i64 a_step, const uint8_t* b, i64 b_step,
                            i64 k0, i64 k1)
{
    double p = 0.0;
    for (i64 k = k0; k < k1; ++k)
        p += (double)g_dec[a[k * a_step]] * (double)g_dec[b[k * b_step]];
    return p;
}

/* Generic promoted dot product for one output element.
 *   a[k * a_step], b[k * b_step] for k in [0, K): the E4M3 operand codes;
 *   sa[blk * sa_step], sb[blk * sb_step]: the scales of K-block blk.
 * acc = sum over blocks, in block order, of fp32(P_b) * fp32(s_a * s_b). */
static float promoted_dot(const uint8_t* a, i64 a_step, const uint8_t* b, i64 b_step,
                          i64 K, const float* sa, i64 sa_step, const float* sb, i64 sb_step)
{
    float acc = 0.0f;
    i64 nb = (K + 127) / 128;
    for (i64 blk = 0; blk < nb; ++blk) {
        if (g_fault == FAULT_DROP_LAST_BLOCK && blk == nb - 1) break;
        i64 k0 = blk * 128, k1 = (k0 + 128 < K) ? k0 + 128 : K;
        double p = block_partial(a, a_step, b, b_step, k0, k1);
        i64 bblk = (g_fault == FAULT_SCALE_NEXT_BLOCK) ? (blk + 1) % nb : blk;
        float s = sa[blk * sa_step] * sb[bblk * sb_step];
        float term = (float)p * s;
        if (g_fault == FAULT_SIGN_FLIP_TERM && blk == 0 && nb > 1) term = -term;
        acc = acc + term;
    }
    return acc;
}

/* Fprop, Y = X W:
 *   Y[i,j] = sum_b s_x[i,b] * s_w[b, j/128] * P_b[i,j],
 *   P_b[i,j] = sum_{k in block b} dec(xq[i,k]) * dec(wq[k,j]).
 * xq: [M x K] row stride ldx; sx(i, b) = sx[i * sx_rs + b * sx_ts].
 * wq: [K x N] row stride ldw; sw(bk, bn) = sw[bk * ldsw + bn].
 * Output (fp32, before the BF16 rounding) for n_out elements at (ii[e], jj[e]),
 * or the whole M x N row-major when ii is NULL. */
void oracle_fprop(const uint8_t* xq, i64 ldx, const float* sx, i64 sx_rs, i64 sx_ts,
                  const uint8_t* wq, i64 ldw, const float* sw, i64 ldsw,
                  i64 M, i64 N, i64 K, const i64* ii, const i64* jj, i64 n_out,
                  float* out)
{
    build_table();
    i64 total = ii ? n_out : M * N;
#pragma omp parallel for schedule(dynamic, 64)
    for (i64 e = 0; e < total; ++e) {
        i64 i = ii ? ii[e] : e / N;
        i64 j = ii ? jj[e] : e % N;
        if (g_fault == FAULT_TRANSPOSED_W)   /* reads W[j, k]: only meaningful for K == N */
            out[e] = promoted_dot(xq + i * ldx, 1, wq + j * ldw, 1, K,
                                  sx + i * sx_rs, sx_ts, sw + (j / 128), ldsw);
        else
            out[e] = promoted_dot(xq + i * ldx, 1, wq + j, ldw, K,
                                  sx + i * sx_rs, sx_ts, sw + (j / 128), ldsw);
    }
}

/* Dgrad, dX = dY W^T (contraction over the N outputs of the layer):
 *   dX[i,k] = sum_b s_dy[i,b] * s_w[k/128, b] * P_b[i,k],
 *   P_b[i,k] = sum_{n in block b} dec(dyq[i,n]) * dec(wq[k,n]).
 * dyq: [M x N] row stride lddy; sdy(i, b) = sdy[i * sdy_rs + b * sdy_ts].
 * wq: [K x N] row stride ldw; sw(bk, bn) = sw[bk * ldsw + bn].
 * Output index (i, k) over M x K. */
void oracle_dgrad(const uint8_t* dyq, i64 lddy, const float* sdy, i64 sdy_rs, i64 sdy_ts,
                  const uint8_t* wq, i64 ldw, const float* sw, i64 ldsw,
                  i64 M, i64 N, i64 K, const i64* ii, const i64* kk, i64 n_out,
                  float* out)
{
    build_table();
    i64 total = ii ? n_out : M * K;
#pragma omp parallel for schedule(dynamic, 64)
    for (i64 e = 0; e < total; ++e) {
        i64 i = ii ? ii[e] : e / K;
        i64 k = ii ? kk[e] : e % K;
        out[e] = promoted_dot(dyq + i * lddy, 1, wq + k * ldw, 1, N,
                              sdy + i * sdy_rs, sdy_ts, sw + (k / 128) * ldsw, 1);
    }
}

/* Wgrad, dW = dY^T X (contraction over tokens), on the 128x1 re-tiled,
 * transposed operands:
 *   dW[n,k] = sum_b s_dyT[b,n] * s_xT[b,k] * P_b[n,k],
 *   P_b[n,k] = sum_{t in block b} dec(dyqT[n,t]) * dec(xqT[k,t]).
 * dyqT: [N x T] row stride lddyT, sdyT(b, n) = sdyT[b * ldsdyT + n].
 * xqT:  [K x T] row stride ldxT,  sxT(b, k) = sxT[b * ldsxT + k].
 * T is the (padded) token count. Output index (n, k) over N x K. */
void oracle_wgrad(const uint8_t* dyqT, i64 lddyT, const float* sdyT, i64 ldsdyT,
                  const uint8_t* xqT, i64 ldxT, const float* sxT, i64 ldsxT,
                  i64 T, i64 N, i64 K, const i64* nn, const i64* kk, i64 n_out,
                  float* out)
{
    build_table();
    i64 total = nn ? n_out : N * K;
#pragma omp parallel for schedule(dynamic, 64)
    for (i64 e = 0; e < total; ++e) {
        i64 n = nn ? nn[e] : e / K;
        i64 k = nn ? kk[e] : e % K;
        out[e] = promoted_dot(dyqT + n * lddyT, 1, xqT + k * ldxT, 1, T,
                              sdyT + n, ldsdyT, sxT + k, ldsxT);
    }
}

/* ------------------------------------------------------------------------- */
/* Reference sums for the pins: fp64 over dequantized operands, and the      */
/* unpromoted low-precision accumulation of the drift model.                 */
/* ------------------------------------------------------------------------- */

/* Round v to m significant bits (m counts the leading bit). mode 0: nearest,
 * ties to even; mode 1: toward zero. No exponent limit (a model of an
 * accumulator's significand width only). */
double oracle_round_sig(double v, int m, int mode)
{
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int e;
    double f = frexp(v, &e);             /* v = f * 2^e, 0.5 <= |f| < 1 */
    double scaled = ldexp(f, m);         /* |scaled| in [2^(m-1), 2^m) */
    double r = (mode == 1) ? trunc(scaled) : nearbyint(scaled);
    return ldexp(r, e - m);
}

/* Fprop element computed two more ways, for the pins:
 *   out_fp64[e]  = sum_k (dec(xq)*s_x) * (dec(wq)*s_w) in fp64 (dequantized truth)
 *   out_unpr[e]  = the drift model with an m-bit accumulator and no promotion:
 *                  s_t = round(s_{t-1} + round(p_t)),
 *                  p_t = dec(xq[i,t]) * dec(wq[t,j]) * (s_x * s_w)   (fp64).
 * Same argument layout as oracle_fprop; element list is required. */
void oracle_fprop_reference_sums(const uint8_t* xq, i64 ldx, const float* sx, i64 sx_rs, i64 sx_ts,
                                 const uint8_t* wq, i64 ldw, const float* sw, i64 ldsw,
                                 i64 K, const i64* ii, const i64* jj, i64 n_out,
                                 int m_bits, int mode, double* out_fp64, double* out_unpr)
{
    build_table();
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 e = 0; e < n_out; ++e) {
        i64 i = ii[e], j = jj[e];
        double truth = 0.0, acc = 0.0;
        for (i64 k = 0; k < K; ++k) {
            double a = (double)g_dec[xq[i * ldx + k]];
            double b = (double)g_dec[wq[k * ldw + j]];
            double s_a = (double)sx[i * sx_rs + (k / 128) * sx_ts];
            double s_b = (double)sw[(k / 128) * ldsw + j / 128];
            truth += (a * s_a) * (b * s_b);
            if (out_unpr) {
                double p = a * b * (double)((float)s_a * (float)s_b);
                acc = oracle_round_sig(acc + oracle_round_sig(p, m_bits, mode), m_bits, mode);
            }
        }
        out_fp64[e] = truth;
        if (out_unpr) out_unpr[e] = acc;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
