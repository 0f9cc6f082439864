// quant.cu -- dynamic absmax quantizers to E4M3 with fp32 scales.
//
// The tile recipe: amax = max |v| over the tile, s = amax / 448 (IEEE fp32
// division; 1 for an all-zero tile), q = E4M3 round-to-nearest-even,
// saturating, of the fp32 quotient v / s. Source: "FP8 动态量化里的 partial sum
// 漂移", section 3, row (a) (per-tile dynamic scales from the absmax, N_c = 128);
// tile shapes from "scratch: the backward pass, unrolled", "What is asserted,
// and from where" (1x128 activations and gradients, 128x128 weights, 128x1
// re-tiling for Wgrad). E4M3 -0 (0x80) is kept apart from +0 (prime-rl PR
// #4073, conventions table, row "Negative zero"): the E4M3 conversion keeps
// the sign of a result that rounds to zero, so every code carries the sign
// of its input (the parity tests include tiles of tiny negatives).
//
// All three kernels are HBM streams: 16-byte vector loads, warp-shuffle
// absmax reductions, coalesced payload and scale stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Largest |bf16| of the four words' halves, as bf16 magnitude bits in [0, 0x7FFF].
// For finite values the magnitude bit patterns order like the values.
__device__ __forceinline__ uint32_t absmax_bits_8(const uint4& d)
{
    uint32_t m = __vmaxu2(__vmaxu2(d.x & 0x7FFF7FFFu, d.y & 0x7FFF7FFFu),
                          __vmaxu2(d.z & 0x7FFF7FFFu, d.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16);
}

// Smallest power of two >= s, for s > 0 (normal or subnormal).
__device__ __forceinline__ float pow2_ceil(float s)
{
    const uint32_t b = __float_as_uint(s);
    if ((b & 0x007FFFFFu) == 0u) return s;                              // already 2^e
    if ((b >> 23) != 0u) return __uint_as_float((b & 0x7F800000u) + 0x00800000u);
    return __uint_as_float(1u << (32 - __clz(b - 1u)));                 // subnormal
}

// Scale of a tile from its absmax. Default rule: s = amax / 448 (IEEE fp32
// division), 1 for an all-zero tile. Options (prime-rl PR #4073, conventions
// table, rows "Weight floors", "Two-stage weights", "Activation floors",
// "Compact formats"): an amax floor applied before the division, a scale
// floor applied after it (a zero tile then gets the floored scale instead of
// 1), and UE8M0 rounding of s up to a power of two, so that amax / s stays
// <= 448 and every scale is an exponent byte.
__device__ __forceinline__ float scale_from_amax(float amax, const ScaleRule& r)
{
    const float a = fmaxf(amax, r.amax_floor);
    float s = (a == 0.0f && r.scale_floor == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
    s = fmaxf(s, r.scale_floor);
    return r.ue8m0 ? pow2_ceil(s) : s;
}

// E4M3 codes of fp32(v / s) for a pair of values, by exact IEEE division.
// Used only for tiles whose scale lies outside the fast path's range (below
// 2^-60 or above 2^100); kept out of line so that it does not weigh on the
// fast path's code.
__device__ __noinline__ uint32_t encode2_exact(float v0, float v1, float s)
{
    return cvt_e4m3x2(__fdiv_rn(v0, s), __fdiv_rn(v1, s));
}

// Quotients fp32(v / s) of a pair of values without a division, encoded to
// E4M3; the result is the correctly rounded quotient RN(v / s) for every
// input, so the codes equal those of an IEEE division.
//
// With r = RN(1/s) (within half an ulp of 1/s):
//   q0 = RN(v r)                    within 1.5 ulp of v/s;
//   q1 = RN(q0 + (v - q0 s) r)      the residual v - q0 s is exact in one FMA,
//                                   and q1 is within 1/2 ulp + 2^-23 ulp of
//                                   v/s, hence a faithful approximation;
//   q2 = RN(q1 + (v - q1 s) r)      = RN(v/s) by Markstein's theorem (a
//                                   faithful quotient corrected once with an
//                                   exact FMA residual and a reciprocal within
//                                   half an ulp is correctly rounded; IBM J.
//                                   Res. Dev. 34(1), 1990).
// The theorem assumes no underflow; quotients small enough to underflow are
// far below 2^-10 and encode to a signed zero whatever their rounding. The
// caller keeps s in [2^-60, 2^100] (other tiles take exact division) so the
// reciprocal and the residuals stay normal.
//
// The steps take the negated inputs nv = -v and nr = -r and form the negated
// residuals (q s - v): a zero input then keeps its sign through the chain
// (v = -0 gives q = -0 + -0), where the textbook order would turn it into
// +0. The E4M3 conversion keeps the sign of a zero result, so -0 inputs and
// tiny negatives encode to 0x80. Pairs use the packed fp32x2 instructions.
__device__ __forceinline__ uint32_t encode2_fast(float2 nv, float s, float nr)
{
    const float2 s2 = make_float2(s, s);
    const float2 nr2 = make_float2(nr, nr);
    const float2 q0 = __fmul2_rn(nv, nr2);
    const float2 q1 = __ffma2_rn(__ffma2_rn(q0, s2, nv), nr2, q0);
    const float2 q2 = __ffma2_rn(__ffma2_rn(q1, s2, nv), nr2, q1);
    return cvt_e4m3x2(q2.x, q2.y);
}

// Negated bf16 halves of a word as fp32: -lo is (w << 16) with its top bit
// flipped, which one integer multiply-add gives (adding 2^31 flips bit 31).
__device__ __forceinline__ float neg_bf16_lo(uint32_t w)
{
    uint32_t r;
    asm("mad.lo.u32 %0, %1, 65536, 0x80000000;" : "=r"(r) : "r"(w));
    return __uint_as_float(r);
}

__device__ __forceinline__ float neg_bf16_hi(uint32_t w)
{
    return __uint_as_float((w & 0xFFFF0000u) ^ 0x80000000u);
}

__device__ __forceinline__ float2 neg_bf16x2(uint32_t w)
{
    return make_float2(neg_bf16_lo(w), neg_bf16_hi(w));
}

// Scale of a tile: s and the negated reciprocal for the fast path (nr = 0
// when s is outside [2^-60, 2^100] and only the exact path may be used).
struct TileScale {
    float s;
    float nr;
};

__device__ __forceinline__ TileScale tile_scale_from_s(float s)
{
    TileScale t;
    t.s = s;
    t.nr = (s >= 0x1p-60f && s <= 0x1p100f) ? -__frcp_rn(s) : 0.0f;
    return t;
}

__device__ __forceinline__ TileScale tile_scale(float amax, const ScaleRule& r)
{
    return tile_scale_from_s(scale_from_amax(amax, r));
}

__device__ __noinline__ uint2 quant8_exact(uint4 d, float s)
{
    uint2 o;
    o.x = encode2_exact(bf16_lo(d.x), bf16_hi(d.x), s) | (encode2_exact(bf16_lo(d.y), bf16_hi(d.y), s) << 16);
    o.y = encode2_exact(bf16_lo(d.z), bf16_hi(d.z), s) | (encode2_exact(bf16_lo(d.w), bf16_hi(d.w), s) << 16);
    return o;
}

// Eight bf16 values (one 16-byte load) divided by s and encoded, low
// element first. Tiles whose scale is outside the fast path's range (nr = 0)
// use exact division.
__device__ __forceinline__ uint2 quant8(const uint4& d, const TileScale& t)
{
    if (t.nr == 0.0f) return quant8_exact(d, t.s);
    const uint32_t c0 = encode2_fast(neg_bf16x2(d.x), t.s, t.nr);
    const uint32_t c1 = encode2_fast(neg_bf16x2(d.y), t.s, t.nr);
    const uint32_t c2 = encode2_fast(neg_bf16x2(d.z), t.s, t.nr);
    const uint32_t c3 = encode2_fast(neg_bf16x2(d.w), t.s, t.nr);
    return make_uint2(__byte_perm(c0, c1, 0x5410), __byte_perm(c2, c3, 0x5410));
}

// ---------------------------------------------------------------------------
// Stochastic rounding. The random word of element idx (its linear
// index in the quantized tensor) under (seed, salt) is word idx % 4 of
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011) with key (seed low,
// seed high) and counter (idx / 4 low, idx / 4 high, salt, 0): stateless,
// independent of launch shape. The quotient x = RN(v / s) then rounds to the
// upper E4M3 neighbour when the 20-bit fraction of its position between the
// two neighbours exceeds the word's top 20 bits (probability = the fraction),
// else to the lower one; |x| >= 448 gives 448; signs (and signed zeros) are
// kept.
// ---------------------------------------------------------------------------
struct SrKey {
    uint64_t seed;
    uint32_t salt;
};

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                               uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Words of elements 4 blk .. 4 blk + 3.
__device__ __forceinline__ uint4 sr_words(const SrKey& k, uint64_t blk)
{
    return philox4x32_10(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), k.salt, 0u,
                         static_cast<uint32_t>(k.seed), static_cast<uint32_t>(k.seed >> 32));
}

// E4M3 code of the fp32 quotient x, stochastically rounded with word r.
__device__ __forceinline__ uint32_t sr_code(float x, uint32_t r)
{
    const uint32_t b = __float_as_uint(x);
    const uint32_t sign = (b >> 24) & 0x80u;
    const uint32_t a = b & 0x7FFFFFFFu;
    const uint32_t r20 = r >> 12;
    if (a >= 0x43E00000u) return sign | 0x7Eu;                // |x| >= 448
    if (a >= 0x3C800000u) {                                    // E4M3 normal range, |x| >= 2^-6
        const uint32_t code = (((a >> 23) - 120u) << 3) | ((a >> 20) & 7u);
        return sign | (code + ((a & 0xFFFFFu) > r20 ? 1u : 0u));
    }
    const float t = __uint_as_float(a) * 512.0f;               // position on the 2^-9 grid (exact)
    const uint32_t n = static_cast<uint32_t>(t);
    const uint32_t f20 = static_cast<uint32_t>((t - static_cast<float>(n)) * 1048576.0f);
    return sign | (n + (f20 > r20 ? 1u : 0u));
}

// Quotients RN(v / s) of a pair (negated inputs, as encode2_fast) without
// the conversion.
__device__ __forceinline__ float2 quotient2(float2 nv, float s, float nr)
{
    const float2 s2 = make_float2(s, s);
    const float2 nr2 = make_float2(nr, nr);
    const float2 q0 = __fmul2_rn(nv, nr2);
    const float2 q1 = __ffma2_rn(__ffma2_rn(q0, s2, nv), nr2, q0);
    return __ffma2_rn(__ffma2_rn(q1, s2, nv), nr2, q1);
}

// Eight bf16 values with stochastic rounding; words w[0..7] for elements
// 0..7 of the group.
__device__ __forceinline__ uint2 quant8_sr(const uint4& d, const TileScale& t, const uint32_t (&w)[8])
{
    const uint32_t wd[4] = {d.x, d.y, d.z, d.w};
    uint32_t c[8];
    if (t.nr == 0.0f) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            c[2 * k] = sr_code(__fdiv_rn(bf16_lo(wd[k]), t.s), w[2 * k]);
            c[2 * k + 1] = sr_code(__fdiv_rn(bf16_hi(wd[k]), t.s), w[2 * k + 1]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 qq = quotient2(neg_bf16x2(wd[k]), t.s, t.nr);
            c[2 * k] = sr_code(qq.x, w[2 * k]);
            c[2 * k + 1] = sr_code(qq.y, w[2 * k + 1]);
        }
    }
    return make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24),
                      c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
}

// Random words of the 8 consecutive elements starting at idx (idx % 8 == 0).
__device__ __forceinline__ void sr_words8(const SrKey& k, uint64_t idx, uint32_t (&w)[8])
{
    const uint4 a = sr_words(k, idx >> 2), b = sr_words(k, (idx >> 2) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// ---------------------------------------------------------------------------
// S1: 1x128 tiles. One warp handles 32 rows x one 128-column tile: each
// half-warp reads one row's 256 bytes per load (16 lanes x 16 bytes), so a
// warp covers two rows per instruction and 32 rows in 16 loads, all issued
// before any arithmetic. Lane l ends up holding the scale of row l, so the
// warp stores its 32 scales as one 128-byte segment.
// ---------------------------------------------------------------------------
constexpr int kQ1Threads = 256;

template <bool kSR>
__global__ void __launch_bounds__(kQ1Threads) quant_1x128_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
    uint8_t* __restrict__ q, float* __restrict__ scales, int64_t scale_ld, const ScaleRule rule,
    const SrKey sr)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int l16 = lane & 15;
    const int64_t col_tiles = (cols + 127) / 128;
    const int64_t row_groups = (rows + 31) / 32;
    const int64_t units = col_tiles * row_groups;
    const int64_t warps_total = (int64_t)gridDim.x * (kQ1Threads / 32);
    int64_t unit = (int64_t)blockIdx.x * (kQ1Threads / 32) + (threadIdx.x >> 5);

    for (; unit < units; unit += warps_total) {
        const int64_t rg = unit / col_tiles;
        const int64_t tc = unit - rg * col_tiles;
        const int64_t col = tc * 128 + l16 * 8;
        const bool col_ok = col < cols;  // cols % 16 == 0: 8-column chunks are all-in or all-out
        const int64_t row0 = rg * 32;

        uint4 d[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int64_t r = row0 + 2 * i + half;
            if (col_ok && r < rows)
                d[i] = __ldcs(reinterpret_cast<const uint4*>(x + r * ldx + col));
            else
                d[i] = make_uint4(0u, 0u, 0u, 0u);
        }

        // Per-row absmax by a reduce-scatter butterfly inside each half-warp:
        // at each level a lane swaps half of its running maxima with the lane
        // `off` away and keeps the half selected by its own lane bit, so after
        // four levels lane (h, j) holds the absmax of row 2j + h (15 shuffles
        // instead of a separate 4-shuffle reduction per row pair).
        const int lh = lane & 15;
        uint32_t m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) m[i] = absmax_bits_8(d[i]);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
            const bool upper = (lh & off) != 0;
#pragma unroll
            for (int j = 0; j < off; ++j) {
                const uint32_t send = upper ? m[j] : m[j + off];
                const uint32_t keep = upper ? m[j + off] : m[j];
                m[j] = max(keep, __shfl_xor_sync(0xFFFFFFFFu, send, off));
            }
        }
        const float amax_mine = __uint_as_float(m[0] << 16);
        const int my_row = 2 * lh + half;
        // one scale (and reciprocal) per lane: lane (h, j) owns row 2j + h
        const TileScale mine = tile_scale(amax_mine, rule);
        if (row0 + my_row < rows) scales[tc * scale_ld + row0 + my_row] = mine.s;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int src = (lane & 16) | i;    // the lane holding row 2i + h
            TileScale ts;
            ts.s = __shfl_sync(0xFFFFFFFFu, mine.s, src);
            ts.nr = __shfl_sync(0xFFFFFFFFu, mine.nr, src);
            const int64_t r = row0 + 2 * i + half;
            if constexpr (kSR) {
                if (col_ok && r < rows) {
                    uint32_t w[8];
                    sr_words8(sr, static_cast<uint64_t>(r * cols + col), w);
                    *reinterpret_cast<uint2*>(q + r * cols + col) = quant8_sr(d[i], ts, w);
                }
            } else {
                if (col_ok && r < rows) *reinterpret_cast<uint2*>(q + r * cols + col) = quant8(d[i], ts);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// S1, streamed (round to nearest): the same tile recipe as
// quant_1x128_kernel with lane = row. A persistent grid (one CTA of eight
// warps per SM) walks 32-row x 128-column units; each warp keeps its next
// units in flight in shared-memory slots of its own (two 64-column TMA boxes
// per unit, 128-byte swizzled so that a lane reading its own row's 16-byte
// chunks hits every bank once per eight lanes), copies a unit into
// registers, refills the slot at once and then encodes. With one row per
// lane the absmax, the scale and the reciprocal are per thread and the
// whole row shares them: no shuffles. The codes go back through a per-warp
// 4 KB stage (same swizzle) and leave with one TMA store per unit. Rows and
// columns outside the tensor arrive as zeros (the load map's out-of-bounds
// fill) and are not stored (the store map clips them).
// ---------------------------------------------------------------------------
constexpr int kQ1sWarps = 8;
constexpr int kQ1sSlots = 3;
constexpr int kQ1sUnitBytes = 32 * 128 * 2;
constexpr int kQ1sOutBytes = 32 * 128;
constexpr int kQ1sWarpBytes = kQ1sSlots * kQ1sUnitBytes + kQ1sOutBytes;
constexpr uint64_t kQ1sDrainNs = 1000000000ull;

__global__ void __launch_bounds__(kQ1sWarps * 32, 1) quant_1x128_stream_kernel(
    const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_q, int64_t rows,
    int64_t cols, float* __restrict__ scales, int64_t scale_ld, const ScaleRule rule, uint64_t limit,
    unsigned int* status)
{
    extern __shared__ uint8_t q1s_smem_raw[];
    __shared__ uint64_t full[kQ1sWarps][kQ1sSlots];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(q1s_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* wsm = smem + warp * kQ1sWarpBytes;              // the warp's slots, then its code stage
    const uint32_t slots = smem_addr(wsm);
    const uint32_t stage = slots + kQ1sSlots * kQ1sUnitBytes;
    const uint32_t sw = static_cast<uint32_t>(lane & 7);     // 128-byte swizzle of this lane's row
    const int64_t col_tiles = (cols + 127) / 128;
    const int64_t units = col_tiles * ((rows + 31) / 32);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kQ1sWarps;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kQ1sWarps + warp;

    auto issue = [&](int64_t unit, int slot) {
        const int64_t rg = unit / col_tiles;
        const int64_t tc = unit - rg * col_tiles;
        uint8_t* dst = wsm + slot * kQ1sUnitBytes;
        mbar_arrive_expect_tx(&full[warp][slot], kQ1sUnitBytes);
        tma_load_2d(dst, &map_x, &full[warp][slot], static_cast<int32_t>(tc * 128), static_cast<int32_t>(rg * 32));
        tma_load_2d(dst + kQ1sUnitBytes / 2, &map_x, &full[warp][slot], static_cast<int32_t>(tc * 128 + 64),
                    static_cast<int32_t>(rg * 32));
    };
    if (lane == 0) {
        for (int j = 0; j < kQ1sSlots; ++j) mbar_init(&full[warp][j], 1);
        fence_mbarrier_init();
        if (warp == 0) {
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_q);
        }
        for (int j = 0; j < kQ1sSlots; ++j)
            if (first + j * stride < units) issue(first + j * stride, j);
    }
    __syncwarp();

    int k = 0;
    for (int64_t unit = first; unit < units; unit += stride, ++k) {
        const int slot = k % kQ1sSlots;
        // lane 0 waits (bounded) and the warp follows its verdict; the other
        // lanes then pass the completed phase themselves (acquire)
        int landed = 0;
        if (lane == 0) landed = mbar_wait(&full[warp][slot], (k / kQ1sSlots) & 1, limit) ? 1 : 0;
        landed = __shfl_sync(0xFFFFFFFFu, landed, 0);
        if (landed) mbar_try_wait(&full[warp][slot], (k / kQ1sSlots) & 1);
        if (!landed) {
            // a load did not land in time: record it, let every issued box
            // land and every store finish before the CTA leaves, and stop
            if (lane == 0) {
                atomicCAS(status, 0u, static_cast<unsigned int>(FP8BS_ERR_TIMEOUT));
                const uint64_t drain = limit > kQ1sDrainNs ? limit : kQ1sDrainNs;
                for (int j = k; j < k + kQ1sSlots && first + j * stride < units; ++j)
                    mbar_wait(&full[warp][j % kQ1sSlots], (j / kQ1sSlots) & 1, drain);
                bulk_wait_group_all();
            }
            __syncwarp();
            return;
        }
        const int64_t rg = unit / col_tiles;
        const int64_t tc = unit - rg * col_tiles;
        const int64_t row = rg * 32 + lane;

        // this lane's row: chunk c of the first box (columns 8c .. 8c + 7)
        // at slot + 128 lane + 16 (c ^ lane % 8), the second box 4 KB on
        uint4 d[16];
        const uint32_t rowp = slots + slot * kQ1sUnitBytes + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            d[c] = ld_shared_v4(rowp + ((c ^ sw) << 4));
            d[8 + c] = ld_shared_v4(rowp + kQ1sUnitBytes / 2 + ((c ^ sw) << 4));
        }
        // every lane has read the slot: refill it with the unit after next
        __syncwarp();
        if (lane == 0) {
            const int64_t nxt = unit + kQ1sSlots * stride;
            if (nxt < units) {
                fence_proxy_async_smem();
                issue(nxt, slot);
            }
        }

        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = max(m, absmax_bits_8(d[i]));
        const TileScale ts = tile_scale(__uint_as_float(m << 16), rule);
        if (row < rows) scales[tc * scale_ld + row] = ts.s;

        // the previous unit's store has read the stage
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        const uint32_t outp = stage + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint2 a = quant8(d[2 * j], ts);
            const uint2 b = quant8(d[2 * j + 1], ts);
            st_shared_v4(outp + ((j ^ sw) << 4), make_uint4(a.x, a.y, b.x, b.y));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(&map_q, stage, static_cast<int32_t>(tc * 128), static_cast<int32_t>(rg * 32));
            bulk_commit_group();
        }
    }
    // the warp's stores have completed before the CTA exits
    if (lane == 0) bulk_wait_group_all();
}

// ---------------------------------------------------------------------------
// S2: 128x128 blocks. One CTA of 256 threads per block: thread t reads the
// 8-column chunk t % 16 of rows t / 16 + 16 i (i < 8), so each row's 256
// bytes come from 16 consecutive threads. Block absmax via warp shuffles and
// shared memory. The optional transposed payload goes through a padded
// shared-memory tile and leaves as 16-byte row segments of qT. With atoms
// (power-of-two scales), the block's exponent byte also fills one 512-byte
// scale atom of each of the two GEMM operands the weight feeds.
// ---------------------------------------------------------------------------
constexpr int kQ2Threads = 256;
constexpr int kQ2Pitch = 132;  // bytes per row of the staging tile (bank-conflict padding)

template <bool kSR>
__global__ void __launch_bounds__(kQ2Threads, 4) quant_128x128_kernel(
    const uint16_t* __restrict__ w, int64_t rows, int64_t cols, int64_t ldw,
    uint8_t* __restrict__ q, uint8_t* __restrict__ qT, float* __restrict__ scales, const ScaleRule rule,
    const SrKey sr, uint8_t* __restrict__ atoms_wT, uint8_t* __restrict__ atoms_w, unsigned int* status)
{
    __shared__ uint32_t red[kQ2Threads / 32];
    __shared__ __align__(16) uint8_t tile[128 * kQ2Pitch];

    const int64_t nbr = (rows + 127) / 128, nbc = (cols + 127) / 128;
    const int64_t blk = blockIdx.x;
    const int64_t b = blk / (nbr * nbc);
    const int64_t rem = blk - b * nbr * nbc;
    const int64_t bi = rem / nbc, bj = rem - bi * nbc;
    const int64_t r0 = bi * 128, c0 = bj * 128;
    const uint16_t* wb = w + b * rows * ldw;

    const int chunk = threadIdx.x & 15;
    const int rgrp = threadIdx.x >> 4;
    const int64_t col = c0 + chunk * 8;
    const bool col_ok = col < cols;

    uint4 d[8];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + rgrp + 16 * i;
        if (col_ok && r < rows)
            d[i] = __ldcs(reinterpret_cast<const uint4*>(wb + r * ldw + col));
        else
            d[i] = make_uint4(0u, 0u, 0u, 0u);
        m = max(m, absmax_bits_8(d[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int i = 0; i < kQ2Threads / 32; ++i) m = max(m, red[i]);
    const TileScale ts = tile_scale(__uint_as_float(m << 16), rule);
    if (threadIdx.x == 0) scales[b * nbr * nbc + bi * nbc + bj] = ts.s;
    if (atoms_wT != nullptr && threadIdx.x < 64) {
        // the block's exponent byte fills one whole atom of each operand:
        // W^T (rows = the block's 128 columns, K-block bi) and W (rows =
        // its 128 rows, K-block bj); 16 bytes per thread
        const uint32_t E = ue8m0_of(ts.s);
        if (E == 255u && threadIdx.x == 0) atomicCAS(status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
        const uint32_t e4 = E * 0x01010101u;
        const int64_t bo = b * nbr * nbc * 512;
        uint8_t* atom = threadIdx.x < 32 ? atoms_wT + bo + (bj * nbr + bi) * 512
                                         : atoms_w + bo + (bi * nbc + bj) * 512;
        *reinterpret_cast<uint4*>(atom + 16 * (threadIdx.x & 31)) = make_uint4(e4, e4, e4, e4);
    }

    uint8_t* qb = q + b * rows * cols;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rl = rgrp + 16 * i;
        const int64_t r = r0 + rl;
        uint2 out;
        if constexpr (kSR) {
            uint32_t wr[8];
            sr_words8(sr, static_cast<uint64_t>(b * rows * cols + r * cols + col), wr);
            out = quant8_sr(d[i], ts, wr);
        } else {
            out = quant8(d[i], ts);
        }
        if (col_ok && r < rows) *reinterpret_cast<uint2*>(qb + r * cols + col) = out;
        if (qT != nullptr) {
            uint32_t* tp = reinterpret_cast<uint32_t*>(tile + rl * kQ2Pitch + chunk * 8);
            tp[0] = out.x;
            tp[1] = out.y;
        }
    }
    if (qT == nullptr) return;
    __syncthreads();
    // qT[b][c][r]: unit = (column j of the block, 16-row segment m)
    uint8_t* qTb = qT + b * rows * cols;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int unit = threadIdx.x + u * kQ2Threads;  // 0..1023
        const int j = unit & 127;
        const int seg = unit >> 7;                       // 0..7
        const int64_t c = c0 + j;
        const int64_t rr = r0 + seg * 16;
        if (c < cols && rr < rows) {  // rows % 16 == 0: segments are all-in or all-out
            uint32_t wv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t acc = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc |= static_cast<uint32_t>(tile[(seg * 16 + 4 * k + e) * kQ2Pitch + j])
                           << (8 * e);
                wv[k] = acc;
            }
            *reinterpret_cast<uint4*>(qTb + c * rows + rr) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
    }
}

// ---------------------------------------------------------------------------
// S3: 128x1 tiles along tokens, transposed output. One CTA per (padded token
// tile, 128-channel block). Phase 1 stages the source block in shared memory
// (coalesced along channels) and keeps per-thread partial column maxima;
// phase 2 reduces them to one scale per channel; phase 3 reads each channel's
// 128 tokens down the staged block and writes them as one 128-byte row of qT.
// ---------------------------------------------------------------------------
constexpr int kQ3Threads = 256;

// Mode B, phase 3 for one channel pair (j, j + 1) and 32 tokens of the staged
// BF16 block [128 tokens x 128 channels]: each 32-bit shared load holds both
// channels of one token. Returns false when a channel's scale is outside the
// fast path's range; the caller then redoes the pair with exact division.
__device__ __forceinline__ bool requant_pair_bf16(const uint8_t* stage, int part, int j,
                                                  const TileScale& t0, const TileScale& t1,
                                                  uint32_t (&w0)[8], uint32_t (&w1)[8])
{
    uint32_t bad = (t0.nr == 0.0f || t1.nr == 0.0f) ? 1u : 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            x[e] = *reinterpret_cast<const uint32_t*>(stage + ((part * 32 + 4 * k + e) * 128 + j) * 2);
        const uint32_t a01 = encode2_fast(make_float2(neg_bf16_lo(x[0]), neg_bf16_lo(x[1])), t0.s, t0.nr);
        const uint32_t a23 = encode2_fast(make_float2(neg_bf16_lo(x[2]), neg_bf16_lo(x[3])), t0.s, t0.nr);
        const uint32_t b01 = encode2_fast(make_float2(neg_bf16_hi(x[0]), neg_bf16_hi(x[1])), t1.s, t1.nr);
        const uint32_t b23 = encode2_fast(make_float2(neg_bf16_hi(x[2]), neg_bf16_hi(x[3])), t1.s, t1.nr);
        w0[k] = __byte_perm(a01, a23, 0x5410);
        w1[k] = __byte_perm(b01, b23, 0x5410);
    }
    return bad == 0u;
}

// Exact-division version of requant_pair_bf16 that stores its results
// itself (kept out of line; it runs only when the fast path reports a
// quotient near an E4M3 rounding boundary).
__device__ __noinline__ void requant_pair_bf16_exact(const uint8_t* stage, int part, int j, float s0,
                                                     float s1, uint8_t* dst0, uint8_t* dst1)
{
    for (int k = 0; k < 8; ++k) {
        uint32_t x[4];
        for (int e = 0; e < 4; ++e)
            x[e] = *reinterpret_cast<const uint32_t*>(stage + ((part * 32 + 4 * k + e) * 128 + j) * 2);
        reinterpret_cast<uint32_t*>(dst0)[k] =
            encode2_exact(bf16_lo(x[0]), bf16_lo(x[1]), s0) | (encode2_exact(bf16_lo(x[2]), bf16_lo(x[3]), s0) << 16);
        reinterpret_cast<uint32_t*>(dst1)[k] =
            encode2_exact(bf16_hi(x[0]), bf16_hi(x[1]), s1) | (encode2_exact(bf16_hi(x[2]), bf16_hi(x[3]), s1) << 16);
    }
}

// Decoded values of the four E4M3 codes in x (channel c = byte c), each
// multiplied by the token's 1x128 scale in fp32 (the fast path passes the
// negated scale, which negates the products exactly).
__device__ __forceinline__ void decode4_scaled(uint32_t x, float s1, float (&v)[4])
{
    const float2 a = e4m3x2_to_f32(static_cast<uint16_t>(x & 0xFFFFu));
    const float2 b = e4m3x2_to_f32(static_cast<uint16_t>(x >> 16));
    v[0] = __fmul_rn(a.x, s1);
    v[1] = __fmul_rn(a.y, s1);
    v[2] = __fmul_rn(b.x, s1);
    v[3] = __fmul_rn(b.y, s1);
}

// Mode Q, phase 3 for one channel quad (j .. j + 3) and 16 tokens of the
// staged E4M3 block: each 32-bit shared load holds the quad of one token.
// Returns false when a channel's scale is outside the fast path's range.
__device__ __forceinline__ bool requant_quad_e4m3(const uint8_t* stage, const float* row_scale,
                                                  int part, int j, const TileScale (&ts)[4],
                                                  uint32_t (&w)[4][4])
{
    uint32_t bad = (ts[0].nr == 0.0f || ts[1].nr == 0.0f || ts[2].nr == 0.0f || ts[3].nr == 0.0f) ? 1u : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t x[4];
        float nv[4][4];   // [token][channel], negated
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int rl = part * 16 + 4 * k + e;
            x[e] = *reinterpret_cast<const uint32_t*>(stage + rl * 128 + j);
            decode4_scaled(x[e], -row_scale[rl], nv[e]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t c01 = encode2_fast(make_float2(nv[0][c], nv[1][c]), ts[c].s, ts[c].nr);
            const uint32_t c23 = encode2_fast(make_float2(nv[2][c], nv[3][c]), ts[c].s, ts[c].nr);
            w[c][k] = __byte_perm(c01, c23, 0x5410);
        }
    }
    return bad == 0u;
}

// Exact-division version of requant_quad_e4m3 that stores its results
// itself (channel c goes to dst + c * mpad).
__device__ __noinline__ void requant_quad_e4m3_exact(const uint8_t* stage, const float* row_scale,
                                                     int part, int j, float s0, float s1, float s2,
                                                     float s3, uint8_t* dst, int64_t mpad)
{
    const float sc[4] = {s0, s1, s2, s3};
    for (int k = 0; k < 4; ++k) {
        uint32_t x[4];
        float v[4][4];
        for (int e = 0; e < 4; ++e) {
            const int rl = part * 16 + 4 * k + e;
            x[e] = *reinterpret_cast<const uint32_t*>(stage + rl * 128 + j);
            decode4_scaled(x[e], row_scale[rl], v[e]);
        }
        for (int c = 0; c < 4; ++c)
            reinterpret_cast<uint32_t*>(dst + c * mpad)[k] =
                encode2_exact(v[0][c], v[1][c], sc[c]) | (encode2_exact(v[2][c], v[3][c], sc[c]) << 16);
    }
}

// Stochastic-rounding versions of the two transposed passes above. Source
// element (token r, channel c) takes word (r * cols + c) % 4 of
// sr_words(key, (r * cols + c) / 4); tok0 is the source row of the part's
// first token, cg the source column of channel j. The quotient is the same
// correctly rounded fp32 v / s as in the nearest-rounding path (or an IEEE
// division for scales outside its range), then rounded by sr_code.
__device__ __forceinline__ uint32_t word_of(const uint4& r, uint32_t i)
{
    return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}

__device__ __forceinline__ void requant_pair_bf16_sr(const uint8_t* stage, int part, int j, const TileScale& t0,
                                                     const TileScale& t1, const SrKey& key, int64_t tok0,
                                                     int64_t cols, int64_t cg, uint32_t (&w0)[8], uint32_t (&w1)[8])
{
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t x[4];
        uint32_t r0[4], r1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[e] = *reinterpret_cast<const uint32_t*>(stage + ((part * 32 + 4 * k + e) * 128 + j) * 2);
            const uint64_t idx = static_cast<uint64_t>((tok0 + 4 * k + e) * cols + cg);   // even
            const uint4 r = sr_words(key, idx >> 2);
            r0[e] = word_of(r, static_cast<uint32_t>(idx & 3u));
            r1[e] = word_of(r, static_cast<uint32_t>(idx & 3u) + 1u);
        }
        float q0[4], q1[4];
        if (t0.nr != 0.0f && t1.nr != 0.0f) {
            const float2 a01 = quotient2(make_float2(neg_bf16_lo(x[0]), neg_bf16_lo(x[1])), t0.s, t0.nr);
            const float2 a23 = quotient2(make_float2(neg_bf16_lo(x[2]), neg_bf16_lo(x[3])), t0.s, t0.nr);
            const float2 b01 = quotient2(make_float2(neg_bf16_hi(x[0]), neg_bf16_hi(x[1])), t1.s, t1.nr);
            const float2 b23 = quotient2(make_float2(neg_bf16_hi(x[2]), neg_bf16_hi(x[3])), t1.s, t1.nr);
            q0[0] = a01.x; q0[1] = a01.y; q0[2] = a23.x; q0[3] = a23.y;
            q1[0] = b01.x; q1[1] = b01.y; q1[2] = b23.x; q1[3] = b23.y;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                q0[e] = __fdiv_rn(bf16_lo(x[e]), t0.s);
                q1[e] = __fdiv_rn(bf16_hi(x[e]), t1.s);
            }
        }
        w0[k] = sr_code(q0[0], r0[0]) | (sr_code(q0[1], r0[1]) << 8) | (sr_code(q0[2], r0[2]) << 16) |
                (sr_code(q0[3], r0[3]) << 24);
        w1[k] = sr_code(q1[0], r1[0]) | (sr_code(q1[1], r1[1]) << 8) | (sr_code(q1[2], r1[2]) << 16) |
                (sr_code(q1[3], r1[3]) << 24);
    }
}

__device__ __forceinline__ void requant_quad_e4m3_sr(const uint8_t* stage, const float* row_scale, int part,
                                                     int j, const TileScale (&ts)[4], const SrKey& key,
                                                     int64_t tok0, int64_t cols, int64_t cg, uint32_t (&w)[4][4])
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float nv[4][4];   // [token][channel], negated
        uint4 r[4];       // words of the token's four channels (cg % 4 == 0)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int rl = part * 16 + 4 * k + e;
            const uint32_t x = *reinterpret_cast<const uint32_t*>(stage + rl * 128 + j);
            decode4_scaled(x, -row_scale[rl], nv[e]);
            r[e] = sr_words(key, static_cast<uint64_t>((tok0 + 4 * k + e) * cols + cg) >> 2);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float q[4];
            if (ts[c].nr != 0.0f) {
                const float2 a = quotient2(make_float2(nv[0][c], nv[1][c]), ts[c].s, ts[c].nr);
                const float2 b = quotient2(make_float2(nv[2][c], nv[3][c]), ts[c].s, ts[c].nr);
                q[0] = a.x; q[1] = a.y; q[2] = b.x; q[3] = b.y;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) q[e] = __fdiv_rn(-nv[e][c], ts[c].s);
            }
            w[c][k] = sr_code(q[0], word_of(r[0], c)) | (sr_code(q[1], word_of(r[1], c)) << 8) |
                      (sr_code(q[2], word_of(r[2], c)) << 16) | (sr_code(q[3], word_of(r[3], c)) << 24);
        }
    }
}

__device__ __forceinline__ int find_group(const int32_t* tile_start, int ng, int tile)
{
    int lo = 0, hi = ng - 1;  // last g with tile_start[g] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Group of padded token tile `tile` from device offsets (all threads of the
// CTA call it; it ends with a CTA barrier, after which `scratch`, 2 KB of
// shared memory, may be reused). Returns false when the tile lies past the
// groups' padded total, or when the offsets are invalid (off[0] != 0, a
// decrease, a total other than p.rows), which CTA (0, 0) records as
// FP8BS_ERR_DEVICE.
__device__ bool device_group(const RequantParams& p, int tile, int32_t* scratch, int& g, int64_t& r0, int& len)
{
    const int G = p.num_groups;
    int32_t* off = scratch;                    // G + 1 offsets
    int32_t* wsum = scratch + kMaxGroups + 1;  // per-warp tile sums
    int32_t* found = wsum + 8;                 // group of this tile, its first tile
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    for (int i = t; i <= G; i += blockDim.x) off[i] = __ldg(p.off_dev + i);
    if (t == 0) *found = -1;
    __syncthreads();
    int bad = 0, cnt = 0;
    if (t < G) {
        const int n = off[t + 1] - off[t];
        if (n < 0) bad = 1;
        cnt = n < 0 ? 0 : (n + 127) / 128;
    }
    if (t == 0 && (off[0] != 0 || static_cast<int64_t>(off[G]) != p.rows)) bad = 1;
    int inc = cnt;   // inclusive scan of the tile counts over the CTA (one group per thread)
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (lane >= d) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    for (int w = 0; w < warp; ++w) inc += wsum[w];
    const int start = inc - cnt;
    if (t < G && cnt > 0 && start <= tile && tile < inc) {
        found[0] = t;
        found[1] = start;
    }
    bad = __syncthreads_or(bad);
    const int fg = found[0], s0 = found[1];
    bool ok = !bad && fg >= 0;
    if (ok) {
        g = fg;
        r0 = static_cast<int64_t>(off[g]) + static_cast<int64_t>(tile - s0) * 128;
        len = static_cast<int>(min(static_cast<int64_t>(128), static_cast<int64_t>(off[g + 1]) - r0));
    }
    if (bad && t == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicCAS(p.status, 0u, (unsigned)FP8BS_ERR_DEVICE);
    __syncthreads();
    return ok;
}

// kDual: also the 1x128 cast of the same BF16 rows (p.q, p.q_scales).
// kStash (with kDual): the transposed cast is taken from that E4M3 result
// (decoded with its row scale, as the E4M3 source mode does) instead of
// from the BF16 values; the 1x128 codes are staged in place of the source.
// kSR: stochastic rounding of both passes (keys in p).
// p.q_atoms / p.qT_atoms (dense, power-of-two scales): the exponent bytes of
// the row and column scales also go to the scale atoms of q and qT; a CTA's
// rows and channels fill exactly one atom of each, written after the
// scales are in shared memory.
template <bool kDual, bool kStash, bool kSR>
__global__ void __launch_bounds__(kQ3Threads, kSR ? 2 : (kStash ? 3 : 4)) requant_128x1_T_kernel(const __grid_constant__ RequantParams p)
{
    static_assert(kDual || !kStash, "the stash mode is a dual cast");
    // staging: BF16 source 128 x 128 x 2 bytes, or E4M3 128 x 128 bytes + row scales
    __shared__ __align__(16) uint8_t stage[128 * 128 * 2];
    __shared__ float row_scale[128];
    __shared__ float col_part[16][128];
    __shared__ TileScale col_scale[128];   // per channel: s and its negated reciprocal

    const int tile = blockIdx.x;                 // padded token tile
    const int64_t c0 = (int64_t)blockIdx.y * 128;
    int g;
    int64_t r0;
    int len;
    if (p.off_dev) {
        if (!device_group(p, tile, reinterpret_cast<int32_t*>(stage), g, r0, len)) return;
    } else {
        g = find_group(p.tile_start, p.num_groups, tile);
        r0 = (int64_t)p.off[g] + (int64_t)(tile - p.tile_start[g]) * 128;
        len = (int)min((int64_t)128, (int64_t)p.off[g + 1] - r0);
    }
    const int nch = (int)min((int64_t)128, p.cols - c0);

    if (p.mode == FP8BS_SRC_BF16) {
        // thread: 8-channel chunk t % 16, rows (t / 16) * 8 .. + 7
        const int chunk = threadIdx.x & 15;
        const int rg = threadIdx.x >> 4;
        const bool ch_ok = chunk * 8 < nch;
        const uint16_t* src = static_cast<const uint16_t*>(p.src);
        uint4 d[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rl = rg * 8 + i;
            if (ch_ok && rl < len)
                d[i] = __ldcs(reinterpret_cast<const uint4*>(src + (r0 + rl) * p.cols + c0 + chunk * 8));
            else
                d[i] = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (!kStash) *reinterpret_cast<uint4*>(stage + (rl * 128 + chunk * 8) * 2) = d[i];
        }
        float cm[8];   // kStash: column maxima of the decoded 1x128 result
#pragma unroll
        for (int e = 0; e < 8; ++e) cm[e] = 0.0f;
        uint32_t mw[4] = {0u, 0u, 0u, 0u};   // otherwise: column maxima of the BF16 magnitudes
        if constexpr (!kStash) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                mw[0] = __vmaxu2(mw[0], d[i].x & 0x7FFF7FFFu);
                mw[1] = __vmaxu2(mw[1], d[i].y & 0x7FFF7FFFu);
                mw[2] = __vmaxu2(mw[2], d[i].z & 0x7FFF7FFFu);
                mw[3] = __vmaxu2(mw[3], d[i].w & 0x7FFF7FFFu);
            }
        }
        if constexpr (kDual) {
            // Row-wise (1x128) cast of the same rows from the registers: a
            // row's 128 channels are the 16 chunks held by 16 consecutive
            // lanes. Their absmax is a reduce-scatter butterfly over those
            // lanes (at xor distances 8, 4, 2 a lane trades half of its
            // running maxima and keeps the half its lane bit selects, then
            // one more step at distance 1), after which lanes 2i and 2i + 1
            // of the group hold row i's absmax. Each lane computes the scale
            // of that one row, and the eight scales (and negated
            // reciprocals) are then read back from their owners.
            uint32_t rm[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) rm[i] = absmax_bits_8(d[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool up = (chunk & 8) != 0;
                const uint32_t send = up ? rm[j] : rm[j + 4];
                rm[j] = max(up ? rm[j + 4] : rm[j], __shfl_xor_sync(0xFFFFFFFFu, send, 8));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const bool up = (chunk & 4) != 0;
                const uint32_t send = up ? rm[j] : rm[j + 2];
                rm[j] = max(up ? rm[j + 2] : rm[j], __shfl_xor_sync(0xFFFFFFFFu, send, 4));
            }
            {
                const bool up = (chunk & 2) != 0;
                const uint32_t send = up ? rm[0] : rm[1];
                rm[0] = max(up ? rm[1] : rm[0], __shfl_xor_sync(0xFFFFFFFFu, send, 2));
            }
            rm[0] = max(rm[0], __shfl_xor_sync(0xFFFFFFFFu, rm[0], 1));
            const TileScale own = tile_scale(__uint_as_float(rm[0] << 16), p.rule);   // row (chunk >> 1)
            const int group = threadIdx.x & 16;   // first lane of this 16-lane group in the warp
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rl = rg * 8 + i;
                TileScale ts;
                ts.s = __shfl_sync(0xFFFFFFFFu, own.s, group | (2 * i));
                ts.nr = __shfl_sync(0xFFFFFFFFu, own.nr, group | (2 * i));
                if (rl >= len) {
                    if constexpr (kStash) {
                        // padding rows: zero codes and scale, as an E4M3 source stages them
                        *reinterpret_cast<uint2*>(stage + rl * 128 + chunk * 8) = make_uint2(0u, 0u);
                        if (chunk == 0) row_scale[rl] = 0.0f;
                    }
                    continue;
                }
                if (chunk == 0) p.q_scales[(c0 / 128) * p.q_scale_ld + r0 + rl] = ts.s;
                // the row scales go to shared memory for the atom writer below
                // (the stash mode stages them there anyway)
                if constexpr (!kStash)
                    if (chunk == 0 && p.q_atoms != nullptr) row_scale[rl] = ts.s;
                // the row's 8 values: from the registers in the stash mode;
                // otherwise read back from this thread's own stage slot, so
                // that the loaded registers are free after the maxima (four
                // CTAs per SM at 64 registers)
                uint4 di;
                if constexpr (kStash) di = d[i];
                else di = *reinterpret_cast<const uint4*>(stage + (rl * 128 + chunk * 8) * 2);
                uint2 codes;
                if constexpr (kSR) {
                    uint32_t wr[8];
                    sr_words8(SrKey{p.sr_seed, p.sr_salt_rows},
                              static_cast<uint64_t>((r0 + rl) * p.cols + c0 + chunk * 8), wr);
                    codes = quant8_sr(di, ts, wr);
                } else {
                    codes = quant8(di, ts);
                }
                if (ch_ok) *reinterpret_cast<uint2*>(p.q + (r0 + rl) * p.cols + c0 + chunk * 8) = codes;
                if constexpr (kStash) {
                    *reinterpret_cast<uint2*>(stage + rl * 128 + chunk * 8) = codes;
                    if (chunk == 0) row_scale[rl] = ts.s;
                    const uint32_t wv[2] = {codes.x, codes.y};
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float2 lo = e4m3x2_to_f32(static_cast<uint16_t>(wv[k] & 0xFFFFu));
                        const float2 hi = e4m3x2_to_f32(static_cast<uint16_t>(wv[k] >> 16));
                        cm[4 * k + 0] = fmaxf(cm[4 * k + 0], fabsf(__fmul_rn(lo.x, ts.s)));
                        cm[4 * k + 1] = fmaxf(cm[4 * k + 1], fabsf(__fmul_rn(lo.y, ts.s)));
                        cm[4 * k + 2] = fmaxf(cm[4 * k + 2], fabsf(__fmul_rn(hi.x, ts.s)));
                        cm[4 * k + 3] = fmaxf(cm[4 * k + 3], fabsf(__fmul_rn(hi.y, ts.s)));
                    }
                }
            }
        }
        if constexpr (kStash) {
#pragma unroll
            for (int e = 0; e < 8; ++e) col_part[rg][chunk * 8 + e] = cm[e];
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                col_part[rg][chunk * 8 + 2 * k] = __uint_as_float(mw[k] << 16);
                col_part[rg][chunk * 8 + 2 * k + 1] = __uint_as_float(mw[k] & 0xFFFF0000u);
            }
        }
    } else {
        // thread: 16-channel chunk t % 8, rows (t / 8) * 4 .. + 3
        const int chunk = threadIdx.x & 7;
        const int rg = threadIdx.x >> 3;
        const bool ch_ok = chunk * 16 < nch;
        const uint8_t* src = static_cast<const uint8_t*>(p.src);
        const int64_t st = c0 / 128;  // the 1x128 tile of these channels
        float cm[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) cm[e] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rl = rg * 4 + i;
            uint4 d = make_uint4(0u, 0u, 0u, 0u);
            float s1 = 0.0f;
            if (ch_ok && rl < len) {
                d = __ldcs(reinterpret_cast<const uint4*>(src + (r0 + rl) * p.cols + c0 + chunk * 16));
                s1 = __ldg(p.src_scales + st * p.src_scale_ld + r0 + rl);
            }
            *reinterpret_cast<uint4*>(stage + rl * 128 + chunk * 16) = d;
            if (chunk == 0) row_scale[rl] = s1;
            const uint32_t wv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 lo = e4m3x2_to_f32(static_cast<uint16_t>(wv[k] & 0xFFFFu));
                const float2 hi = e4m3x2_to_f32(static_cast<uint16_t>(wv[k] >> 16));
                cm[4 * k + 0] = fmaxf(cm[4 * k + 0], fabsf(__fmul_rn(lo.x, s1)));
                cm[4 * k + 1] = fmaxf(cm[4 * k + 1], fabsf(__fmul_rn(lo.y, s1)));
                cm[4 * k + 2] = fmaxf(cm[4 * k + 2], fabsf(__fmul_rn(hi.x, s1)));
                cm[4 * k + 3] = fmaxf(cm[4 * k + 3], fabsf(__fmul_rn(hi.y, s1)));
            }
        }
        // fold the 32 row groups into 16 partial slots: pairs of neighbouring
        // row groups sit in lanes l and l ^ 8 of the same warp
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            cm[e] = fmaxf(cm[e], __shfl_xor_sync(0xFFFFFFFFu, cm[e], 8));
        }
        if ((rg & 1) == 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) col_part[rg >> 1][chunk * 16 + e] = cm[e];
        }
    }
    __syncthreads();

    if (threadIdx.x < 128) {
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, col_part[i][threadIdx.x]);
        const float s = scale_from_amax(m, p.rule);
        col_scale[threadIdx.x] = tile_scale_from_s(s);
        if (threadIdx.x < nch) p.scT[(int64_t)tile * p.cols + c0 + threadIdx.x] = s;
    }
    __syncthreads();

    // Exponent-byte atoms (dense, power-of-two scales): the CTA's 128 rows
    // fill one 512-byte atom of q (K-block c0 / 128) and its 128 channels one
    // atom of qT (K-block = this token tile). Lane t of the first warp writes
    // rows t, t + 32, t + 64, t + 96 of q's atom as one 16-byte word, lane t
    // of the second warp the same channels of qT's; padding rows and
    // channels past cols hold scale 1.
    if (threadIdx.x < 64 && (threadIdx.x < 32 ? p.q_atoms : p.qT_atoms) != nullptr) {
        const int t = threadIdx.x & 31;
        const bool rows_side = threadIdx.x < 32;
        uint32_t wv[4];
        bool bad = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = t + 32 * k;
            uint32_t E = 127u;
            if (rows_side ? i < len : i < nch) {
                E = ue8m0_of(rows_side ? row_scale[i] : col_scale[i].s);
                bad |= E == 255u;
            }
            wv[k] = E * 0x01010101u;
        }
        if (bad) atomicCAS(p.status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
        uint8_t* atom = rows_side ? p.q_atoms + ((r0 / 128) * (p.cols / 128) + c0 / 128) * 512
                                  : p.qT_atoms + ((c0 / 128) * (p.mpad / 128) + tile) * 512;
        *reinterpret_cast<uint4*>(atom + 16 * t) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }

    if (p.mode == FP8BS_SRC_BF16 && !kStash) {
        // unit = (channel pair 2jp, 2jp + 1; 32-token part): 64 x 4 = 256 units
        const int j = 2 * (threadIdx.x & 63);
        const int part = threadIdx.x >> 6;
        if (j < nch) {   // nch % 16 == 0: pairs are all-in or all-out
            const TileScale t0 = col_scale[j];
            const TileScale t1 = col_scale[j + 1];
            uint8_t* dst0 = p.qT + (c0 + j) * p.mpad + (int64_t)tile * 128 + part * 32;
            uint8_t* dst1 = dst0 + p.mpad;
            uint32_t w0[8], w1[8];
            if constexpr (kSR) {
                requant_pair_bf16_sr(stage, part, j, t0, t1, SrKey{p.sr_seed, p.sr_salt_cols},
                                     r0 + part * 32, p.cols, c0 + j, w0, w1);
                reinterpret_cast<uint4*>(dst0)[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
                reinterpret_cast<uint4*>(dst0)[1] = make_uint4(w0[4], w0[5], w0[6], w0[7]);
                reinterpret_cast<uint4*>(dst1)[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                reinterpret_cast<uint4*>(dst1)[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
            } else if (requant_pair_bf16(stage, part, j, t0, t1, w0, w1)) {
                reinterpret_cast<uint4*>(dst0)[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
                reinterpret_cast<uint4*>(dst0)[1] = make_uint4(w0[4], w0[5], w0[6], w0[7]);
                reinterpret_cast<uint4*>(dst1)[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                reinterpret_cast<uint4*>(dst1)[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
            } else {
                requant_pair_bf16_exact(stage, part, j, t0.s, t1.s, dst0, dst1);
            }
        }
    } else {
        // unit = (channel quad 4jq .. 4jq + 3; 16-token part): 32 x 8 = 256 units
        const int j = 4 * (threadIdx.x & 31);
        const int part = threadIdx.x >> 5;
        if (j < nch) {
            TileScale ts[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) ts[c] = col_scale[j + c];
            uint8_t* dst = p.qT + (c0 + j) * p.mpad + (int64_t)tile * 128 + part * 16;
            uint32_t w[4][4];
            if constexpr (kSR) {
                requant_quad_e4m3_sr(stage, row_scale, part, j, ts, SrKey{p.sr_seed, p.sr_salt_cols},
                                     r0 + part * 16, p.cols, c0 + j, w);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(dst + c * p.mpad) = make_uint4(w[c][0], w[c][1], w[c][2], w[c][3]);
            } else if (requant_quad_e4m3(stage, row_scale, part, j, ts, w)) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(dst + c * p.mpad) = make_uint4(w[c][0], w[c][1], w[c][2], w[c][3]);
            } else {
                requant_quad_e4m3_exact(stage, row_scale, part, j, ts[0].s, ts[1].s, ts[2].s, ts[3].s,
                                        dst, p.mpad);
            }
        }
    }
}


// ---------------------------------------------------------------------------
// Dense dual cast and fused forward cast + stash requant
// with round-to-nearest codes: a persistent kernel, two CTAs of 256 threads
// per SM, each CTA working through 128 x 128 blocks. A block arrives by TMA
// as two boxes of 64 columns x 128 rows (128-byte swizzle: 16-byte chunk c
// of row r at slot c ^ r % 8) into one of two buffers, so the next block
// loads while the current one is worked on.
//
// Row pass: a lane takes one half (64 values) of one row straight from the
// staged block, so the row absmax is in-thread plus one shuffle with the
// lane holding the other half, and each lane encodes its 64 values with the
// row's scale. The 1x128 codes go to a code stage in the same swizzle and
// leave with one TMA store.
//
// Transposed pass: a thread takes a few channels over a part of the block's
// tokens and keeps their values in registers (dual cast: a channel pair of
// BF16 values over 32 tokens; stash cast: a channel quad of the staged codes
// times their row scales, 16 tokens) while the parts' column maxima meet in
// shared memory; 128 threads turn them into the channel scales, and each
// thread then encodes its values and writes its pieces of the qT rows.
//
// The arithmetic is that of requant_128x1_T_kernel (the same scale,
// quotient and decode helpers, in the same order), so the bytes are
// identical; the work split is what differs (no shuffles for the row
// maxima or scales, one decode of the stash per element, loads overlapped
// with the work).
//
// Grouped form (kGrouped: expert groups from host or device offsets): block
// rt of the padded token axis belongs to group g, whose rows start at
// off[g]; the block is read from source row off[g] + 128 (rt - first tile of
// g), and its rows past the group's end (the next group's rows) count as
// zeros: the stash codes of those rows are staged as zeros, the dual cast's
// values are masked, and a group's last block stores only its own rows of
// the 1x128 codes (plain stores, where a whole block leaves with a TMA
// store). The transposed output keeps the padded token index rt.
// ---------------------------------------------------------------------------
constexpr int kDtThreads = 256;
constexpr int kDtXBytes = 128 * 128 * 2;                   // one BF16 block
constexpr int kDtQOff = 2 * kDtXBytes;                     // 1x128 code stage, 128 x 128 bytes
constexpr int kDtCpartOff = kDtQOff + 128 * 128;           // float [8][128] column partial maxima
constexpr int kDtRowScaleOff = kDtCpartOff + 8 * 128 * 4;  // float [128]
constexpr int kDtColTsOff = kDtRowScaleOff + 128 * 4;      // TileScale [128]
constexpr int kDtBarOff = kDtColTsOff + 128 * 8;           // two mbarriers
constexpr int kDtGroupOff = kDtBarOff + 16;                // grouped form: int32 off[257], tile start[257], 8 sums
constexpr int kDtSmemBytes = kDtGroupOff + (2 * (kMaxGroups + 1) + 8) * 4 + 1023;   // + alignment slack
constexpr uint64_t kDtDrainNs = 1000000000ull;

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Group table of the grouped tile kernel in shared memory (all threads of
// the CTA call it; it ends with a CTA barrier): the row offsets off[0..G]
// (host offsets from the parameters, or device offsets) and the first padded
// token block of each group, tstart[0..G] (tstart[G] = the blocks of all
// groups). Returns tstart[G], or 0 when the offsets are invalid (off[0] !=
// 0, a decrease, a total other than p.rows, more blocks than p.mpad holds),
// which CTA 0 records as FP8BS_ERR_DEVICE.
__device__ int dt_group_table(const RequantParams& p, int32_t* off, int32_t* tstart, int32_t* wsum)
{
    const int G = p.num_groups;   // <= kMaxGroups = kDtThreads
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    for (int i = t; i <= G; i += kDtThreads) off[i] = p.off_dev ? __ldg(p.off_dev + i) : p.off[i];
    __syncthreads();
    int bad = 0, cnt = 0;
    if (t < G) {
        const int n = off[t + 1] - off[t];
        if (n < 0) bad = 1;
        cnt = n < 0 ? 0 : (n + 127) / 128;
    }
    if (t == 0 && (off[0] != 0 || static_cast<int64_t>(off[G]) != p.rows)) bad = 1;
    int inc = cnt;   // inclusive scan of the block counts (one group per thread)
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (lane >= d) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    for (int w = 0; w < warp; ++w) inc += wsum[w];
    if (t < G) tstart[t] = inc - cnt;
    if (t == G - 1) tstart[G] = inc;
    bad = __syncthreads_or(bad);
    const int total = tstart[G];
    if (static_cast<int64_t>(total) * 128 > p.mpad) bad = 1;
    if (bad && t == 0 && blockIdx.x == 0) atomicCAS(p.status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
    __syncthreads();
    return bad ? 0 : total;
}

template <bool kStash, bool kGrouped>
__global__ void __launch_bounds__(kDtThreads, 2) dual_tile_kernel(const __grid_constant__ CUtensorMap map_x,
                                                                  const __grid_constant__ CUtensorMap map_q,
                                                                  const __grid_constant__ RequantParams p,
                                                                  int64_t col_tiles, int64_t tiles, uint64_t limit)
{
    extern __shared__ uint8_t dt_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(dt_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t xs0 = smem_addr(smem);         // two buffers of [2 column halves][128 rows][128 bytes]
    const uint32_t qs = xs0 + kDtQOff;            // [128 rows][128 bytes]
    float (*cpart)[128] = reinterpret_cast<float (*)[128]>(smem + kDtCpartOff);
    float* row_scale = reinterpret_cast<float*>(smem + kDtRowScaleOff);
    TileScale* col_ts = reinterpret_cast<TileScale*>(smem + kDtColTsOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDtBarOff);
    int32_t* g_off = reinterpret_cast<int32_t*>(smem + kDtGroupOff);
    int32_t* g_start = g_off + kMaxGroups + 1;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if constexpr (kGrouped) {
        // padded token blocks past the groups' total (device offsets size the
        // grid for the largest total) are skipped
        const int64_t total = dt_group_table(p, g_off, g_start, g_start + kMaxGroups + 1);
        if (total * col_tiles < tiles) tiles = total * col_tiles;
    }

    // first source row of padded token block rt (its group's rows from there on)
    auto src_row = [&](int64_t rt, int& g) -> int64_t {
        if constexpr (kGrouped) {
            int lo = 0, hi = p.num_groups - 1;   // last g with g_start[g] <= rt
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (g_start[mid] <= rt) lo = mid; else hi = mid - 1;
            }
            g = lo;
            return static_cast<int64_t>(g_off[lo]) + (rt - g_start[lo]) * 128;
        } else {
            g = 0;
            return rt * 128;
        }
    };
    auto issue = [&](int64_t tile, int buf) {
        const int64_t rt = tile / col_tiles;
        const int64_t ct = tile - rt * col_tiles;
        int g;
        const int64_t y = src_row(rt, g);
        uint8_t* dst = smem + buf * kDtXBytes;
        mbar_arrive_expect_tx(&full[buf], kDtXBytes);
        tma_load_2d(dst, &map_x, &full[buf], static_cast<int32_t>(ct * 128), static_cast<int32_t>(y));
        tma_load_2d(dst + kDtXBytes / 2, &map_x, &full[buf], static_cast<int32_t>(ct * 128 + 64),
                    static_cast<int32_t>(y));
    };
    if (t == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbarrier_init();
        tma_prefetch_desc(&map_x);
        tma_prefetch_desc(&map_q);
        for (int j = 0; j < 2; ++j)
            if (blockIdx.x + static_cast<int64_t>(j) * gridDim.x < tiles) issue(blockIdx.x + j * gridDim.x, j);
    }
    __syncthreads();

    int it = 0;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
        const uint32_t xs = xs0 + buf * kDtXBytes;
        const int64_t rt = tile / col_tiles;
        const int64_t ct = tile - rt * col_tiles;
        int g;
        const int64_t r0 = src_row(rt, g);        // first source row
        const int64_t tk0 = rt * 128;             // first padded token (qT column)
        const int64_t c0 = ct * 128;
        const int64_t row_end = kGrouped ? static_cast<int64_t>(g_off[g + 1]) : p.rows;
        const int len = static_cast<int>(min(static_cast<int64_t>(128), row_end - r0));
        const int nch = static_cast<int>(min(static_cast<int64_t>(128), p.cols - c0));

        // thread 0 waits (bounded) for the block and for the previous store's
        // read of the code stage; the CTA follows its verdict, and the other
        // threads then pass the completed phase themselves (acquire)
        int landed = 1;
        if (t == 0) {
            bulk_wait_group_read<0>();
            landed = mbar_wait(&full[buf], ph, limit) ? 1 : 0;
        }
        landed = __syncthreads_and(landed);
        if (!landed) {
            if (t == 0) {
                atomicCAS(p.status, 0u, static_cast<unsigned int>(FP8BS_ERR_TIMEOUT));
                // the boxes in flight land before the CTA leaves
                const uint64_t drain = limit > kDtDrainNs ? limit : kDtDrainNs;
                for (int j = it; j < it + 2; ++j)
                    if (blockIdx.x + static_cast<int64_t>(j) * gridDim.x < tiles)
                        mbar_wait(&full[j & 1], static_cast<uint32_t>(j >> 1) & 1u, drain);
                bulk_wait_group_all();
            }
            return;
        }
        mbar_try_wait(&full[buf], ph);

        // ---- row pass: lane = (row, column half) ----
        {
            const int h = lane >> 4;
            const int r = warp * 16 + (lane & 15);
            const uint32_t sw = static_cast<uint32_t>(r & 7);
            const uint32_t rowp = xs + h * (kDtXBytes / 2) + r * 128;
            uint4 d[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) d[c] = ld_shared_v4(rowp + ((c ^ sw) << 4));
            uint32_t m = 0;
#pragma unroll
            for (int c = 0; c < 8; ++c) m = max(m, absmax_bits_8(d[c]));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
            const TileScale ts = tile_scale(__uint_as_float(m << 16), p.rule);
            const uint32_t outp = qs + r * 128;
            // grouped: a row of the next group is staged as zero codes
            const bool live = !kGrouped || r < len;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint2 a = quant8(d[2 * j], ts);
                uint2 b = quant8(d[2 * j + 1], ts);
                if (!live) a = b = make_uint2(0u, 0u);
                st_shared_v4(outp + (((4 * h + j) ^ sw) << 4), make_uint4(a.x, a.y, b.x, b.y));
            }
            if (h == 0) {
                row_scale[r] = ts.s;
                if (r < len) p.q_scales[ct * p.q_scale_ld + r0 + r] = ts.s;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // a whole block, or one whose rows run to the tensor's end (the store
        // stops there), leaves with one TMA store; a group's last block with
        // rows of later groups after it stores only its own rows
        const bool whole = !kGrouped || len == 128 || r0 + len >= p.rows;
        if (whole) {
            if (t == 0) {
                tma_store_2d(&map_q, qs, static_cast<int32_t>(c0), static_cast<int32_t>(r0));
                bulk_commit_group();
            }
        } else {
            for (int i = t; i < len * 8; i += kDtThreads) {
                const int rr = i >> 3, cc = i & 7;
                if (16 * cc < nch) {
                    const uint4 v = ld_shared_v4(qs + rr * 128 + ((cc ^ (rr & 7)) << 4));
                    *reinterpret_cast<uint4*>(p.q + (r0 + rr) * p.cols + c0 + 16 * cc) = v;
                }
            }
        }

        // ---- transposed pass, part 1: the values and the parts' column maxima ----
        uint32_t w[32];     // dual cast: BF16 pairs of channels (c, c + 1), tokens 32 part + k
        float nv[16][4];    // stash cast: -dec(q) s_row of channels c .. c + 3, tokens 16 part + k
        if constexpr (!kStash) {
            const int c = 2 * (t & 63);
            const int part = t >> 6;
            const uint32_t colp = xs + (c >> 6) * (kDtXBytes / 2) + ((c & 7) << 1);
            const uint32_t chunk = static_cast<uint32_t>((c & 63) >> 3);
            uint32_t mm = 0;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int r = part * 32 + k;
                w[k] = ld_shared_u32(colp + r * 128 + ((chunk ^ static_cast<uint32_t>(r & 7)) << 4));
                if (kGrouped && r >= len) w[k] = 0u;   // the next group's row
                mm = __vmaxu2(mm, w[k] & 0x7FFF7FFFu);
            }
            cpart[part][c] = __uint_as_float(mm << 16);
            cpart[part][c + 1] = __uint_as_float(mm & 0xFFFF0000u);
        } else {
            const int jq = t & 31;
            const int part = t >> 5;
            const int c = 4 * jq;
            const uint32_t colp = qs + ((jq & 3) << 2);
            const uint32_t chunk = static_cast<uint32_t>(jq >> 2);
            float cm[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int r = part * 16 + k;
                const uint32_t x = ld_shared_u32(colp + r * 128 + ((chunk ^ static_cast<uint32_t>(r & 7)) << 4));
                decode4_scaled(x, -row_scale[r], nv[k]);
#pragma unroll
                for (int e = 0; e < 4; ++e) cm[e] = fmaxf(cm[e], fabsf(nv[k][e]));
            }
            *reinterpret_cast<float4*>(&cpart[part][c]) = make_float4(cm[0], cm[1], cm[2], cm[3]);
        }
        __syncthreads();
        if (t < 128) {
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < (kStash ? 8 : 4); ++i) m = fmaxf(m, cpart[i][t]);
            const float s = scale_from_amax(m, p.rule);
            col_ts[t] = tile_scale_from_s(s);
            if (t < nch) p.scT[rt * p.cols + c0 + t] = s;
        }
        __syncthreads();
        // every read of this buffer is done: load the block after next into it
        if (t == 0 && tile + 2 * static_cast<int64_t>(gridDim.x) < tiles) {
            fence_proxy_async_smem();
            issue(tile + 2 * static_cast<int64_t>(gridDim.x), buf);
        }

        // exponent-byte atoms (power-of-two scales), as in requant_128x1_T_kernel
        if (t < 64 && (t < 32 ? p.q_atoms : p.qT_atoms) != nullptr) {
            const int l = t & 31;
            const bool rows_side = t < 32;
            uint32_t wv[4];
            bool bad = false;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = l + 32 * k;
                uint32_t E = 127u;
                if (rows_side ? i < len : i < nch) {
                    E = ue8m0_of(rows_side ? row_scale[i] : col_ts[i].s);
                    bad |= E == 255u;
                }
                wv[k] = E * 0x01010101u;
            }
            if (bad) atomicCAS(p.status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
            uint8_t* atom = rows_side ? p.q_atoms + (rt * (p.cols / 128) + ct) * 512
                                      : p.qT_atoms + (ct * (p.mpad / 128) + rt) * 512;
            *reinterpret_cast<uint4*>(atom + 16 * l) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }

        // ---- transposed pass, part 2: encode with the channel scales ----
        if constexpr (!kStash) {
            const int c = 2 * (t & 63);
            const int part = t >> 6;
            if (c < nch) {   // nch % 16 == 0: pairs are all-in or all-out
                const TileScale t0 = col_ts[c];
                const TileScale t1 = col_ts[c + 1];
                uint32_t o0[8], o1[8];
                if (t0.nr != 0.0f && t1.nr != 0.0f) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t* x = w + 4 * k;
                        const uint32_t a01 =
                            encode2_fast(make_float2(neg_bf16_lo(x[0]), neg_bf16_lo(x[1])), t0.s, t0.nr);
                        const uint32_t a23 =
                            encode2_fast(make_float2(neg_bf16_lo(x[2]), neg_bf16_lo(x[3])), t0.s, t0.nr);
                        const uint32_t b01 =
                            encode2_fast(make_float2(neg_bf16_hi(x[0]), neg_bf16_hi(x[1])), t1.s, t1.nr);
                        const uint32_t b23 =
                            encode2_fast(make_float2(neg_bf16_hi(x[2]), neg_bf16_hi(x[3])), t1.s, t1.nr);
                        o0[k] = __byte_perm(a01, a23, 0x5410);
                        o1[k] = __byte_perm(b01, b23, 0x5410);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t* x = w + 4 * k;
                        o0[k] = encode2_exact(bf16_lo(x[0]), bf16_lo(x[1]), t0.s) |
                                (encode2_exact(bf16_lo(x[2]), bf16_lo(x[3]), t0.s) << 16);
                        o1[k] = encode2_exact(bf16_hi(x[0]), bf16_hi(x[1]), t1.s) |
                                (encode2_exact(bf16_hi(x[2]), bf16_hi(x[3]), t1.s) << 16);
                    }
                }
                uint8_t* dst0 = p.qT + (c0 + c) * p.mpad + tk0 + part * 32;
                uint8_t* dst1 = dst0 + p.mpad;
                reinterpret_cast<uint4*>(dst0)[0] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
                reinterpret_cast<uint4*>(dst0)[1] = make_uint4(o0[4], o0[5], o0[6], o0[7]);
                reinterpret_cast<uint4*>(dst1)[0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                reinterpret_cast<uint4*>(dst1)[1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
            }
        } else {
            const int jq = t & 31;
            const int part = t >> 5;
            const int c = 4 * jq;
            if (c < nch) {
                TileScale ts[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) ts[e] = col_ts[c + e];
                uint32_t o[4][4];
                if (ts[0].nr != 0.0f && ts[1].nr != 0.0f && ts[2].nr != 0.0f && ts[3].nr != 0.0f) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            const uint32_t c01 = encode2_fast(make_float2(nv[4 * k][ch], nv[4 * k + 1][ch]),
                                                              ts[ch].s, ts[ch].nr);
                            const uint32_t c23 = encode2_fast(make_float2(nv[4 * k + 2][ch], nv[4 * k + 3][ch]),
                                                              ts[ch].s, ts[ch].nr);
                            o[ch][k] = __byte_perm(c01, c23, 0x5410);
                        }
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch)
                            o[ch][k] = encode2_exact(-nv[4 * k][ch], -nv[4 * k + 1][ch], ts[ch].s) |
                                       (encode2_exact(-nv[4 * k + 2][ch], -nv[4 * k + 3][ch], ts[ch].s) << 16);
                }
                uint8_t* dst = p.qT + (c0 + c) * p.mpad + tk0 + part * 16;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    *reinterpret_cast<uint4*>(dst + ch * p.mpad) = make_uint4(o[ch][0], o[ch][1], o[ch][2], o[ch][3]);
            }
        }
    }
    // the last code stage has been read, and every store has completed, before the CTA exits
    if (t == 0) bulk_wait_group_all();
}


// ---------------------------------------------------------------------------
// S2 with round-to-nearest codes on a TMA-fed persistent kernel: two CTAs of
// 256 threads per SM work through the 128x128 blocks of all batch entries.
// A block arrives by TMA (three-dimensional map [batch][rows][cols], so a
// block never reads rows of the next batch entry: they are out of bounds
// and arrive as zeros) into one of two buffers, so the next block loads
// while the current one is worked on. A lane holds one half (64 values) of
// one row; the block absmax is a warp reduction plus one value per warp in
// shared memory, and lane 0 of each warp turns it into the scale. The codes
// go through a swizzled stage and leave with one TMA store; the transposed
// copy is read back from the stage four channels x four tokens at a time,
// transposed in registers with byte permutes, and written as 16-token
// pieces of the qT rows. Same arithmetic as quant_128x128_kernel.
// ---------------------------------------------------------------------------
constexpr int kWtThreads = 256;
constexpr int kWtXBytes = 128 * 128 * 2;
constexpr int kWtQOff = 2 * kWtXBytes;
constexpr int kWtRedOff = kWtQOff + 128 * 128;
constexpr int kWtBarOff = kWtRedOff + 64;
constexpr int kWtSmemBytes = kWtBarOff + 16 + 1023;

// Rows of a 4 x 4 byte matrix held as four words (word i = row i, byte j =
// column j) -> its columns (word j = column j, byte i = row i).
__device__ __forceinline__ void transpose4x4_bytes(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                                   uint32_t (&o)[4])
{
    const uint32_t t0 = __byte_perm(w0, w1, 0x5140);   // w0.b0 w1.b0 w0.b1 w1.b1
    const uint32_t t1 = __byte_perm(w0, w1, 0x7362);   // w0.b2 w1.b2 w0.b3 w1.b3
    const uint32_t t2 = __byte_perm(w2, w3, 0x5140);
    const uint32_t t3 = __byte_perm(w2, w3, 0x7362);
    o[0] = __byte_perm(t0, t2, 0x5410);
    o[1] = __byte_perm(t0, t2, 0x7632);
    o[2] = __byte_perm(t1, t3, 0x5410);
    o[3] = __byte_perm(t1, t3, 0x7632);
}

__global__ void __launch_bounds__(kWtThreads, 2) wcast_tile_kernel(
    const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_q, int64_t rows,
    int64_t cols, uint8_t* __restrict__ qT, float* __restrict__ scales, const ScaleRule rule,
    uint8_t* __restrict__ atoms_wT, uint8_t* __restrict__ atoms_w, unsigned int* status, int64_t tiles,
    uint64_t limit)
{
    extern __shared__ uint8_t wt_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(wt_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t xs0 = smem_addr(smem);
    const uint32_t qs = xs0 + kWtQOff;
    uint32_t* red = reinterpret_cast<uint32_t*>(smem + kWtRedOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWtBarOff);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t nbr = (rows + 127) / 128, nbc = (cols + 127) / 128;
    const int64_t per_b = nbr * nbc;

    auto issue = [&](int64_t tile, int buf) {
        const int64_t b = tile / per_b;
        const int64_t rem = tile - b * per_b;
        const int64_t bi = rem / nbc, bj = rem - bi * nbc;
        uint8_t* dst = smem + buf * kWtXBytes;
        mbar_arrive_expect_tx(&full[buf], kWtXBytes);
        tma_load_3d(dst, &map_w, &full[buf], static_cast<int32_t>(bj * 128), static_cast<int32_t>(bi * 128),
                    static_cast<int32_t>(b));
        tma_load_3d(dst + kWtXBytes / 2, &map_w, &full[buf], static_cast<int32_t>(bj * 128 + 64),
                    static_cast<int32_t>(bi * 128), static_cast<int32_t>(b));
    };
    if (t == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbarrier_init();
        tma_prefetch_desc(&map_w);
        tma_prefetch_desc(&map_q);
        for (int j = 0; j < 2; ++j)
            if (blockIdx.x + static_cast<int64_t>(j) * gridDim.x < tiles) issue(blockIdx.x + j * gridDim.x, j);
    }
    __syncthreads();

    int it = 0;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
        const uint32_t xs = xs0 + buf * kWtXBytes;
        const int64_t b = tile / per_b;
        const int64_t rem = tile - b * per_b;
        const int64_t bi = rem / nbc, bj = rem - bi * nbc;
        const int64_t r0 = bi * 128, c0 = bj * 128;

        int landed = 1;
        if (t == 0) {
            bulk_wait_group_read<0>();   // the previous block's code stage has been read
            landed = mbar_wait(&full[buf], ph, limit) ? 1 : 0;
        }
        landed = __syncthreads_and(landed);
        if (!landed) {
            if (t == 0) {
                atomicCAS(status, 0u, static_cast<unsigned int>(FP8BS_ERR_TIMEOUT));
                const uint64_t drain = limit > kDtDrainNs ? limit : kDtDrainNs;
                for (int j = it; j < it + 2; ++j)
                    if (blockIdx.x + static_cast<int64_t>(j) * gridDim.x < tiles)
                        mbar_wait(&full[j & 1], static_cast<uint32_t>(j >> 1) & 1u, drain);
                bulk_wait_group_all();
            }
            return;
        }
        mbar_try_wait(&full[buf], ph);

        // ---- block absmax: lane = (row, column half) ----
        const int h = lane >> 4;
        const int r = warp * 16 + (lane & 15);
        const uint32_t sw = static_cast<uint32_t>(r & 7);
        const uint32_t rowp = xs + h * (kWtXBytes / 2) + r * 128;
        uint4 d[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) d[c] = ld_shared_v4(rowp + ((c ^ sw) << 4));
        uint32_t m = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) m = max(m, absmax_bits_8(d[c]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) red[warp] = m;
        __syncthreads();
        // every block is the same: lane 0 of each warp derives the scale,
        // which the warp then shares
        TileScale ts{0.0f, 0.0f};
        if (lane == 0) {
            uint32_t mb = 0;
#pragma unroll
            for (int i = 0; i < kWtThreads / 32; ++i) mb = max(mb, red[i]);
            ts = tile_scale(__uint_as_float(mb << 16), rule);
        }
        ts.s = __shfl_sync(0xFFFFFFFFu, ts.s, 0);
        ts.nr = __shfl_sync(0xFFFFFFFFu, ts.nr, 0);
        if (t == 0) scales[b * per_b + bi * nbc + bj] = ts.s;
        if (atoms_wT != nullptr && t < 64) {
            // the block's exponent byte fills one whole atom of each operand:
            // W^T (rows = the block's 128 columns, K-block bi) and W (rows =
            // its 128 rows, K-block bj); 16 bytes per thread
            const uint32_t E = ue8m0_of(ts.s);
            if (E == 255u && t == 0) atomicCAS(status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
            const uint32_t e4 = E * 0x01010101u;
            const int64_t bo = b * per_b * 512;
            uint8_t* atom = t < 32 ? atoms_wT + bo + (bj * nbr + bi) * 512 : atoms_w + bo + (bi * nbc + bj) * 512;
            *reinterpret_cast<uint4*>(atom + 16 * (t & 31)) = make_uint4(e4, e4, e4, e4);
        }
        const uint32_t outp = qs + r * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint2 a = quant8(d[2 * j], ts);
            const uint2 c = quant8(d[2 * j + 1], ts);
            st_shared_v4(outp + (((4 * h + j) ^ sw) << 4), make_uint4(a.x, a.y, c.x, c.y));
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (t == 0) {
            tma_store_3d(&map_q, qs, static_cast<int32_t>(c0), static_cast<int32_t>(r0), static_cast<int32_t>(b));
            bulk_commit_group();
            // every read of this buffer is done: load the block after next into it
            if (tile + 2 * static_cast<int64_t>(gridDim.x) < tiles) {
                fence_proxy_async_smem();
                issue(tile + 2 * static_cast<int64_t>(gridDim.x), buf);
            }
        }

        // ---- the transposed copy: channels 4 jq .. 4 jq + 3, tokens 16 part .. + 15 ----
        if (qT != nullptr) {
            const int jq = t & 31;
            const int part = t >> 5;
            const int64_t c = c0 + 4 * jq;
            const int64_t rr = r0 + part * 16;
            if (c < cols && rr < rows) {   // rows, cols % 16 == 0: quads and segments are all-in or all-out
                const uint32_t colp = qs + ((jq & 3) << 2);
                const uint32_t chunk = static_cast<uint32_t>(jq >> 2);
                uint32_t o[4][4];   // [channel][4-token group]
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int rl = part * 16 + 4 * k + e;
                        x[e] = ld_shared_u32(colp + rl * 128 + ((chunk ^ static_cast<uint32_t>(rl & 7)) << 4));
                    }
                    uint32_t y[4];
                    transpose4x4_bytes(x[0], x[1], x[2], x[3], y);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) o[ch][k] = y[ch];
                }
                uint8_t* dst = qT + b * rows * cols + c * rows + rr;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    *reinterpret_cast<uint4*>(dst + ch * rows) = make_uint4(o[ch][0], o[ch][1], o[ch][2], o[ch][3]);
            }
        }
    }
    if (t == 0) bulk_wait_group_all();
}

}  // namespace

cudaError_t launch_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t* q, float* scales, int64_t scale_ld, const ScaleRule& rule,
                               const SrParams* sr, int num_sms, cudaStream_t stream)
{
    if (rows == 0) return cudaSuccess;
    // One unit (32 rows x 128 columns) per warp: blocks run in as many waves
    // as the tensor needs, which balances better than a capped grid-stride
    // loop when the unit count is a few times the resident warp count.
    const int64_t units = ((cols + 127) / 128) * ((rows + 31) / 32);
    const int64_t warps_per_block = kQ1Threads / 32;
    int64_t blocks = (units + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)num_sms * 512;  // grid-stride only for very large tensors
    if (blocks > cap) blocks = cap;
    if (sr) {
        const SrKey key{sr->seed, sr->salt};
        quant_1x128_kernel<true><<<(unsigned)blocks, kQ1Threads, 0, stream>>>(x, rows, cols, ldx, q, scales,
                                                                             scale_ld, rule, key);
    } else {
        quant_1x128_kernel<false><<<(unsigned)blocks, kQ1Threads, 0, stream>>>(x, rows, cols, ldx, q, scales,
                                                                              scale_ld, rule, SrKey{0, 0});
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_1x128_stream(const CUtensorMap& map_x, const CUtensorMap& map_q, int64_t rows,
                                      int64_t cols, float* scales, int64_t scale_ld, const ScaleRule& rule,
                                      uint64_t limit, unsigned int* status, int num_sms, cudaStream_t stream)
{
    if (rows == 0) return cudaSuccess;
    constexpr int kSmem = kQ1sWarps * kQ1sWarpBytes + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory");
    // once per device: the shared-memory opt-in
    static std::atomic<uint64_t> ready{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(ready.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(quant_1x128_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        ready.fetch_or(bit, std::memory_order_release);
    }
    // as many SMs as the units can keep busy (one unit per warp at least):
    // a small tensor then finishes in about one unit's latency
    const int64_t units = ((cols + 127) / 128) * ((rows + 31) / 32);
    int64_t blocks = (units + kQ1sWarps - 1) / kQ1sWarps;
    if (blocks > num_sms) blocks = num_sms;
    quant_1x128_stream_kernel<<<static_cast<unsigned>(blocks), kQ1sWarps * 32, kSmem, stream>>>(
        map_x, map_q, rows, cols, scales, scale_ld, rule, limit, status);
    return cudaGetLastError();
}

cudaError_t launch_quant_128x128(const uint16_t* w, int64_t batch, int64_t rows, int64_t cols,
                                 int64_t ldw, uint8_t* q, uint8_t* qT, float* scales,
                                 const ScaleRule& rule, const SrParams* sr, cudaStream_t stream,
                                 uint8_t* atoms_wT, uint8_t* atoms_w, unsigned int* status)
{
    const int64_t blocks = batch * ((rows + 127) / 128) * ((cols + 127) / 128);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    if (sr) {
        const SrKey key{sr->seed, sr->salt};
        quant_128x128_kernel<true><<<(unsigned)blocks, kQ2Threads, 0, stream>>>(
            w, rows, cols, ldw, q, qT, scales, rule, key, atoms_wT, atoms_w, status);
    } else {
        quant_128x128_kernel<false><<<(unsigned)blocks, kQ2Threads, 0, stream>>>(
            w, rows, cols, ldw, q, qT, scales, rule, SrKey{0, 0}, atoms_wT, atoms_w, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_dual_tile(const CUtensorMap& map_x, const CUtensorMap& map_q, const RequantParams& p,
                             uint64_t limit, int num_sms, cudaStream_t stream)
{
    const int64_t col_tiles = (p.cols + 127) / 128;
    const int64_t tiles = (p.mpad / 128) * col_tiles;
    if (tiles == 0) return cudaSuccess;
    static_assert(2 * (kDtSmemBytes + 1024) <= 233472, "two CTAs per SM");
    // once per device: the shared-memory opt-in of both instances
    static std::atomic<uint64_t> ready{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(ready.load(std::memory_order_acquire) & bit)) {
        for (auto k : {dual_tile_kernel<false, false>, dual_tile_kernel<true, false>, dual_tile_kernel<false, true>,
                       dual_tile_kernel<true, true>}) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kDtSmemBytes);
            if (e != cudaSuccess) return e;
        }
        ready.fetch_or(bit, std::memory_order_release);
    }
    int64_t blocks = 2 * static_cast<int64_t>(num_sms);   // two resident CTAs per SM
    if (blocks > tiles) blocks = tiles;
    // groups (more than one, or device offsets): the grouped form
    const bool grouped = p.num_groups > 1 || p.off_dev != nullptr;
    auto kernel = p.stash ? (grouped ? dual_tile_kernel<true, true> : dual_tile_kernel<true, false>)
                          : (grouped ? dual_tile_kernel<false, true> : dual_tile_kernel<false, false>);
    kernel<<<static_cast<unsigned>(blocks), kDtThreads, kDtSmemBytes, stream>>>(map_x, map_q, p, col_tiles, tiles,
                                                                                limit);
    return cudaGetLastError();
}

cudaError_t launch_wcast_tile(const CUtensorMap& map_w, const CUtensorMap& map_q, int64_t batch, int64_t rows,
                              int64_t cols, uint8_t* qT, float* scales, const ScaleRule& rule, uint8_t* atoms_wT,
                              uint8_t* atoms_w, unsigned int* status, uint64_t limit, int num_sms,
                              cudaStream_t stream)
{
    const int64_t tiles = batch * ((rows + 127) / 128) * ((cols + 127) / 128);
    if (tiles == 0) return cudaSuccess;
    static_assert(2 * (kWtSmemBytes + 1024) <= 233472, "two CTAs per SM");
    static std::atomic<uint64_t> ready{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(ready.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(wcast_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWtSmemBytes);
        if (e != cudaSuccess) return e;
        ready.fetch_or(bit, std::memory_order_release);
    }
    int64_t blocks = 2 * static_cast<int64_t>(num_sms);
    if (blocks > tiles) blocks = tiles;
    wcast_tile_kernel<<<static_cast<unsigned>(blocks), kWtThreads, kWtSmemBytes, stream>>>(
        map_w, map_q, rows, cols, qT, scales, rule, atoms_wT, atoms_w, status, tiles, limit);
    return cudaGetLastError();
}

cudaError_t launch_requant_128x1_T(const RequantParams& p, cudaStream_t stream)
{
    const int64_t tiles = p.mpad / 128;
    if (tiles == 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)tiles, (unsigned)((p.cols + 127) / 128));
    if (grid.y > 65535) return cudaErrorInvalidValue;
    const bool dual = p.q != nullptr, stash = dual && p.stash;
    if (p.sr) {
        if (stash)
            requant_128x1_T_kernel<true, true, true><<<grid, kQ3Threads, 0, stream>>>(p);
        else if (dual)
            requant_128x1_T_kernel<true, false, true><<<grid, kQ3Threads, 0, stream>>>(p);
        else
            requant_128x1_T_kernel<false, false, true><<<grid, kQ3Threads, 0, stream>>>(p);
    } else {
        if (stash)
            requant_128x1_T_kernel<true, true, false><<<grid, kQ3Threads, 0, stream>>>(p);
        else if (dual)
            requant_128x1_T_kernel<true, false, false><<<grid, kQ3Threads, 0, stream>>>(p);
        else
            requant_128x1_T_kernel<false, false, false><<<grid, kQ3Threads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace fp8bs
