// quant.cu -- dynamic absmax quantizers to E4M3 with fp32 scales.
//
// The tile recipe: amax = max |v| over the tile, s = amax / 448 (IEEE fp32
// division; 1 for an all-zero tile), q = E4M3 round-to-nearest-even,
// saturating, of the fp32 quotient v / s. Source: "FP8 动态量化里的 partial sum
// 漂移", section 3, row (a) (per-tile dynamic scales from the absmax, N_c = 128);
// tile shapes from "scratch: the backward pass, unrolled", "What is asserted,
// and from where" (1x128 activations and gradients, 128x128 weights, 128x1
// re-tiling for Wgrad). E4M3 -0 (0x80) is kept apart from +0 (prime-rl PR
// #4073, conventions table, row "Negative zero"): the sign bit of every code
// is the sign of its input.
//
// All three kernels are HBM streams: 16-byte vector loads, warp-shuffle
// absmax reductions, coalesced payload and scale stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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

__device__ __forceinline__ float scale_from_amax(float amax)
{
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Sign bits of the four bf16 values held in (w0, w1), moved to bit 7 of the
// corresponding code bytes.
__device__ __forceinline__ uint32_t sign_bits_4(uint32_t w0, uint32_t w1)
{
    return ((w0 >> 8) & 0x80u) | ((w0 >> 16) & 0x8000u) | ((w1 << 8) & 0x800000u) |
           (w1 & 0x80000000u);
}

// Four bf16 values (two words) divided by s and encoded, low element first.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float s)
{
    uint32_t c01 = cvt_e4m3x2(__fdiv_rn(bf16_lo(w0), s), __fdiv_rn(bf16_hi(w0), s));
    uint32_t c23 = cvt_e4m3x2(__fdiv_rn(bf16_lo(w1), s), __fdiv_rn(bf16_hi(w1), s));
    return (c01 | (c23 << 16)) | sign_bits_4(w0, w1);
}

// ---------------------------------------------------------------------------
// S1: 1x128 tiles. One warp handles 32 rows x one 128-column tile: each
// half-warp reads one row's 256 bytes per load (16 lanes x 16 bytes), so a
// warp covers two rows per instruction and 32 rows in 16 loads, all issued
// before any arithmetic. Lane l ends up holding the scale of row l, so the
// warp stores its 32 scales as one 128-byte segment.
// ---------------------------------------------------------------------------
constexpr int kQ1Threads = 256;

__global__ void __launch_bounds__(kQ1Threads) quant_1x128_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
    uint8_t* __restrict__ q, float* __restrict__ scales, int64_t scale_ld)
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

        float my_scale = 1.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint32_t m = absmax_bits_8(d[i]);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            const float s = scale_from_amax(__uint_as_float(m << 16));
            // row 2i + h's scale goes to lane 2i + h
            const float t = __shfl_sync(0xFFFFFFFFu, s, (lane & 1) * 16);
            if (i == (lane >> 1)) my_scale = t;

            const int64_t r = row0 + 2 * i + half;
            if (col_ok && r < rows) {
                uint2 out;
                out.x = quant4(d[i].x, d[i].y, s);
                out.y = quant4(d[i].z, d[i].w, s);
                *reinterpret_cast<uint2*>(q + r * cols + col) = out;
            }
        }
        const int64_t r = row0 + lane;
        if (r < rows) scales[tc * scale_ld + r] = my_scale;
    }
}

// ---------------------------------------------------------------------------
// S2: 128x128 blocks. One CTA of 256 threads per block: thread t reads the
// 8-column chunk t % 16 of rows t / 16 + 16 i (i < 8), so each row's 256
// bytes come from 16 consecutive threads. Block absmax via warp shuffles and
// shared memory. The optional transposed payload goes through a padded
// shared-memory tile and leaves as 16-byte row segments of qT.
// ---------------------------------------------------------------------------
constexpr int kQ2Threads = 256;
constexpr int kQ2Pitch = 132;  // bytes per row of the staging tile (bank-conflict padding)

__global__ void __launch_bounds__(kQ2Threads) quant_128x128_kernel(
    const uint16_t* __restrict__ w, int64_t rows, int64_t cols, int64_t ldw,
    uint8_t* __restrict__ q, uint8_t* __restrict__ qT, float* __restrict__ scales)
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
    const float s = scale_from_amax(__uint_as_float(m << 16));
    if (threadIdx.x == 0) scales[b * nbr * nbc + bi * nbc + bj] = s;

    uint8_t* qb = q + b * rows * cols;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rl = rgrp + 16 * i;
        const int64_t r = r0 + rl;
        uint2 out;
        out.x = quant4(d[i].x, d[i].y, s);
        out.y = quant4(d[i].z, d[i].w, s);
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

__device__ __forceinline__ int find_group(const int32_t* tile_start, int ng, int tile)
{
    int lo = 0, hi = ng - 1;  // last g with tile_start[g] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kQ3Threads) requant_128x1_T_kernel(const __grid_constant__ RequantParams p)
{
    // staging: BF16 source 128 x 128 x 2 bytes, or E4M3 128 x 128 bytes + row scales
    __shared__ __align__(16) uint8_t stage[128 * 128 * 2];
    __shared__ float row_scale[128];
    __shared__ float col_part[16][128];
    __shared__ float col_scale[128];

    const int tile = blockIdx.x;                 // padded token tile
    const int64_t c0 = (int64_t)blockIdx.y * 128;
    const int g = find_group(p.tile_start, p.num_groups, tile);
    const int64_t r0 = (int64_t)p.off[g] + (int64_t)(tile - p.tile_start[g]) * 128;
    const int len = (int)min((int64_t)128, (int64_t)p.off[g + 1] - r0);
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
            *reinterpret_cast<uint4*>(stage + (rl * 128 + chunk * 8) * 2) = d[i];
        }
        uint32_t mw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mw[0] = __vmaxu2(mw[0], d[i].x & 0x7FFF7FFFu);
            mw[1] = __vmaxu2(mw[1], d[i].y & 0x7FFF7FFFu);
            mw[2] = __vmaxu2(mw[2], d[i].z & 0x7FFF7FFFu);
            mw[3] = __vmaxu2(mw[3], d[i].w & 0x7FFF7FFFu);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            col_part[rg][chunk * 8 + 2 * k] = __uint_as_float(mw[k] << 16);
            col_part[rg][chunk * 8 + 2 * k + 1] = __uint_as_float(mw[k] & 0xFFFF0000u);
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
        const float s = scale_from_amax(m);
        col_scale[threadIdx.x] = s;
        if (threadIdx.x < nch) p.scT[(int64_t)tile * p.cols + c0 + threadIdx.x] = s;
    }
    __syncthreads();

    // unit = (channel j, 32-token part): 512 units, two per thread
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int unit = threadIdx.x + u * kQ3Threads;
        const int j = unit & 127;
        const int part = unit >> 7;  // 0..3
        if (j >= nch) continue;
        const float s = col_scale[j];
        uint32_t outw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int rl = part * 32 + 4 * k + e;
                if (p.mode == FP8BS_SRC_BF16) {
                    const uint16_t h = *reinterpret_cast<const uint16_t*>(stage + (rl * 128 + j) * 2);
                    v[e] = __uint_as_float(static_cast<uint32_t>(h) << 16);
                } else {
                    const uint8_t c = stage[rl * 128 + j];
                    const float2 dv = e4m3x2_to_f32(static_cast<uint16_t>(c));
                    v[e] = __fmul_rn(dv.x, row_scale[rl]);
                }
            }
            uint32_t w = cvt_e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s)) |
                         (cvt_e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s)) << 16);
            w |= ((__float_as_uint(v[0]) >> 24) & 0x80u) | ((__float_as_uint(v[1]) >> 16) & 0x8000u) |
                 ((__float_as_uint(v[2]) >> 8) & 0x800000u) | (__float_as_uint(v[3]) & 0x80000000u);
            // tokens past the group's end are padding: 0x00
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (part * 32 + 4 * k + e >= len) w &= ~(0xFFu << (8 * e));
            outw[k] = w;
        }
        uint8_t* dst = p.qT + (c0 + j) * p.mpad + (int64_t)tile * 128 + part * 32;
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
    }
}

}  // namespace

cudaError_t launch_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t* q, float* scales, int64_t scale_ld, int num_sms,
                               cudaStream_t stream)
{
    if (rows == 0) return cudaSuccess;
    const int64_t units = ((cols + 127) / 128) * ((rows + 31) / 32);
    const int64_t warps_per_block = kQ1Threads / 32;
    int64_t blocks = (units + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)num_sms * 4;  // grid-stride beyond a few resident waves
    if (blocks > cap) blocks = cap;
    quant_1x128_kernel<<<(unsigned)blocks, kQ1Threads, 0, stream>>>(x, rows, cols, ldx, q, scales,
                                                                   scale_ld);
    return cudaGetLastError();
}

cudaError_t launch_quant_128x128(const uint16_t* w, int64_t batch, int64_t rows, int64_t cols,
                                 int64_t ldw, uint8_t* q, uint8_t* qT, float* scales,
                                 cudaStream_t stream)
{
    const int64_t blocks = batch * ((rows + 127) / 128) * ((cols + 127) / 128);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    quant_128x128_kernel<<<(unsigned)blocks, kQ2Threads, 0, stream>>>(w, rows, cols, ldw, q, qT,
                                                                     scales);
    return cudaGetLastError();
}

cudaError_t launch_requant_128x1_T(const RequantParams& p, cudaStream_t stream)
{
    const int64_t tiles = p.mpad / 128;
    if (tiles == 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)tiles, (unsigned)((p.cols + 127) / 128));
    if (grid.y > 65535) return cudaErrorInvalidValue;
    requant_128x1_T_kernel<<<grid, kQ3Threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fp8bs
