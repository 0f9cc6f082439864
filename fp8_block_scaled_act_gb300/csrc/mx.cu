// mx.cu -- MXFP8: 1x32 blocks with power-of-two exponent scales,
// and a GEMM whose block scaling runs in the tensor core.
//
// Format (OCP Microscaling Formats (MX) v1.0): 32 consecutive elements along
// K share one 8-bit exponent scale X = 2^(E - 127); elements are E4M3. The
// scale is the smallest power of two >= fp32(amax / 448) (X = 1 for an
// all-zero block), so no element saturates; q = E4M3_RN(v / X), an exact
// division. This is the B300 practice the TransformerEngine pages benchmark
// (PR #3573, "Changes" and "Performance": MXFP8 operands for dgrad) next to
// the software-promoted recipe of the rest of this library.
//
// Scale layout ("scale atoms", the layout tcgen05.cp.32x128b.warpx4 takes):
// for a matrix of R rows (padded to a multiple of 128) and K columns, atom
// (r / 128, k / 128) is 512 contiguous bytes; inside it the scale of row
// m = r % 128 = m0 + 32 m1 (m0 < 32) and 32-block j = (k / 32) % 4 sits at
// byte 16 m0 + 4 m1 + j. Atoms are ordered [R/128][K/128].
//
// GEMM: out[i, j] = sum_k A[i, k] B[j, k] with both operands blocked along
// K (A = activations [M x K], B = the other operand [N x K]), fp32
// accumulation in tensor memory over the whole K, BF16 or FP32 output. One CTA per SM,
// 128 x 256 tiles, a 4-stage TMA ring of (A, B, A scales, B scales); per
// 128-K stage one thread of warp 2 copies the scales into tensor memory
// (tcgen05.cp.32x128b.warpx4) and commits to a barrier, and the MMA thread
// (warp 1), which waits for that barrier, issues four
// tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each, the scale byte of
// each 32-block selected through the instruction descriptor). With the
// copies on the MMA thread the loop ran ~12% slower: its issue work per
// K-block is on the critical path. The epilogue
// runs once per tile: it reads the accumulator into registers, hands tensor
// memory back to the MMA issuer, and stores the tile as boxes of 32 rows x
// 64 bytes through a per-warp stage with TMA stores (plain stores for the
// rows of a ragged last row tile). The same kernel runs the 1x128 / 128x128
// recipe's GEMMs when their scales are powers of two (fp8_pack_ue8m0 below
// writes those scales into the atom layout).
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

// ---------------------------------------------------------------------------
// Quantizer: 16 threads per (row, 128-column group); a thread holds 8
// consecutive columns, so a 32-block is 4 adjacent lanes.
// ---------------------------------------------------------------------------
constexpr int kMxQThreads = 256;

__device__ __forceinline__ uint32_t mx_pow2_at_least(float s)
{
    // bits of the smallest power of two >= s > 0
    const uint32_t b = __float_as_uint(s);
    if ((b & 0x007FFFFFu) == 0u) return b;
    if ((b >> 23) != 0u) return (b & 0x7F800000u) + 0x00800000u;
    return 1u << (32 - __clz(b - 1u));
}

// Exponent byte E of a block with absmax `amax` (X = 2^(E - 127)).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax)
{
    if (amax == 0.0f) return 127u;
    const uint32_t b = mx_pow2_at_least(__fdiv_rn(amax, 448.0f));
    int e;
    if ((b >> 23) != 0u)
        e = static_cast<int>(b >> 23) - 127;
    else
        e = -118 - __clz(b);              // subnormal power of two 2^(31 - clz - 149)
    int E = e + 127;
    E = E < 0 ? 0 : (E > 254 ? 254 : E);
    return static_cast<uint32_t>(E);
}

__global__ void __launch_bounds__(kMxQThreads) mx_quant_1x32_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t rows_pad, int64_t cols, uint8_t* __restrict__ q,
    uint8_t* __restrict__ atoms)
{
    const int64_t groups = cols / 128;
    const int64_t units = rows_pad * groups;
    const int t = threadIdx.x & 15;
    int64_t unit = (static_cast<int64_t>(blockIdx.x) * kMxQThreads + threadIdx.x) >> 4;
    const int64_t stride = (static_cast<int64_t>(gridDim.x) * kMxQThreads) >> 4;
    for (; unit < units; unit += stride) {
        const int64_t r = unit / groups;
        const int64_t g = unit - r * groups;
        const int64_t c = g * 128 + t * 8;
        uint4 d = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) d = __ldcs(reinterpret_cast<const uint4*>(x + r * cols + c));
        uint32_t m = __vmaxu2(__vmaxu2(d.x & 0x7FFF7FFFu, d.y & 0x7FFF7FFFu),
                              __vmaxu2(d.z & 0x7FFF7FFFu, d.w & 0x7FFF7FFFu));
        m = max(m & 0xFFFFu, m >> 16);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        const uint32_t E = mx_scale_byte(__uint_as_float(m << 16));
        // 1 / X = 2^(127 - E): exact, and v * (1 / X) is the exact quotient v / X
        // (or its correctly rounded value when it falls below the normal range)
        const float inv = E >= 1u && E <= 253u ? __uint_as_float((254u - E) << 23) : 0.0f;
        const float X = __uint_as_float(E >= 1u ? (E << 23) : 0x00400000u);   // 2^(E - 127)
        uint2 o;
        const uint32_t wd[4] = {d.x, d.y, d.z, d.w};
        uint32_t code[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(wd[k] << 16), hi = __uint_as_float(wd[k] & 0xFFFF0000u);
            const float qlo = inv != 0.0f ? __fmul_rn(lo, inv) : __fdiv_rn(lo, X);
            const float qhi = inv != 0.0f ? __fmul_rn(hi, inv) : __fdiv_rn(hi, X);
            code[k] = cvt_e4m3x2(qlo, qhi);
        }
        o.x = code[0] | (code[1] << 16);
        o.y = code[2] | (code[3] << 16);
        if (r < rows) *reinterpret_cast<uint2*>(q + r * cols + c) = o;
        // the four exponent bytes of this (row, 128-column group) are contiguous in the atom
        const uint32_t e0 = __shfl_sync(0xFFFFFFFFu, E, (threadIdx.x & 16) | 0);
        const uint32_t e1 = __shfl_sync(0xFFFFFFFFu, E, (threadIdx.x & 16) | 4);
        const uint32_t e2 = __shfl_sync(0xFFFFFFFFu, E, (threadIdx.x & 16) | 8);
        const uint32_t e3 = __shfl_sync(0xFFFFFFFFu, E, (threadIdx.x & 16) | 12);
        if (t == 0) {
            const int64_t mrow = r & 127;
            uint8_t* atom = atoms + ((r >> 7) * groups + g) * 512;
            *reinterpret_cast<uint32_t*>(atom + 16 * (mrow & 31) + 4 * (mrow >> 5)) =
                e0 | (e1 << 8) | (e2 << 16) | (e3 << 24);
        }
    }
}

// ---------------------------------------------------------------------------
// Transposed quantizer: the 1x32 cast of x^T, i.e. 32-token blocks along the
// rows of qT [cols x rows_pad]. One CTA per (128-token tile, 128-channel
// block): the BF16 block is staged in shared memory (coalesced along
// channels), then each thread casts two (channel, 32-token block) units read
// down the staged columns, and the CTA's 512 exponent bytes (exactly one
// scale atom of qT) leave as one contiguous 512-byte write.
// ---------------------------------------------------------------------------
constexpr int kMxTThreads = 256;

__global__ void __launch_bounds__(kMxTThreads) mx_quant_1x32_T_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t rows_pad, uint8_t* __restrict__ qT,
    uint8_t* __restrict__ atoms)
{
    __shared__ __align__(16) uint16_t stage[128][128];
    __shared__ __align__(16) uint8_t sf[512];
    const int tile = blockIdx.x;                       // 128-token tile
    const int cb = blockIdx.y;                         // 128-channel block
    const int64_t r0 = static_cast<int64_t>(tile) * 128;
    const int64_t c0 = static_cast<int64_t>(cb) * 128;
    {
        const int chunk = threadIdx.x & 15, rg = threadIdx.x >> 4;
        const int64_t c = c0 + chunk * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rl = rg * 8 + i;
            const int64_t r = r0 + rl;
            uint4 d = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows && c < cols) d = __ldcs(reinterpret_cast<const uint4*>(x + r * cols + c));
            *reinterpret_cast<uint4*>(&stage[rl][chunk * 8]) = d;
        }
    }
    __syncthreads();
    const int ch = threadIdx.x & 127;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int j = 2 * (threadIdx.x >> 7) + u;     // 32-token block of the tile
        uint32_t v[32];
        uint32_t m = 0u;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            v[k] = stage[32 * j + k][ch];
            m = max(m, v[k] & 0x7FFFu);
        }
        const uint32_t E = mx_scale_byte(__uint_as_float(m << 16));
        const float inv = E >= 1u && E <= 253u ? __uint_as_float((254u - E) << 23) : 0.0f;
        const float X = __uint_as_float(E >= 1u ? (E << 23) : 0x00400000u);   // 2^(E - 127)
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float val = __uint_as_float(v[4 * k + e] << 16);
                f[e] = inv != 0.0f ? __fmul_rn(val, inv) : __fdiv_rn(val, X);
            }
            w[k] = cvt_e4m3x2(f[0], f[1]) | (cvt_e4m3x2(f[2], f[3]) << 16);
        }
        if (c0 + ch < cols) {
            uint4* dst = reinterpret_cast<uint4*>(qT + (c0 + ch) * rows_pad + r0 + 32 * j);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        // row ch of the atom, 32-block j: byte 16 (ch % 32) + 4 (ch / 32) + j
        sf[16 * (ch & 31) + 4 * (ch >> 5) + j] = static_cast<uint8_t>(E);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        uint8_t* atom = atoms + (static_cast<int64_t>(cb) * (rows_pad / 128) + tile) * 512;
        reinterpret_cast<uint4*>(atom)[threadIdx.x] = reinterpret_cast<const uint4*>(sf)[threadIdx.x];
    }
}

// ---------------------------------------------------------------------------
// GEMM
// ---------------------------------------------------------------------------
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK;              // 16 KB
constexpr int kBBytes = kBN * kBK;              // 32 KB
constexpr int kSfaBytes = 512;                  // one atom: 128 rows x 4 blocks
constexpr int kSfbBytes = 1024;                 // two atoms: 256 rows
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 4;
constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kProducerRegs = 40;
constexpr uint32_t kEpilogueRegs = 232;
static_assert(128 * kProducerRegs + 256 * kEpilogueRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;                  // accumulator 256 + scale slots
constexpr int kSfCol0 = kBN;                    // first scale column
constexpr int kSfColsPerStage = 12;             // 4 (A) + 8 (B)
constexpr uint64_t kDrainLimitNs = 1000000000ull;
constexpr int kCtlBytes = 2048;
// Output stage: per epilogue warp one box of 32 rows x 64 bytes (32 BF16 or
// 16 FP32 columns) in the 64-byte swizzle: 16-byte chunk c of row r at slot
// c ^ ((r / 2) % 4), conflict-free for 32 lanes writing one row each.
constexpr int kOutBoxBytes = 32 * 32 * 2;
constexpr int kOutStageBytes = kEpiWarps * kOutBoxBytes;
constexpr int kRingBytes = kStages * (kABytes + kBBytes + kSfaBytes + kSfbBytes);
static_assert(kRingBytes % 512 == 0, "the output stage needs 512-byte alignment");
constexpr int kSmemBytes = kRingBytes + kOutStageBytes + kCtlBytes + 1024;

struct MxCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t sfull[kStages];   // the stage's scales are in tensor memory
    uint64_t sf_done;
    uint64_t tfull;
    uint64_t tempty;
    uint64_t mma_done;
    uint32_t tmem_base;
    volatile int abort;
    // groups: row groups, the first M-tile of each group (exclusive scan of
    // their 128-row tiles); token groups, the first padded K-block of each
    int32_t tstart[kMaxGroups + 1];
    int32_t total_tiles;
};

struct MxParams {
    const uint8_t* sfa;   // A scale atoms (see MxGroups for the grouped layouts)
    const uint8_t* sfb;   // B scale atoms
    int m_tiles, n_tiles, kblocks;
    int M, N;
    uint16_t* out;        // BF16 [M x N], or
    float* out_f32;       // FP32 [M x N] (when not null)
    int tma_store;        // whole 32-row boxes leave through the output map
    uint64_t wait_limit_ns;
    unsigned int* status;
    MxGroups grp;
};

// Where the tile's operands, scales and output rows are (all roles decode
// the same tiles in the same order).
struct MxTile {
    int a_row, k0, b_row, nkb;     // TMA coordinates of A / B row 0 and K-block 0; K-blocks
                                   // (MN-major B: b_row = the group's first K row, col0 its column)
    int64_t sfa, sfb0, sfb1;       // byte offsets of K-block 0's atoms (then + 512 per K-block)
    int out_row0, row_end;         // output-map row of the tile's row 0; rows from row_end on are not stored
    int col0;                      // first output column
};

__device__ __forceinline__ int mx_group_off(const MxGroups& gp, int g)
{
    return gp.off_dev ? __ldg(gp.off_dev + g) : gp.off[g];
}

// Builds the group table (all threads take part; ends with a CTA barrier).
// Invalid offsets (off[0] != 0, a decrease, a total other than rows, more
// padded K-blocks than the operands hold) leave no tiles and record
// FP8BS_ERR_DEVICE.
__device__ void mx_build_tab(const MxParams& p, MxCtl* ctl)
{
    const MxGroups& gp = p.grp;
    if (gp.layout == kMxDense) {
        if (threadIdx.x == 0) ctl->total_tiles = p.m_tiles * p.n_tiles;
        __syncthreads();
        return;
    }
    const int G = gp.num_groups;
    int bad = 0;
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const int n = mx_group_off(gp, g + 1) - mx_group_off(gp, g);
        if (n < 0) bad = 1;
        ctl->tstart[g] = n < 0 ? 0 : (n + 127) / 128;
    }
    if (threadIdx.x == 0 && (mx_group_off(gp, 0) != 0 || mx_group_off(gp, G) != gp.rows_total)) bad = 1;
    bad = __syncthreads_or(bad);
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (G + 31) / 32;
        const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
        int sum = 0;
        for (int g = g0; g < g1; ++g) sum += ctl->tstart[g];
        int inc = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if (lane >= d) inc += v;
        }
        int run = inc - sum;
        for (int g = g0; g < g1; ++g) {
            const int c = ctl->tstart[g];
            ctl->tstart[g] = run;
            run += c;
        }
        if (lane == 31) {
            ctl->tstart[G] = inc;
            const bool over = gp.layout == kMxTokenGroups && inc > gp.kb_cap;
            const int total = gp.layout == kMxRowGroups ? inc * p.n_tiles : G * (gp.out_rows / kBM) * p.n_tiles;
            ctl->total_tiles = (bad || over) ? 0 : total;
            if ((bad || over) && blockIdx.x == 0) atomicCAS(p.status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
        }
    }
    __syncthreads();
}

template <bool kBMn>
__device__ __forceinline__ MxTile mx_tile(const MxParams& p, const MxCtl* ctl, int t)
{
    const MxGroups& gp = p.grp;
    MxTile d;
    if (gp.layout == kMxDense) {
        const int mt = t / p.n_tiles, nt = t - mt * p.n_tiles;
        d.a_row = mt * kBM;
        d.k0 = 0;
        d.b_row = kBMn ? 0 : nt * kBN;
        d.nkb = p.kblocks;
        d.sfa = static_cast<int64_t>(mt) * gp.kb_atoms_a * 512;
        d.sfb0 = static_cast<int64_t>(2 * nt) * gp.kb_atoms_b * 512;
        d.sfb1 = d.sfb0 + static_cast<int64_t>(gp.kb_atoms_b) * 512;
        d.out_row0 = d.a_row;
        d.row_end = p.M;
        d.col0 = nt * kBN;
    } else if (gp.layout == kMxRowGroups) {
        const int lt = t / p.n_tiles, nt = t - lt * p.n_tiles;   // lt: M-tile over all groups
        int lo = 0, hi = gp.num_groups - 1;                       // last g with tstart[g] <= lt
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ctl->tstart[mid] <= lt) lo = mid; else hi = mid - 1;
        }
        const int g = lo, mt = lt - ctl->tstart[g];
        const int o0 = mx_group_off(gp, g);
        d.a_row = o0 + mt * kBM;
        d.k0 = 0;
        d.b_row = kBMn ? g * p.kblocks * kBK : g * gp.b_group_rows + nt * kBN;
        d.nkb = p.kblocks;
        d.sfa = static_cast<int64_t>(lt) * gp.kb_atoms_a * 512;
        d.sfb0 = (static_cast<int64_t>(g) * (gp.b_group_rows / 128) + 2 * nt) * gp.kb_atoms_b * 512;
        d.sfb1 = d.sfb0 + static_cast<int64_t>(gp.kb_atoms_b) * 512;
        d.out_row0 = d.a_row;
        d.row_end = mx_group_off(gp, g + 1);
        d.col0 = nt * kBN;
    } else {
        const int per = (gp.out_rows / kBM) * p.n_tiles;
        const int g = t / per, local = t - g * per;
        const int mt = local / p.n_tiles, nt = local - mt * p.n_tiles;
        const int kb0 = ctl->tstart[g];
        d.a_row = mt * kBM;
        d.k0 = kb0 * kBK;
        d.b_row = nt * kBN;
        d.nkb = ctl->tstart[g + 1] - kb0;
        d.sfa = (static_cast<int64_t>(mt) * gp.kb_atoms_a + kb0) * 512;
        d.sfb0 = (static_cast<int64_t>(2 * nt) * gp.kb_atoms_b + kb0) * 512;
        d.sfb1 = d.sfb0 + static_cast<int64_t>(gp.kb_atoms_b) * 512;
        d.out_row0 = g * gp.out_rows + mt * kBM;
        d.row_end = (g + 1) * gp.out_rows;
        d.col0 = nt * kBN;
    }
    return d;
}

// Shared-memory descriptor of a scale atom (32 rows of 16 bytes, no swizzle;
// 8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t sdesc_atom(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (one core matrix wide)
    d |= static_cast<uint64_t>(128u >> 4) << 32;          // stride byte offset: 8 rows x 16 bytes
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
    return d;                                             // swizzle: none
}

__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with E4M3 A and B (K-major),
// UE8M0 scales, shape M x N (x 32); sf_id selects the scale byte of the
// 32-block inside each 32-bit tensor-memory cell.
__device__ __forceinline__ uint32_t idesc_mx(int M, int N, uint32_t sf_id)
{
    return (sf_id << 4)                                   // B scale byte
           | (0u << 7) | (0u << 10)                       // A, B: E4M3
           | (static_cast<uint32_t>(N >> 3) << 17)
           | (1u << 23)                                   // scale format: UE8M0
           | (static_cast<uint32_t>(M >> 4) << 24)
           | (sf_id << 29);                               // A scale byte
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void record_status(unsigned int* status, unsigned int code)
{
    atomicCAS(status, 0u, code);
}

// kF32: FP32 output (p.out_f32) instead of BF16 (p.out). kBMn: B's codes
// are [K x N] and reach the tensor core MN-major (p.grp.b_mn; BF16 only).
template <bool kF32, bool kBMn>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_out, const __grid_constant__ MxParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + kStages * kABytes;
    uint8_t* sSfa = sB + kStages * kBBytes;
    uint8_t* sSfb = sSfa + kStages * kSfaBytes;
    uint8_t* sOut = smem + kRingBytes;
    MxCtl* ctl = reinterpret_cast<MxCtl*>(sOut + kOutStageBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int s = 0; s < kStages; ++s) mbar_init(&ctl->sfull[s], 1);
        mbar_init(&ctl->sf_done, 1);
        mbar_init(&ctl->tfull, 1);
        mbar_init(&ctl->tempty, kEpiWarps);
        mbar_init(&ctl->mma_done, 1);
        ctl->abort = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        if (p.tma_store) tma_prefetch_desc(&map_out);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    tc_fence_after_sync();
    mx_build_tab(p, ctl);
    const int total = ctl->total_tiles;
    const uint32_t tmem_base = ctl->tmem_base;
    const uint64_t limit = p.wait_limit_ns;

    if (warp < kFirstEpiWarp) setmaxnreg_dec<kProducerRegs>();

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const MxTile d = mx_tile<kBMn>(p, ctl, t);
                for (int kb = 0; kb < d.nkb; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (ctl->abort || !mbar_wait(&ctl->empty[s], ph ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ctl->full[s], kABytes + kBBytes + kSfaBytes + kSfbBytes);
                    tma_load_2d(sA + s * kABytes, &map_a, &ctl->full[s], d.k0 + kb * kBK, d.a_row);
                    if constexpr (kBMn) {
                        // MN-major B: K rows x 128 columns per box, the
                        // tile's two column halves one box apart
                        const int yk = d.b_row + d.k0 + kb * kBK;
                        tma_load_2d(sB + s * kBBytes, &map_b, &ctl->full[s], d.col0, yk);
                        tma_load_2d(sB + s * kBBytes + kBBytes / 2, &map_b, &ctl->full[s], d.col0 + kBN / 2, yk);
                    } else {
                        tma_load_2d(sB + s * kBBytes, &map_b, &ctl->full[s], d.k0 + kb * kBK, d.b_row);
                    }
                    bulk_load(sSfa + s * kSfaBytes, p.sfa + d.sfa + static_cast<int64_t>(kb) * 512, kSfaBytes,
                              &ctl->full[s]);
                    bulk_load(sSfb + s * kSfbBytes, p.sfb + d.sfb0 + static_cast<int64_t>(kb) * 512, 512,
                              &ctl->full[s]);
                    bulk_load(sSfb + s * kSfbBytes + 512, p.sfb + d.sfb1 + static_cast<int64_t>(kb) * 512, 512,
                              &ctl->full[s]);
                }
            }
            if (!ok) {
                record_status(p.status, FP8BS_ERR_TIMEOUT);
                ctl->abort = 1;
            }
            const uint32_t first = it > kStages ? it - kStages : 0u;
            const uint64_t drain = limit > kDrainLimitNs ? limit : kDrainLimitNs;
            for (uint32_t j = first; j < it; ++j)
                mbar_wait(&ctl->full[j % kStages], (j / kStages) & 1u, drain);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0, tile_it = 0;
            bool ok = true;
            constexpr uint32_t b_major = kBMn ? kIdescBMajorMN : 0u;
            // start-address step of B per 32 K (16-byte units; see gemm.cu)
            constexpr uint64_t b_step = kBMn ? 4096u >> 4 : 32u >> 4;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tile_it) {
                // the accumulator is free once the epilogue has read the previous tile
                if (ctl->abort || !mbar_wait(&ctl->tempty, (tile_it & 1u) ^ 1u, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int nkb = mx_tile<kBMn>(p, ctl, t).nkb;   // a tile of an empty group issues no MMA
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (ctl->abort || !mbar_wait(&ctl->sfull[s], ph, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sf_a = tmem_base + kSfCol0 + s * kSfColsPerStage;
                    const uint32_t sf_b = sf_a + 4;
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(sA + s * kABytes));
                    const uint64_t bdesc = kBMn ? sdesc_mnmajor_sw128(smem_addr(sB + s * kBBytes), kBBytes / 2)
                                                : sdesc_kmajor_sw128(smem_addr(sB + s * kBBytes));
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        mma_mx(tmem_base, adesc + 2u * kk, bdesc + b_step * kk, idesc_mx(kBM, kBN, kk) | b_major,
                               sf_a, sf_b, (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&ctl->empty[s]);
                }
                if (!ok) break;
                mma_commit(&ctl->tfull);
            }
            if (!ok) {
                record_status(p.status, FP8BS_ERR_TIMEOUT);
                ctl->abort = 1;
            }
            mma_commit(&ctl->mma_done);
            const uint64_t drain = limit > kDrainLimitNs ? limit : kDrainLimitNs;
            mbar_wait(&ctl->mma_done, 0u, drain);
        }
    } else if (warp == 2) {
        // scale copier: the stage's scale atoms into tensor memory, then a
        // commit that the MMA issuer waits for
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int nkb = mx_tile<kBMn>(p, ctl, t).nkb;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (ctl->abort || !mbar_wait(&ctl->full[s], ph, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sf_a = tmem_base + kSfCol0 + s * kSfColsPerStage;
                    const uint32_t sf_b = sf_a + 4;
                    tmem_cp_32x128b_x4(sf_a, sdesc_atom(smem_addr(sSfa + s * kSfaBytes)));
                    tmem_cp_32x128b_x4(sf_b, sdesc_atom(smem_addr(sSfb + s * kSfbBytes)));
                    tmem_cp_32x128b_x4(sf_b + 4, sdesc_atom(smem_addr(sSfb + s * kSfbBytes + 512)));
                    mma_commit(&ctl->sfull[s]);
                }
            }
            if (!ok) {
                record_status(p.status, FP8BS_ERR_TIMEOUT);
                ctl->abort = 1;
            }
            // drain: every copy this thread issued has completed
            mma_commit(&ctl->sf_done);
            const uint64_t drain = limit > kDrainLimitNs ? limit : kDrainLimitNs;
            mbar_wait(&ctl->sf_done, 0u, drain);
        }
    } else if (warp >= kFirstEpiWarp) {
        setmaxnreg_inc<kEpilogueRegs>();
        const int ew = warp - kFirstEpiWarp;
        const int quarter = warp & 3;
        const int half = ew >> 2;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t tile_it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tile_it) {
            const MxTile d = mx_tile<kBMn>(p, ctl, t);
            if (ctl->abort || !mbar_wait(&ctl->tfull, tile_it & 1u, limit)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int row0 = d.out_row0 + quarter * 32;           // first output row of this warp
            const int row = row0 + lane;
            const int col0 = d.col0 + half * 128;
            if (d.nkb == 0) {
                // a tile of an empty group: no MMA wrote the accumulator; its
                // output is zero
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty);
                if (row < d.row_end) {
                    if constexpr (kF32) {
                        float4* y = reinterpret_cast<float4*>(p.out_f32 + static_cast<int64_t>(row) * p.N + col0);
#pragma unroll
                        for (int v = 0; v < 32; ++v) y[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else {
                        uint4* y = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row) * p.N + col0);
#pragma unroll
                        for (int v = 0; v < 16; ++v) y[v] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                continue;
            }
            uint32_t ra[32], rb[32];
            if constexpr (kF32) {
                // FP32 output: the whole 128-column row in registers, the
                // accumulator released, then (whole 32-row boxes) eight boxes
                // of 16 columns through the warp's stage with TMA stores, or
                // (a ragged last row tile) plain 16-byte stores
                uint32_t rc[32], rd[32];
                tmem_ld_x32(tmem_base + lane_addr + half * 128, ra);
                tmem_ld_x32(tmem_base + lane_addr + half * 128 + 32, rb);
                tmem_ld_x32(tmem_base + lane_addr + half * 128 + 64, rc);
                tmem_ld_x32(tmem_base + lane_addr + half * 128 + 96, rd);
                tmem_ld_wait(ra);
                tmem_regs_ready(rb);
                tmem_regs_ready(rc);
                tmem_regs_ready(rd);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty);
                if (p.tma_store && row0 + 32 <= d.row_end && col0 < p.N) {
                    const uint32_t box = smem_addr(sOut) + ew * kOutBoxBytes;
                    auto put = [&](const uint32_t (&r)[32], int b) {
                        if (lane == 0) bulk_wait_group_read<0>();    // the previous box has been read
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int v = 16 * (b & 1) + 4 * c;
                            st_shared_v4(box + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4),
                                         make_uint4(r[v], r[v + 1], r[v + 2], r[v + 3]));
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&map_out, box, col0 + 16 * b, row0);
                            bulk_commit_group();
                        }
                    };
                    put(ra, 0); put(ra, 1); put(rb, 2); put(rb, 3);
                    put(rc, 4); put(rc, 5); put(rd, 6); put(rd, 7);
                } else if (row < d.row_end && col0 < p.N) {
                    float4* y = reinterpret_cast<float4*>(p.out_f32 + static_cast<int64_t>(row) * p.N + col0);
                    auto put = [&](const uint32_t (&r)[32], int c) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            y[8 * c + v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                       __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                    };
                    put(ra, 0); put(rb, 1); put(rc, 2); put(rd, 3);
                }
                continue;
            }
            uint32_t pk[64];
            tmem_ld_x32(tmem_base + lane_addr + half * 128, ra);
            tmem_ld_x32(tmem_base + lane_addr + half * 128 + 32, rb);
            tmem_ld_wait(ra);
            tmem_ld_wait(rb);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                pk[i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
                pk[16 + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
            }
            tmem_ld_x32(tmem_base + lane_addr + half * 128 + 64, ra);
            tmem_ld_x32(tmem_base + lane_addr + half * 128 + 96, rb);
            tmem_ld_wait(ra);
            tmem_ld_wait(rb);
            // the accumulator is in registers: hand it back to the MMA issuer
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->tempty);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                pk[32 + i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
                pk[48 + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
            }
            if (p.tma_store && row0 + 32 <= d.row_end && col0 < p.N) {
                // four boxes of 32 columns through the warp's stage, each
                // leaving with one TMA store while the warp goes on
                const uint32_t box = smem_addr(sOut) + ew * kOutBoxBytes;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if (lane == 0) bulk_wait_group_read<0>();    // the previous box has been read
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_shared_v4(box + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4),
                                     make_uint4(pk[16 * b + 4 * c], pk[16 * b + 4 * c + 1], pk[16 * b + 4 * c + 2],
                                                pk[16 * b + 4 * c + 3]));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&map_out, box, col0 + 32 * b, row0);
                        bulk_commit_group();
                    }
                }
            } else if (row < d.row_end && col0 < p.N) {
                uint4* y = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row) * p.N + col0);
#pragma unroll
                for (int v = 0; v < 16; ++v) y[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
        }
        // the warp's TMA stores have completed before the CTA exits
        if (lane == 0) bulk_wait_group_all();
        if (!ok) {
            record_status(p.status, FP8BS_ERR_TIMEOUT);
            ctl->abort = 1;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Packing of power-of-two fp32 block scales into the scale-atom layout: the
// 128-element K-blocks of the 1x128 / 128x128 recipe become four 32-element
// blocks with the same exponent byte, so the MX GEMM applies them with the
// tensor core's block scaling. One thread per (operand row, K-block): the
// row's four bytes of that K-block are one 32-bit word of the atom.
// ---------------------------------------------------------------------------

namespace {

__global__ void __launch_bounds__(256) pack_ue8m0_kernel(const float* __restrict__ scales, int64_t rows,
                                                         int64_t rows_pad, int64_t kblocks, int row_block,
                                                         int64_t row_stride, int64_t kb_stride,
                                                         uint8_t* __restrict__ atoms, unsigned int* status)
{
    const int64_t n = rows_pad * kblocks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // i = (row tile, K-block, row within the tile): consecutive threads
        // fill consecutive rows of one atom
        const int64_t kb = (i >> 7) % kblocks;
        const int64_t r = ((i >> 7) / kblocks) * 128 + (i & 127);
        uint32_t E = 127u;   // padding rows: scale 1
        if (r < rows) {
            E = ue8m0_of(__ldg(scales + (r / row_block) * row_stride + kb * kb_stride));
            if (E == 255u) atomicCAS(status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
        }
        *reinterpret_cast<uint32_t*>(atoms + atom_offset(r, kb, kblocks)) = E * 0x01010101u;
    }
}

// Grouped rows (the A operand of a grouped MX Fprop / Dgrad): row l of
// group g (source row off[g] + l) goes to row l % 128 of the group's tile
// l / 128; tiles are numbered over the groups in order. One thread per
// (tile row, K-block); rows of a group's last tile past its end get 127.
__global__ void __launch_bounds__(256) pack_ue8m0_grouped_kernel(const float* __restrict__ scales, int64_t kblocks,
                                                                 int64_t kb_stride, PackGroups pg, int64_t tiles_cap,
                                                                 uint8_t* __restrict__ atoms, unsigned int* status)
{
    __shared__ int32_t off[kMaxGroups + 1];
    __shared__ int32_t tstart[kMaxGroups + 1];
    __shared__ int32_t wsum[8];
    const int G = pg.num_groups, t = threadIdx.x;
    for (int i = t; i <= G; i += blockDim.x) off[i] = pg.off_dev ? __ldg(pg.off_dev + i) : pg.off[i];
    __syncthreads();
    int bad = 0, cnt = 0;
    if (t < G) {
        const int n = off[t + 1] - off[t];
        if (n < 0) bad = 1;
        cnt = n < 0 ? 0 : (n + 127) / 128;
    }
    if (t == 0 && (off[0] != 0 || off[G] != pg.rows_total)) bad = 1;
    int inc = cnt;   // inclusive scan of the tile counts (one group per thread)
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if ((t & 31) >= d) inc += v;
    }
    if ((t & 31) == 31) wsum[t >> 5] = inc;
    __syncthreads();
    for (int w = 0; w < (t >> 5); ++w) inc += wsum[w];
    if (t < G) tstart[t] = inc - cnt;
    if (t == G - 1) tstart[G] = inc;
    bad = __syncthreads_or(bad);
    if (bad || tstart[G] > tiles_cap) {
        if (t == 0 && blockIdx.x == 0) atomicCAS(status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
        return;
    }
    const int64_t n = static_cast<int64_t>(tstart[G]) * 128 * kblocks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + t; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t kb = (i >> 7) % kblocks;
        const int lt = static_cast<int>((i >> 7) / kblocks);
        const int m = static_cast<int>(i & 127);
        int lo = 0, hi = G - 1;   // last g with tstart[g] <= lt
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tstart[mid] <= lt) lo = mid; else hi = mid - 1;
        }
        const int l = (lt - tstart[lo]) * 128 + m;
        uint32_t E = 127u;   // padding rows: scale 1
        if (l < off[lo + 1] - off[lo]) {
            E = ue8m0_of(__ldg(scales + static_cast<int64_t>(off[lo] + l) + kb * kb_stride));
            if (E == 255u) atomicCAS(status, 0u, static_cast<unsigned int>(FP8BS_ERR_DEVICE));
        }
        *reinterpret_cast<uint32_t*>(atoms + atom_offset(static_cast<int64_t>(lt) * 128 + m, kb, kblocks)) =
            E * 0x01010101u;
    }
}

}  // namespace

cudaError_t launch_pack_ue8m0_grouped(const float* scales, int64_t K, int64_t kb_stride, const PackGroups& pg,
                                      int64_t tiles_cap, uint8_t* atoms, unsigned int* status, int num_sms,
                                      cudaStream_t stream)
{
    const int64_t n = tiles_cap * 128 * (K / 128);
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    pack_ue8m0_grouped_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(scales, K / 128, kb_stride, pg,
                                                                                  tiles_cap, atoms, status);
    return cudaGetLastError();
}

cudaError_t launch_pack_ue8m0(const float* scales, int64_t rows, int64_t K, int row_block, int64_t row_stride,
                              int64_t kb_stride, uint8_t* atoms, unsigned int* status, int num_sms,
                              cudaStream_t stream)
{
    const int64_t rows_pad = (rows + 127) / 128 * 128;
    const int64_t n = rows_pad * (K / 128);
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    pack_ue8m0_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(scales, rows, rows_pad, K / 128, row_block,
                                                                         row_stride, kb_stride, atoms, status);
    return cudaGetLastError();
}

cudaError_t launch_mx_quant_1x32(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* atoms,
                                 int num_sms, cudaStream_t stream)
{
    const int64_t rows_pad = (rows + 127) / 128 * 128;
    const int64_t units = rows_pad * (cols / 128);
    if (units == 0) return cudaSuccess;
    int64_t blocks = (units * 16 + kMxQThreads - 1) / kMxQThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 64;
    if (blocks > cap) blocks = cap;
    mx_quant_1x32_kernel<<<static_cast<unsigned>(blocks), kMxQThreads, 0, stream>>>(x, rows, rows_pad, cols, q,
                                                                                    atoms);
    return cudaGetLastError();
}

cudaError_t launch_mx_quant_1x32_T(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* qT, uint8_t* atoms,
                                   cudaStream_t stream)
{
    const int64_t rows_pad = (rows + 127) / 128 * 128;
    const int64_t tiles = rows_pad / 128, cblocks = (cols + 127) / 128;
    if (tiles == 0 || cblocks == 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF || cblocks > 65535) return cudaErrorInvalidValue;
    mx_quant_1x32_T_kernel<<<dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(cblocks)), kMxTThreads, 0,
                             stream>>>(x, rows, cols, rows_pad, qT, atoms);
    return cudaGetLastError();
}

cudaError_t launch_mx_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap* map_out,
                           const uint8_t* sfa, const uint8_t* sfb, int M, int N, int K, uint16_t* out,
                           float* out_f32, const MxGroups& grp, int64_t max_tiles, uint64_t wait_limit_ns,
                           unsigned int* status, int num_sms, cudaStream_t stream)
{
    static_assert(sizeof(MxCtl) <= kCtlBytes, "control block");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    MxParams p;
    std::memset(&p, 0, sizeof(p));
    p.sfa = sfa;
    p.sfb = sfb;
    p.m_tiles = (M + kBM - 1) / kBM;
    p.n_tiles = N / kBN;
    p.kblocks = K / kBK;
    p.M = M;
    p.N = N;
    p.out = out;
    p.out_f32 = out_f32;
    p.tma_store = map_out != nullptr ? 1 : 0;
    p.grp = grp;
    CUtensorMap mo;
    if (p.tma_store) mo = *map_out;
    else std::memset(&mo, 0, sizeof(mo));
    p.wait_limit_ns = wait_limit_ns;
    p.status = status;
    if (max_tiles <= 0) return cudaSuccess;
    if (grp.b_mn && out_f32 != nullptr) return cudaErrorInvalidValue;
    auto kernel = out_f32 != nullptr ? mx_gemm_kernel<true, false>
                  : grp.b_mn         ? mx_gemm_kernel<false, true>
                                     : mx_gemm_kernel<false, false>;
    // once per device and kernel variant: the shared-memory opt-in, and a
    // check that the launch allocation covers the setmaxnreg split
    static std::atomic<uint64_t> ready[3];
    const int var = out_f32 != nullptr ? 1 : grp.b_mn ? 2 : 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(ready[var].load(std::memory_order_acquire) & bit)) {
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, kernel);
        if (e != cudaSuccess) return e;
        if (128u * kProducerRegs + 256u * kEpilogueRegs > static_cast<uint32_t>(kThreads) * attr.numRegs)
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        ready[var].fetch_or(bit, std::memory_order_release);
    }
    const int grid = max_tiles < num_sms ? static_cast<int>(max_tiles) : num_sms;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, mo, p);
    return cudaGetLastError();
}

}  // namespace fp8bs
