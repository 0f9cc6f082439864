// gemm.cu -- block-scaled E4M3 GEMM with per-128-K fp32 promotion on tcgen05.
//
// What it computes ("FP8 动态量化里的 partial sum 漂移", sections 3 and 5;
// "scratch: the backward pass, unrolled", "What is asserted, and from where",
// bullet 1): for every output element and every 128-element block b of the
// contraction, the tensor core forms the partial P_b over that block only;
// the partial is multiplied by s_a * s_b and added to an fp32 accumulator;
// the next block starts from zero. Output is BF16 (Fprop, Dgrad) or FP32
// (Wgrad).
//
// The pages describe this on Hopper (WGMMA into registers, promotion on the
// CUDA cores of the same warps). On sm_103a the partial lives in tensor
// memory instead, which decouples the two halves of the work:
//
//   warp 0      TMA producer: one thread streams 128x128 (A) and 256x128 (B)
//               E4M3 tiles (K-major, 128-byte swizzle; Fprop's B may instead
//               be W as stored, [K x N], which arrives MN-major in two
//               128-column boxes) into a 4-stage (Wgrad: 3)
//               shared-memory ring. For Wgrad it also copies each K-block's
//               scales (the tile's 128 row scales and 256 column scales) into
//               an 8-slot shared-memory ring with two untiled bulk copies
//               inside the stage's transaction (Fprop / Dgrad epilogue threads
//               need one scalar per K-block and prefetch it themselves, two
//               K-blocks ahead).
//   warp 1      MMA issuer: one thread issues four tcgen05.mma (K = 32 each)
//               per K-block into a fresh TMEM accumulator (the first with
//               accumulate = 0), double-buffered over 2 x 256 TMEM columns,
//               and commits to mbarriers that free the smem stage and hand
//               the partial to the epilogue.
//   warps 2-3   idle (they complete the first warpgroup, which gives its
//               registers to the epilogue with setmaxnreg).
//   warps 4-11  promotion epilogue: each warp owns 32 TMEM lanes (rows) and
//               128 columns; per K-block it loads the fp32 partial with
//               tcgen05.ld, releases the TMEM buffer, and does
//               acc = fma(P_b, s_a * s_b, acc) in registers; at the end of a
//               tile it converts and stores the accumulator (Fprop / Dgrad:
//               BF16 boxes through a per-warp swizzled stage, each leaving
//               with a TMA store; Wgrad: FP32 pairs from registers).
//
// The kernel is persistent (one CTA per SM, 128x256 output tiles in a
// grid-stride order) and handles groups (MoE experts) through a per-group
// table in its parameter block. Every wait is bounded: when one gives up the
// kernel records FP8BS_ERR_TIMEOUT, stops issuing work, drains its in-flight
// copies and MMAs, frees its tensor memory and returns.
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int kStages = 4;        // operand ring depth (Fprop / Dgrad; see num_stages)
constexpr int kABytes = kBM * kBK;  // 16 KB
constexpr int kBBytes = kBN * kBK;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 4;
constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;  // 384: three warpgroups
// Register split: the kernel is launched with kLaunchRegs per thread (the
// __launch_bounds__ budget); the producer warpgroup gives registers back and
// the two epilogue warpgroups take them. Before the first launch on a device
// the host checks that the compiled launch allocation covers the split, so
// that the split never asks for more than exists.
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kProducerRegs = 40;
constexpr uint32_t kEpilogueRegs = 232;
static_assert(128 * kProducerRegs + 256 * kEpilogueRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 2 * kBN;              // two accumulator buffers
// Waits that drain in-flight copies and MMAs before exit use at least this
// limit, so that a small user limit never lets a CTA exit with work in flight.
constexpr uint64_t kDrainLimitNs = 1000000000ull;
constexpr int kCtlBytes = 2048;                 // barriers, flags and the group table
// Wgrad scale ring: slot = the K-block's scales of the tile's 128 rows, then
// of its 256 columns.
constexpr int kScaleSlots = 8;
constexpr int kScaleSlotFloats = kBM + kBN;
constexpr int kScaleBytes = kScaleSlots * kScaleSlotFloats * 4;
// Fprop / Dgrad output stage: per epilogue warp 32 rows x 64 BF16 columns.
constexpr int kOutStageWarpBytes = 32 * 64 * 2;
constexpr int kOutStageBytes = kEpiWarps * kOutStageWarpBytes;
// Dynamic shared memory (1024-byte aligned pieces, as the 128-byte swizzle
// of the TMA boxes requires): the operand ring; the Fprop / Dgrad output
// stage or the Wgrad scale ring; the control block.
// Operand ring depth per kind: Wgrad, bound by its epilogue, measured
// faster with three stages than with four (78.5 against 80.5 us on the dense
// workload).
template <GemmKind kKind>
__host__ __device__ constexpr int num_stages()
{
    return kKind == GemmKind::kVectorScaleF32 ? 3 : kStages;
}
template <GemmKind kKind>
constexpr int extra_bytes()
{
    return kKind == GemmKind::kVectorScaleF32 ? kScaleBytes : kOutStageBytes;
}
static_assert(kStageBytes % 1024 == 0 && kScaleBytes % 1024 == 0 && kOutStageBytes % 1024 == 0,
              "shared-memory pieces keep 1024-byte alignment");
template <GemmKind kKind>
constexpr int smem_bytes()
{
    return num_stages<kKind>() * kStageBytes + extra_bytes<kKind>() + kCtlBytes + 1024 /* alignment */;
}

// Per-group table built at kernel start from the group offsets: for row
// groups the first tile of each group, for token groups the first K-block
// of each group in the padded token axis (its tiles start at g times the
// tiles per group). The offsets themselves are read again from the
// parameters or device memory when a tile starts.
struct GroupTab {
    int32_t start[kMaxGroups + 1];
    int32_t total_tiles;
    int32_t valid;
};

struct SharedCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t sempty[kScaleSlots];  // scale slot read by every epilogue warp
    uint64_t mma_done;        // final commit of the MMA thread (drain before exit)
    uint64_t sk_part;         // stream-K: every epilogue warp has written its part of the partial
    uint64_t sk_ready;        // stream-K: the continuation's partial has been published
    int sk_ok;                // stream-K: verdict of the wait for it
    uint32_t tmem_base;
    volatile int abort;
    GroupTab tab;
};

__device__ __forceinline__ void record_status(unsigned int* status, unsigned int code)
{
    atomicCAS(status, 0u, code);
}

// Everything the roles need about group g (see GroupLayout).
struct GroupInfo {
    int a_row0;      // first A row (= first output row)
    int a_rows;      // output rows
    int k0;          // first K element (TMA x coordinate)
    int kblocks;     // 128-element K-blocks
    int b_row0;      // first B row (TMA y coordinate)
    int sa_kb0;      // first scale K-block of A
    int64_t sb_off;  // float offset of the group's B scales
    int64_t out_off; // element offset of the group's output origin
    int out_row0;    // row of the output tensor map holding the group's output row 0
};

__device__ __forceinline__ int group_off(const GemmParams& p, int g)
{
    return p.off_dev ? __ldg(p.off_dev + g) : p.off[g];
}

__device__ __forceinline__ GroupInfo group_info(const GemmParams& p, const GroupTab& tab, int g)
{
    GroupInfo gi;
    if (p.layout == kRowGroups) {
        const int o0 = group_off(p, g), o1 = group_off(p, g + 1);
        gi.a_row0 = o0;
        gi.a_rows = o1 - o0;
        gi.k0 = 0;
        gi.kblocks = p.kblocks;
        gi.b_row0 = g * p.b_group_rows;
        gi.sa_kb0 = 0;
        gi.sb_off = static_cast<int64_t>(g) * p.sb_group_stride;
        gi.out_off = 0;
        gi.out_row0 = o0;
    } else {
        gi.a_row0 = 0;
        gi.a_rows = p.out_rows;
        gi.k0 = tab.start[g] * kBK;
        gi.kblocks = tab.start[g + 1] - tab.start[g];
        gi.b_row0 = 0;
        gi.sa_kb0 = tab.start[g];
        gi.sb_off = static_cast<int64_t>(tab.start[g]) * p.sb_kstride;
        gi.out_off = static_cast<int64_t>(g) * p.out_group_stride;
        gi.out_row0 = g * p.out_rows;
    }
    return gi;
}

// Builds the group table (all threads of the CTA take part; ends with a CTA
// barrier). Invalid offsets (off[0] != 0, a decrease, a total other than
// rows_total for row groups, more padded tokens than tcap for token groups)
// leave no tiles and record FP8BS_ERR_DEVICE.
__device__ void build_group_tab(const GemmParams& p, GroupTab& tab)
{
    const int G = p.num_groups;
    int bad = 0;
    // per-group counts (row groups: tiles; token groups: K-blocks), then an
    // exclusive scan by warp 0 (up to eight groups per lane)
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const int n = group_off(p, g + 1) - group_off(p, g);
        if (n < 0) bad = 1;
        const int nb = n < 0 ? 0 : (n + kBK - 1) / kBK;
        tab.start[g] = p.layout == kRowGroups ? nb * p.n_tiles : nb;
    }
    if (threadIdx.x == 0) {
        if (group_off(p, 0) != 0) bad = 1;
        if (p.layout == kRowGroups && group_off(p, G) != p.rows_total) bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (G + 31) / 32;
        const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
        int sum = 0;
        for (int g = g0; g < g1; ++g) sum += tab.start[g];
        int inc = sum;   // inclusive warp scan of the lanes' sums
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if (lane >= d) inc += v;
        }
        int run = inc - sum;   // exclusive prefix of this lane's first group
        for (int g = g0; g < g1; ++g) {
            const int c = tab.start[g];
            tab.start[g] = run;
            run += c;
        }
        if (lane == 31) {
            tab.start[G] = inc;
            const int total = p.layout == kRowGroups ? inc : G * (p.out_rows / kBM) * p.n_tiles;
            const bool over = p.layout == kTokenGroups && static_cast<int64_t>(inc) * kBK > p.tcap;
            tab.valid = (bad || over) ? 0 : 1;
            tab.total_tiles = (bad || over) ? 0 : total;
            if ((bad || over) && blockIdx.x == 0) record_status(p.status, FP8BS_ERR_DEVICE);
        }
    }
    __syncthreads();
}

__device__ __forceinline__ void decode_tile(const GemmParams& p, const GroupTab& tab, int t, int& g, int& mt,
                                            int& nt)
{
    int local;
    if (p.layout == kRowGroups) {
        int lo = 0, hi = p.num_groups - 1;  // last g with start[g] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tab.start[mid] <= t) lo = mid; else hi = mid - 1;
        }
        g = lo;
        local = t - tab.start[g];
    } else {
        const int per = (p.out_rows / kBM) * p.n_tiles;
        g = t / per;
        local = t - g * per;
    }
    mt = local / p.n_tiles;
    nt = local - mt * p.n_tiles;
}

// Work unit u of the persistent loop (CTA u % gridDim.x, its (u / gridDim.x)-th
// unit): tile u / splits and its split-K range, or with stream-K the
// (u / gridDim.x)-th tile segment of CTA u % gridDim.x's K-block range
// (nkb = 0 past the CTA's last segment). The host enables stream-K only when
// tiles x K-blocks fits in 31 bits.
__device__ __forceinline__ GroupInfo decode_unit(const GemmParams& p, const GroupTab& tab, int u, int& g, int& mt,
                                                 int& nt, int& split, int& kb0, int& nkb)
{
    if (p.sk_len != 0) {
        const int c = u % static_cast<int>(gridDim.x);
        const int j = u / static_cast<int>(gridDim.x);
        const int nk = p.kblocks;
        const int begin = c * p.sk_len;
        const int end = min(tab.total_tiles * nk, begin + p.sk_len);
        const int t0 = begin / nk;
        const int start = j == 0 ? begin : (t0 + j) * nk;
        const int t = min(t0 + j, tab.total_tiles - 1);
        kb0 = start - t * nk;
        nkb = start < end ? min(end, (t + 1) * nk) - start : 0;
        split = 0;
        decode_tile(p, tab, t, g, mt, nt);
        return group_info(p, tab, g);
    }
    const int t = u / p.splits;
    split = u - t * p.splits;
    decode_tile(p, tab, t, g, mt, nt);
    const GroupInfo gi = group_info(p, tab, g);
    kb0 = split * p.kb_per_split;
    const int end = min(gi.kblocks, kb0 + p.kb_per_split);
    nkb = max(0, end - kb0);
    return gi;
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned int* p, unsigned int v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Promotion epilogues (warps 4-11). Each warp owns the 32 TMEM lanes (tile
// rows) of its quarter and one 128-column half of the tile. Both return
// false when a wait gave up.
// ---------------------------------------------------------------------------

// Fprop / Dgrad (row groups: A rows are output rows, no K offset, B scales
// at g * sb_group_stride): s_b is one value per 128 output columns, so a K-block's
// scale is one scalar per thread (row) and half. Layout 32x32b: thread =
// row, 128 columns in registers. The BF16 output goes through a per-warp
// shared-memory stage so that every global store instruction writes four
// whole 128-byte row segments (the tile ends of all CTAs coincide, and
// 16-byte pieces of 32 different rows per instruction made those bursts
// several times longer).
__device__ __forceinline__ bool epilogue_block_scale(const GemmParams& p, SharedCtl* ctl, uint8_t* out_stage,
                                                     const CUtensorMap* map_out, uint32_t tmem_base, int warp,
                                                     int lane, uint64_t limit)
{
    const int ew = warp - kFirstEpiWarp;
    const int quarter = warp & 3;   // TMEM lanes this warp may access
    const int half = ew >> 2;       // 128-column half of the tile
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc_it = 0;

    const int units = p.sk_len ? static_cast<int>(gridDim.x) * p.sk_units : ctl->tab.total_tiles * p.splits;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        int g, mt, nt, split, kb0, nkb;
        int row0, nrows;   // the group's first row and row count (row groups: A rows = output rows)
        int tile_kb;       // the tile's K-blocks (stream-K: nkb may cover part of them)
        {
            const GroupInfo gi = decode_unit(p, ctl->tab, u, g, mt, nt, split, kb0, nkb);
            row0 = gi.a_row0;
            nrows = gi.a_rows;
            tile_kb = gi.kblocks;
        }
        if (p.sk_len != 0 && nkb == 0) continue;   // stream-K: past this CTA's last segment
        // stream-K role of this segment: 1 = continuation of a cut tile (the
        // CTA's first segment), 2 = owner of a cut tile (its last), 0 = whole tile
        const int sk_role = p.sk_len == 0 ? 0 : (kb0 > 0 ? 1 : (nkb < tile_kb ? 2 : 0));
        const int row = row0 + mt * kBM + r_in_tile;
        const bool row_ok = (mt * kBM + r_in_tile) < nrows;
        const int col0 = nt * kBN + half * 128;
        const bool cols_ok = col0 < p.n_cols;                  // n_cols % 128 == 0
        const bool sa_ok = row < p.sa_rows;
        const float* sa_ptr = p.sa + static_cast<int64_t>(kb0) * p.sa_ld + row;
        const float* sb_ptr = p.sb + static_cast<int64_t>(g) * p.sb_group_stride + static_cast<int64_t>(col0 / 128) * p.sb_cstride +
                              static_cast<int64_t>(kb0) * p.sb_kstride;

        auto load_sa = [&](int kb) -> float {
            return (sa_ok && kb < nkb) ? __ldg(sa_ptr + static_cast<int64_t>(kb) * p.sa_ld) : 0.0f;
        };
        auto load_sb = [&](int kb) -> float {
            return (cols_ok && kb < nkb) ? __ldg(sb_ptr + static_cast<int64_t>(kb) * p.sb_kstride) : 0.0f;
        };

        float2 acc[64];     // 128 fp32 accumulators as 64 pairs (packed f32x2 math)
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = make_float2(0.f, 0.f);

        // scalar scales two K-blocks ahead in registers
        float sa0 = load_sa(0), sa1 = load_sa(1), sb0 = load_sb(0), sb1 = load_sb(1);

        for (int kb = 0; kb < nkb; ++kb, ++acc_it) {
            const float s_blk = sa0 * sb0;
            sa0 = sa1;
            sa1 = load_sa(kb + 2);
            sb0 = sb1;
            sb1 = load_sb(kb + 2);
            const float2 s_blk2 = make_float2(s_blk, s_blk);

            const uint32_t buf = acc_it & 1u;
            const uint32_t aph = (acc_it >> 1) & 1u;
            if (ctl->abort || !mbar_wait(&ctl->tfull[buf], aph, limit)) return false;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + lane_addr + buf * kBN + half * 128;

            // promote one 32-column chunk of the partial held in r
            auto promote = [&](int c, uint32_t (&r)[32]) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[c * 16 + i] = __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                                 s_blk2, acc[c * 16 + i]);
            };
            // TMEM loads double-buffered: chunk c + 1 is in flight while
            // chunk c is promoted
            uint32_t ra[32], rb[32];
            tmem_ld_x32(taddr + 0, ra);
            tmem_ld_wait(ra);
            tmem_ld_x32(taddr + 32, rb);
            promote(0, ra);
            tmem_ld_wait(rb);
            tmem_ld_x32(taddr + 64, ra);
            promote(1, rb);
            tmem_ld_wait(ra);
            tmem_ld_x32(taddr + 96, rb);
            promote(2, ra);
            tmem_ld_wait(rb);
            // the partial is in registers: hand the TMEM buffer back
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0 && !p.hold_release) mbar_arrive(&ctl->tempty[buf]);
            promote(3, rb);
        }

        if (sk_role == 1) {
            // stream-K continuation (this CTA's first segment): the fp32 sum
            // goes to the CTA's workspace slot, float4 v of thread et at
            // [v][et], and the slot is published for the tile's owner (CTA
            // blockIdx.x - 1) once all eight warps have written their parts
            const int et = ew * 32 + lane;
            float4* slot = reinterpret_cast<float4*>(p.sk_ws) + static_cast<int64_t>(blockIdx.x) * 32 * 256;
#pragma unroll
            for (int v = 0; v < 32; ++v)
                slot[v * 256 + et] = make_float4(acc[2 * v].x, acc[2 * v].y, acc[2 * v + 1].x, acc[2 * v + 1].y);
            __threadfence();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->sk_part);
            if (ew == 0 && lane == 0) {
                if (!mbar_wait(&ctl->sk_part, 0u, limit)) return false;
                st_release_gpu(p.sk_flags + blockIdx.x, 1u);
            }
            continue;
        }
        if (sk_role == 2) {
            // stream-K owner of a cut tile (this CTA's last segment): add the
            // rest of the tile, which CTA blockIdx.x + 1 computed first
            if (ew == 0 && lane == 0) {
                unsigned int* flag = p.sk_flags + blockIdx.x + 1;
                bool got = ld_acquire_gpu(flag) == 1u;
                const uint64_t t0 = global_timer_ns();
                while (!got && !ctl->abort) {
                    __nanosleep(64);
                    got = ld_acquire_gpu(flag) == 1u;
                    if (!got && global_timer_ns() - t0 > limit) break;
                }
                if (got) *flag = 0u;   // consumed: the slot is free for the next launch
                ctl->sk_ok = got ? 1 : 0;
                mbar_arrive(&ctl->sk_ready);
            }
            int ready = 0;
            if (lane == 0) ready = mbar_wait(&ctl->sk_ready, 0u, limit) ? 1 : 0;
            ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
            if (ready) mbar_try_wait(&ctl->sk_ready, 0u);
            if (!ready || !ctl->sk_ok) return false;
            const int et = ew * 32 + lane;
            const float4* slot =
                reinterpret_cast<const float4*>(p.sk_ws) + static_cast<int64_t>(blockIdx.x + 1) * 32 * 256;
#pragma unroll
            for (int v = 0; v < 32; ++v) {
                const float4 x = __ldcg(slot + v * 256 + et);
                acc[2 * v] = make_float2(acc[2 * v].x + x.x, acc[2 * v].y + x.y);
                acc[2 * v + 1] = make_float2(acc[2 * v + 1].x + x.z, acc[2 * v + 1].y + x.w);
            }
        }

        if (p.ws != nullptr) {
            if (cols_ok) {
                // split-K: this range's fp32 sum of the tile goes to its own
                // slot of the workspace, float4 v of thread et at [v][et], so
                // every warp store is 512 contiguous bytes (rows past the
                // output hold zeros and are never read back)
                const int et = ew * 32 + lane;
                float4* slot = reinterpret_cast<float4*>(p.ws + static_cast<int64_t>(split) * p.ws_split_stride) +
                               (static_cast<int64_t>(mt) * p.n_tiles + nt) * 32 * 256;
#pragma unroll
                for (int v = 0; v < 32; ++v)
                    slot[v * 256 + et] = make_float4(acc[2 * v].x, acc[2 * v].y, acc[2 * v + 1].x, acc[2 * v + 1].y);
            }
        } else if (cols_ok) {
            // Two rounds of 64 columns: each thread writes its row's 64 values
            // as eight 16-byte chunks (chunk c of row r at slot c ^ (r % 8):
            // conflict-free, and the 128-byte swizzle of a TMA box). When the
            // warp's 32 rows all belong to this group, one TMA store per round
            // writes the box while the warp goes on; otherwise lanes 8q .. 8q + 7
            // store one row's 128 contiguous bytes, four rows per instruction.
            const int rows_left = nrows - (mt * kBM + quarter * 32);   // valid rows of this warp
            const int out_row = row0 + mt * kBM + quarter * 32;
            const bool tma = p.tma_store && rows_left >= 32;
            uint16_t* y0 = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(out_row) * p.out_ld + col0;
            const uint32_t st_base = smem_addr(out_stage) + ew * kOutStageWarpBytes;
#pragma unroll
            for (int rnd = 0; rnd < 2; ++rnd) {
                // the stage's previous box has been read by its TMA store
                if (lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float2 a0 = acc[32 * rnd + 4 * c + 0];
                    const float2 a1 = acc[32 * rnd + 4 * c + 1];
                    const float2 a2 = acc[32 * rnd + 4 * c + 2];
                    const float2 a3 = acc[32 * rnd + 4 * c + 3];
                    uint4 pk;
                    pk.x = pack_bf16x2(a0.x, a0.y);
                    pk.y = pack_bf16x2(a1.x, a1.y);
                    pk.z = pack_bf16x2(a2.x, a2.y);
                    pk.w = pack_bf16x2(a3.x, a3.y);
                    st_shared_v4(st_base + lane * 128 + ((c ^ (lane & 7)) << 4), pk);
                }
                if (tma) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(map_out, st_base, col0 + 64 * rnd, out_row);
                        bulk_commit_group();
                    }
                } else {
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = 4 * i + (lane >> 3);
                        const int c = lane & 7;
                        const uint4 v = ld_shared_v4(st_base + rr * 128 + ((c ^ (rr & 7)) << 4));
                        if (rr < rows_left)
                            *reinterpret_cast<uint4*>(y0 + static_cast<int64_t>(rr) * p.out_ld + 64 * rnd + 8 * c) = v;
                    }
                    __syncwarp();
                }
            }
        }
    }
    return true;
}

// Wgrad: both scales are vectors (one per output row and one per output
// column for every K-block), so every element needs its own s_a * s_b. With
// the 32x32b layout each thread would need all 128 column scales of its half
// every K-block, read as shared-memory broadcasts that cost more load
// bandwidth than the MMA leaves room for. The 16x256b layout spreads the
// tile as 4 rows x 32 columns per thread: a K-block then needs 4 row scales
// and 16 column-scale pairs per thread, read from the slot of the scale ring
// that the TMA producer filled with the K-block's operand stage (the tile's
// 128 row scales, then its 256 column scales).
__device__ __forceinline__ bool epilogue_vector_scale(const GemmParams& p, SharedCtl* ctl, const float* ring,
                                                      uint32_t tmem_base, int warp, int lane, uint64_t limit)
{
    const int ew = warp - kFirstEpiWarp;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const int g4 = lane >> 2;       // row within each group of 8
    const int t4 = lane & 3;        // column pair within each group of 8
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc_it = 0;

    const int units = ctl->tab.total_tiles * p.splits;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        int g, mt, nt, split, kb0, nkb;
        const GroupInfo gi = decode_unit(p, ctl->tab, u, g, mt, nt, split, kb0, nkb);
        const int qrow0 = mt * kBM + quarter * 32;             // first tile row of this quarter
        const int col0 = nt * kBN + half * 128;
        const bool cols_ok = col0 < p.n_cols;                  // n_cols % 128 == 0

        float2 acc[4][16];   // [row i: g4 + 8 i][column group j: 8 j + 2 t4, + 1]
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[i][j] = make_float2(0.f, 0.f);

        for (int kb = 0; kb < nkb; ++kb, ++acc_it) {
            const uint32_t ss = acc_it % kScaleSlots;
            const float* slot = ring + ss * kScaleSlotFloats;
            const uint32_t buf = acc_it & 1u;
            const uint32_t aph = (acc_it >> 1) & 1u;
            if (ctl->abort || !mbar_wait(&ctl->tfull[buf], aph, limit)) return false;
            tc_fence_after_sync();
            // this K-block's scales from the ring: the warp's 4 row scales in
            // registers, the column scales read from the slot while promoting
            // (the slot landed with the K-block's operand stage, before its
            // MMAs were issued, so the wait for the partial above orders it)
            float2 sa2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float v = slot[quarter * 32 + g4 + 8 * i];
                sa2[i] = make_float2(v, v);
            }
            const float2* sbp = reinterpret_cast<const float2*>(slot + kBM + half * 128) + t4;
            const uint32_t taddr = tmem_base + lane_addr + buf * kBN + half * 128;

            // promote the 32-column group c (rows g4, g4 + 8 in r[0..15],
            // rows g4 + 16, g4 + 24 in r[16..31])
            auto promote = [&](int c, uint32_t (&r)[32]) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = 4 * c + jj;
                    const float2 sb = sbp[4 * j];     // columns 8 j + 2 t4, + 1
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int k = 16 * (i >> 1) + 4 * jj + 2 * (i & 1);
                        acc[i][j] = __ffma2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                                               __fmul2_rn(sa2[i], sb), acc[i][j]);
                    }
                }
            };
            uint32_t ra[32], rb[32];
            tmem_ld_16x256b_x4_pair(taddr + 0, ra);
            tmem_ld_wait(ra);
            tmem_ld_16x256b_x4_pair(taddr + 32, rb);
            promote(0, ra);
            tmem_ld_wait(rb);
            tmem_ld_16x256b_x4_pair(taddr + 64, ra);
            promote(1, rb);
            tmem_ld_wait(ra);
            tmem_ld_16x256b_x4_pair(taddr + 96, rb);
            promote(2, ra);
            tmem_ld_wait(rb);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0 && !p.hold_release) mbar_arrive(&ctl->tempty[buf]);
            promote(3, rb);
            // the slot's column scales have been read
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->sempty[ss]);
        }

        if (cols_ok) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r_tile = qrow0 + g4 + 8 * i;
                if (r_tile >= gi.a_rows) continue;
                float* y = static_cast<float*>(p.out) + gi.out_off +
                           static_cast<int64_t>(gi.a_row0 + r_tile) * p.out_ld + col0 + 2 * t4;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float2 v = acc[i][j];
                    float2* dst = reinterpret_cast<float2*>(y + 8 * j);
                    if (p.accumulate) {
                        const float2 prev = *dst;
                        v = __fadd2_rn(v, prev);
                    }
                    *dst = v;
                }
            }
        }
    }
    return true;
}

template <GemmKind kKind>
__global__ void __launch_bounds__(kThreads, 1)
    block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                             const __grid_constant__ CUtensorMap map_b,
                             const __grid_constant__ CUtensorMap map_out,
                             const __grid_constant__ GemmParams p)
{
    constexpr int kS = num_stages<kKind>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kS * kABytes;
    uint8_t* extra = smem + kS * kStageBytes;   // output stage or scale ring
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(extra + extra_bytes<kKind>());
    float* scale_ring = reinterpret_cast<float*>(extra);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&ctl->tfull[a], 1);
            mbar_init(&ctl->tempty[a], kEpiWarps);
        }
        for (int a = 0; a < kScaleSlots; ++a) mbar_init(&ctl->sempty[a], kEpiWarps);
        mbar_init(&ctl->mma_done, 1);
        mbar_init(&ctl->sk_part, kEpiWarps);
        mbar_init(&ctl->sk_ready, 1);
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
    build_group_tab(p, ctl->tab);
    const uint32_t tmem_base = ctl->tmem_base;
    const uint64_t limit = p.wait_limit_ns;

    if (warp < kFirstEpiWarp) {
        setmaxnreg_dec<kProducerRegs>();
    }
    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            const int units = p.sk_len ? static_cast<int>(gridDim.x) * p.sk_units : ctl->tab.total_tiles * p.splits;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int g, mt, nt, split, kb0, nkb;
                const GroupInfo gi = decode_unit(p, ctl->tab, u, g, mt, nt, split, kb0, nkb);
                const int ya = gi.a_row0 + mt * kBM;
                const int yb = gi.b_row0 + nt * kBN;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % kS;
                    const uint32_t ph = (it / kS) & 1u;
                    if (ctl->abort || !mbar_wait(&ctl->empty[s], ph ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    const int x = gi.k0 + (kb0 + kb) * kBK;
                    if constexpr (kKind == GemmKind::kVectorScaleF32) {
                        // Wgrad: this K-block's 128 row scales and the tile's
                        // column scales go into the scale ring as part of the
                        // stage's transaction, so they have landed before the
                        // stage's MMAs are issued and hence before the
                        // epilogue sees the partial (it needs no wait of its
                        // own); the slot is reused once the epilogue released it
                        const uint32_t ss = it % kScaleSlots;
                        if (ctl->abort || !mbar_wait(&ctl->sempty[ss], ((it / kScaleSlots) & 1u) ^ 1u, limit)) {
                            ok = false;
                            break;
                        }
                        const uint32_t b_bytes = static_cast<uint32_t>(min(kBN, p.n_cols - nt * kBN)) * 4u;
                        float* slot = scale_ring + ss * kScaleSlotFloats;
                        mbar_arrive_expect_tx(&ctl->full[s], kStageBytes + kBM * 4u + b_bytes);
                        bulk_load(slot, p.sa + static_cast<int64_t>(gi.sa_kb0 + kb0 + kb) * p.sa_ld + ya, kBM * 4u,
                                  &ctl->full[s]);
                        bulk_load(slot + kBM,
                                  p.sb + gi.sb_off + static_cast<int64_t>(kb0 + kb) * p.sb_kstride + nt * kBN,
                                  b_bytes, &ctl->full[s]);
                    } else {
                        mbar_arrive_expect_tx(&ctl->full[s], kStageBytes);
                    }
                    tma_load_2d(sA + s * kABytes, &map_a, &ctl->full[s], x, ya);
                    if (kKind == GemmKind::kBlockScaleBf16 && p.b_mn) {
                        // MN-major B: K rows x 128 columns per box, the
                        // tile's two column halves one box apart
                        const int yk = gi.b_row0 + x;
                        tma_load_2d(sB + s * kBBytes, &map_b, &ctl->full[s], nt * kBN, yk);
                        tma_load_2d(sB + s * kBBytes + kBBytes / 2, &map_b, &ctl->full[s], nt * kBN + kBN / 2, yk);
                    } else {
                        tma_load_2d(sB + s * kBBytes, &map_b, &ctl->full[s], x, yb);
                    }
                }
            }
            if (!ok) {
                record_status(p.status, FP8BS_ERR_TIMEOUT);
                ctl->abort = 1;
            }
            // drain: every issued copy has landed before the CTA can exit
            const uint32_t first = it > kS ? it - kS : 0u;
            const uint64_t drain = limit > kDrainLimitNs ? limit : kDrainLimitNs;
            for (uint32_t j = first; j < it; ++j)
                mbar_wait(&ctl->full[j % kS], (j / kS) & 1u, drain);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer
        // ------------------------------------------------------------------
        if (lane == 0) {
            const bool b_mn = kKind == GemmKind::kBlockScaleBf16 && p.b_mn != 0;   // Fprop only
            const uint32_t idesc = idesc_e4m3_f32(kBM, kBN) | (b_mn ? kIdescBMajorMN : 0u);
            // start-address step of B per 32 K (in 16-byte units): 32 bytes
            // inside the swizzle row (K-major), 32 K rows = 4096 bytes (MN-major)
            const uint64_t b_step = b_mn ? 4096u >> 4 : 32u >> 4;
            uint32_t it = 0, acc_it = 0;
            bool ok = true;
            const int units = p.sk_len ? static_cast<int>(gridDim.x) * p.sk_units : ctl->tab.total_tiles * p.splits;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int g, mt, nt, split, kb0, nkb;
                const GroupInfo gi = decode_unit(p, ctl->tab, u, g, mt, nt, split, kb0, nkb);
                for (int kb = 0; kb < nkb; ++kb, ++it, ++acc_it) {
                    const uint32_t s = it % kS;
                    const uint32_t ph = (it / kS) & 1u;
                    const uint32_t buf = acc_it & 1u;
                    const uint32_t aph = (acc_it >> 1) & 1u;
                    if (ctl->abort || !mbar_wait(&ctl->tempty[buf], aph ^ 1u, limit) ||
                        !mbar_wait(&ctl->full[s], ph, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(sA + s * kABytes));
                    const uint64_t bdesc = b_mn ? sdesc_mnmajor_sw128(smem_addr(sB + s * kBBytes), kBBytes / 2)
                                                : sdesc_kmajor_sw128(smem_addr(sB + s * kBBytes));
                    const uint32_t d = tmem_base + buf * kBN;
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        mma_e4m3(d, adesc + 2u * kk, bdesc + b_step * kk, idesc, kk > 0 ? 1u : 0u);
                    mma_commit(&ctl->empty[s]);
                    mma_commit(&ctl->tfull[buf]);
                }
            }
            if (!ok) {
                record_status(p.status, FP8BS_ERR_TIMEOUT);
                ctl->abort = 1;
            }
            // drain: every MMA this thread issued has completed
            mma_commit(&ctl->mma_done);
            const uint64_t drain = limit > kDrainLimitNs ? limit : kDrainLimitNs;
            mbar_wait(&ctl->mma_done, 0u, drain);
        }
    } else if (warp >= kFirstEpiWarp) {
        // ------------------------------------------------------------------
        // Promotion epilogue
        // ------------------------------------------------------------------
        setmaxnreg_inc<kEpilogueRegs>();
        bool ok;
        if constexpr (kKind == GemmKind::kBlockScaleBf16)
            ok = epilogue_block_scale(p, ctl, extra, &map_out, tmem_base, warp, lane, limit);
        else
            ok = epilogue_vector_scale(p, ctl, scale_ring, tmem_base, warp, lane, limit);
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

// Split-K reduction: out = BF16(sum over splits s = 0, 1, ... of ws[s]), in
// that order (the result does not depend on scheduling). Eight elements per
// thread: two 16-byte loads per split, one 16-byte store.
// The split-K reduction: the ranges' fp32 sums of output tile t, laid out
// by the GEMM epilogue as [v][et] float4 (thread et = epilogue warp w x 32
// + lane holds row 32 (w % 4) + lane and columns 128 (w / 4) + 4 v .. + 3 of
// the tile), are added in range order and rounded to BF16 once. One thread
// per float4: reads coalesced along et, 8-byte writes of four BF16 values.
__global__ void __launch_bounds__(256) splitk_reduce_bf16_kernel(const float4* __restrict__ ws, int splits,
                                                                 int64_t split_stride4, int n_tiles, int64_t rows,
                                                                 int64_t cols, uint16_t* __restrict__ out)
{
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < split_stride4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = i / (32 * 256);
        const int rem = static_cast<int>(i - tile * (32 * 256));
        const int v = rem >> 8, et = rem & 255;
        const int w = et >> 5, lane = et & 31;
        const int64_t mt = tile / n_tiles, nt = tile - mt * n_tiles;
        const int64_t row = mt * kBM + (w & 3) * 32 + lane;
        const int64_t col = nt * kBN + (w >> 2) * 128 + 4 * v;
        if (row >= rows || col >= cols) continue;
        float4 a = __ldcs(ws + i);
        for (int s = 1; s < splits; ++s) {
            const float4 c = __ldcs(ws + s * split_stride4 + i);
            a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
        }
        *reinterpret_cast<uint2*>(out + row * cols + col) = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
    }
}

__global__ void selftest_wait_kernel(unsigned int* status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // nothing ever arrives: phase 0 never completes, so the wait must give up
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, limit_ns)) record_status(status, FP8BS_ERR_TIMEOUT);
}

template <GemmKind kKind>
cudaError_t launch_kind(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                        const GemmParams& p, int64_t max_units, int num_sms, cudaStream_t stream)
{
    static_assert(sizeof(SharedCtl) <= kCtlBytes, "control block");
    auto kernel = block_scaled_gemm_kernel<kKind>;
    constexpr int kSmemBytes = smem_bytes<kKind>();
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    // once per device: the shared-memory opt-in, and a check that the
    // launch allocation covers the setmaxnreg split (a split above it would
    // wait forever)
    static std::atomic<uint64_t> ready{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(ready.load(std::memory_order_acquire) & bit)) {
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, kernel);
        if (e != cudaSuccess) return e;
        if (128u * kProducerRegs + 256u * kEpilogueRegs > static_cast<uint32_t>(kThreads) * attr.numRegs)
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        ready.fetch_or(bit, std::memory_order_release);
    }
    const int grid = max_units < num_sms ? static_cast<int>(max_units) : num_sms;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, map_out, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_splitk_reduce(const float* ws, int splits, int64_t rows, int64_t cols, uint16_t* out, int num_sms,
                                 cudaStream_t stream)
{
    const int64_t n_tiles = (cols + kBN - 1) / kBN;
    const int64_t split_stride4 = splitk_tile_floats(rows, cols) / 4;
    if (split_stride4 <= 0) return cudaSuccess;
    int64_t blocks = (split_stride4 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    splitk_reduce_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(ws), splits, split_stride4, static_cast<int>(n_tiles), rows, cols, out);
    return cudaGetLastError();
}

cudaError_t launch_gemm(GemmKind kind, const CUtensorMap& map_a, const CUtensorMap& map_b,
                        const CUtensorMap& map_out, const GemmParams& p, int64_t max_units, int num_sms,
                        cudaStream_t stream)
{
    if (max_units <= 0) return cudaSuccess;
    if (kind == GemmKind::kBlockScaleBf16)
        return launch_kind<GemmKind::kBlockScaleBf16>(map_a, map_b, map_out, p, max_units, num_sms, stream);
    return launch_kind<GemmKind::kVectorScaleF32>(map_a, map_b, map_out, p, max_units, num_sms, stream);
}

cudaError_t launch_selftest_wait(unsigned int* status, uint64_t limit_ns, cudaStream_t stream)
{
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace fp8bs
