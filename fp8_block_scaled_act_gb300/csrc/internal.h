// internal.h -- declarations shared by the library's translation units
// (kernel launchers and their parameter blocks). Not part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8bs.h"

namespace fp8bs {

constexpr int kMaxGroups = FP8BS_MAX_GROUPS;

// ---------------------------------------------------------------------------
// Quantizers
// ---------------------------------------------------------------------------

// How a tile's scale follows from its absmax (the default {0, 0, 0} is the
// plain rule s = amax / 448, 1 for an all-zero tile).
struct ScaleRule {
    int ue8m0;          // 1: round s up to a power of two
    float amax_floor;   // amax = max(amax, amax_floor) before the division
    float scale_floor;  // s = max(s, scale_floor)
};

// Stochastic rounding key (NULL pointer: round to nearest).
struct SrParams {
    uint64_t seed;
    uint32_t salt;
};

cudaError_t launch_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t* q, float* scales, int64_t scale_ld, const ScaleRule& rule,
                               const SrParams* sr, int num_sms, cudaStream_t stream);

// The round-to-nearest 1x128 cast fed by TMA: map_x is a BF16 map over the
// source [rows x cols] (row pitch of the caller's leading dimension) with a
// box of 64 columns x 32 rows, 128-byte swizzle, zero fill out of bounds;
// map_q a byte map over the codes [rows x cols] with a box of 128 columns x
// 32 rows, 128-byte swizzle. A load that does not land within limit_ns
// records FP8BS_ERR_TIMEOUT in *status.
cudaError_t launch_quant_1x128_stream(const CUtensorMap& map_x, const CUtensorMap& map_q, int64_t rows,
                                      int64_t cols, float* scales, int64_t scale_ld, const ScaleRule& rule,
                                      uint64_t limit, unsigned int* status, int num_sms, cudaStream_t stream);

// atoms_wT / atoms_w (nullable; rows and cols multiples of 128): the MX
// scale atoms of the two GEMM operands the weight feeds, W^T [cols x rows]
// and W [rows x cols] (contraction along cols), per batch entry; a scale
// without an exponent byte records FP8BS_ERR_DEVICE in *status.
cudaError_t launch_quant_128x128(const uint16_t* w, int64_t batch, int64_t rows, int64_t cols,
                                 int64_t ldw, uint8_t* q, uint8_t* qT, float* scales,
                                 const ScaleRule& rule, const SrParams* sr, cudaStream_t stream,
                                 uint8_t* atoms_wT = nullptr, uint8_t* atoms_w = nullptr,
                                 unsigned int* status = nullptr);

struct RequantParams {
    int mode;                  // FP8BS_SRC_BF16 or FP8BS_SRC_E4M3
    const void* src;           // [rows x cols], dense
    const float* src_scales;   // mode E4M3: 1x128 scales, tile-major
    int64_t src_scale_ld;
    int64_t rows, cols;
    uint8_t* qT;               // [cols x mpad]
    float* scT;                // [mpad/128 x cols]
    int64_t mpad;
    int num_groups;
    int32_t off[kMaxGroups + 1];         // row offsets of the groups
    int32_t tile_start[kMaxGroups + 1];  // first padded token tile of each group
    // Device offsets (num_groups + 1 entries): when set, off / tile_start
    // are unused and each CTA derives its group from them; the grid covers
    // the largest padded token count any split of `rows` can need, and CTAs
    // past the actual count do nothing.
    const int32_t* off_dev;
    // Optional, BF16 source only: the same block's 1x128 (row-wise) cast in
    // the same pass, q [rows x cols] and its scales [cols/128 x q_scale_ld].
    uint8_t* q;
    float* q_scales;
    int64_t q_scale_ld;
    // With q: take the transposed cast from the E4M3 result q instead of
    // from the BF16 source (the E4M3 source mode applied to q, q_scales).
    int stash;
    ScaleRule rule;
    // Stochastic rounding (sr != 0): the 1x128 part takes (seed, salt_rows),
    // the transposed part (seed, salt_cols); source element (r, c) uses the
    // word of index r * cols + c.
    int sr;
    uint64_t sr_seed;
    uint32_t sr_salt_rows, sr_salt_cols;
    // Optional (dense only): the exponent bytes of the scales in the MX
    // scale atoms of q [rows x cols] and of qT [cols x mpad]; a scale
    // without a byte records FP8BS_ERR_DEVICE in *status.
    uint8_t* q_atoms;
    uint8_t* qT_atoms;
    unsigned int* status;
};

cudaError_t launch_requant_128x1_T(const RequantParams& p, cudaStream_t stream);
// The round-to-nearest 128x128 cast on the TMA-fed tile kernel: map_w over
// the BF16 weights as [batch][rows][cols] (box 64 columns x 128 rows x 1,
// 128-byte swizzle), map_q over q the same way (box 128 bytes x 128 rows x 1).
cudaError_t launch_wcast_tile(const CUtensorMap& map_w, const CUtensorMap& map_q, int64_t batch, int64_t rows,
                              int64_t cols, uint8_t* qT, float* scales, const ScaleRule& rule, uint8_t* atoms_wT,
                              uint8_t* atoms_w, unsigned int* status, uint64_t limit, int num_sms,
                              cudaStream_t stream);
// The dense, round-to-nearest dual and stash casts (p.q set, p.mode BF16, no
// groups, no stochastic rounding) on the TMA-fed tile kernel: map_x over the
// BF16 source (box 64 columns x 128 rows, 128-byte swizzle), map_q over q
// (box 128 bytes x 128 rows, 128-byte swizzle).
cudaError_t launch_dual_tile(const CUtensorMap& map_x, const CUtensorMap& map_q, const RequantParams& p,
                             uint64_t limit, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Block-scaled GEMM (tcgen05)
// ---------------------------------------------------------------------------

// One output problem of the persistent GEMM kernel is a set of groups given
// by row offsets off[0..num_groups] (off[0] = 0, non-decreasing). The kernel
// derives each group's tiles, K range and operand offsets from the offsets
// in shared memory at start-up, reading them from off_dev (device memory)
// when it is set and from off[] otherwise. Dense GEMMs are one group.
//   kRowGroups (Fprop / Dgrad): group g owns output rows [off[g], off[g+1]),
//     contracts over all kblocks K-blocks, reads B rows g * b_group_rows ...
//     and B scales at g * sb_group_stride; off[num_groups] must equal
//     rows_total.
//   kTokenGroups (Wgrad): group g owns tokens [off[g], off[g+1]), padded to
//     whole 128-token K-blocks laid end to end (at most tcap tokens); every
//     group has the same b_rows x n_cols output at g * out_group_stride.
enum GroupLayout { kRowGroups = 0, kTokenGroups = 1 };

struct GemmParams {
    int layout;                   // GroupLayout
    int num_groups;
    int n_cols;                   // output columns (same for all groups)
    int n_tiles;                  // column tiles of BN per group
    int kblocks;                  // kRowGroups: 128-element K-blocks of the contraction
    int b_group_rows;             // kRowGroups: B rows per group
    // kRowGroups: 1 when B is stored [contraction x width] with the width
    // (output column) index contiguous, e.g. Fprop's W [K x N] as the
    // 128x128 cast wrote it; the tile then reaches the tensor core as an
    // MN-major operand (two 128-column TMA boxes per K-block) and B row
    // g * b_group_rows + k holds contraction index k of group g. 0: B is
    // stored [width x contraction] (K-major).
    int b_mn;
    int out_rows;                 // kTokenGroups: output rows per group (the A rows)
    int rows_total;               // kRowGroups: off[num_groups] must equal this
    int tcap;                     // kTokenGroups: padded tokens available in the operands
    int64_t sb_group_stride;      // kRowGroups: floats between consecutive groups' B scales
    int64_t out_group_stride;     // kTokenGroups: elements between consecutive groups' outputs
    const int32_t* off_dev;       // device offsets (num_groups + 1), or null
    int32_t off[kMaxGroups + 1];  // host offsets (used when off_dev is null)
    const float* sa;              // A scale of (row, kb): sa[(sa_kb0 + kb) * sa_ld + row]
    int64_t sa_ld;
    int32_t sa_rows;              // rows that may be read from sa
    const float* sb;              // B scale: see GemmKind
    int64_t sb_kstride, sb_cstride;
    void* out;
    int64_t out_ld;
    int accumulate;
    // 1: the output tensor map passed with the launch is valid, and whole
    // 32-row pieces of the BF16 output are stored from shared memory with
    // TMA (Fprop / Dgrad without split-K)
    int tma_store;
    int splits;                   // split-K ranges per tile (1: none)
    int kb_per_split;             // K-blocks per range
    float* ws;                    // split-K: fp32 range sums, [splits][tiles][32][256] float4, else null
    int64_t ws_split_stride;      // floats between consecutive ranges' slices (splitk_tile_floats)
    uint64_t wait_limit_ns;
    unsigned int* status;
    // Test hook (fp8bs_selftest_gemm_timeout only): the epilogue never hands
    // a tensor-memory buffer back, so the MMA thread's wait for the third
    // K-block's buffer can only give up, which exercises the bounded waits,
    // the abort and the drain of a real GEMM without a fault.
    int hold_release;
    // Stream-K (Fprop / Dgrad, one group, no split-K): sk_len > 0 gives CTA c
    // the K-blocks [c sk_len, (c + 1) sk_len) of the tile-major (tile,
    // K-block) sequence, so every CTA does the same work whatever the tile
    // count. A tile cut between CTAs c and c + 1 (sk_len >= the tile's
    // K-blocks, so at most one cut per tile) is finished by c, which adds the
    // fp32 sum that c + 1 left in its workspace slot.
    int sk_len;
    int sk_units;                 // units per CTA (its most segments: stream-K loops run gridDim.x x sk_units)
    float* sk_ws;                 // [grid][32][256] float4: one partial tile per CTA
    unsigned int* sk_flags;       // [grid]: 1 while a slot holds a partial not yet added
};

enum class GemmKind {
    kBlockScaleBf16,   // B scale per (K-block, 128-column block), BF16 output (Fprop, Dgrad)
    kVectorScaleF32,   // B scale per (K-block, column), FP32 output (Wgrad)
};

// map_out: the BF16 output [rows x out_ld] (box 64 x 32, 128-byte swizzle),
// used when p.tma_store is set.
// max_units: an upper bound on the work units (tiles x splits), which
// sizes the persistent grid when the offsets live on the device.
cudaError_t launch_gemm(GemmKind kind, const CUtensorMap& map_a, const CUtensorMap& map_b,
                        const CUtensorMap& map_out, const GemmParams& p, int64_t max_units, int num_sms,
                        cudaStream_t stream);

// GEMM tile shape and pipeline depth (exported for host-side planning).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 128;

// Split-K workspace: per range, one slot of 128 x 256 fp32 per output tile
// (tile-major, the tile's values as [32][256] float4 in the GEMM epilogue's
// thread order); this many floats per range for an output of rows x cols.
constexpr int64_t splitk_tile_floats(int64_t rows, int64_t cols)
{
    return ((rows + kBM - 1) / kBM) * ((cols + kBN - 1) / kBN) * static_cast<int64_t>(kBM) * kBN;
}

// out [rows x cols] BF16 = the sum over `splits` ranges of the workspace
// slots, in range order, rounded once.
cudaError_t launch_splitk_reduce(const float* ws, int splits, int64_t rows, int64_t cols, uint16_t* out, int num_sms,
                                 cudaStream_t stream);

// MXFP8 (mx.cu): 1x32 quantizer writing scale atoms, and the block-scaled GEMM.
cudaError_t launch_mx_quant_1x32(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* atoms,
                                 int num_sms, cudaStream_t stream);
cudaError_t launch_mx_quant_1x32_T(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* qT, uint8_t* atoms,
                                   cudaStream_t stream);
// Group layouts of the MX GEMM.
//   kMxDense:       one problem; A atoms [ceil(M/128)][K/128], B atoms [N/128][K/128].
//   kMxRowGroups:   Fprop / Dgrad of experts: group g owns A rows
//                   [off[g], off[g+1]) and B rows [g * b_group_rows, + b_group_rows);
//                   A's atoms are laid out by the groups' 128-row tiles in order
//                   (tile t of all groups: atoms [t][K/128]), B's per group
//                   [g][b_group_rows/128][K/128]; output rows = A rows.
//   kMxTokenGroups: Wgrad of experts: A [out_rows x Tpad], B [N x Tpad] over
//                   padded tokens (each group's tokens padded to 128, laid end
//                   to end); group g contracts over its own K-blocks; its
//                   output [out_rows x N] sits at rows g * out_rows of the output.
enum MxLayout { kMxDense = 0, kMxRowGroups = 1, kMxTokenGroups = 2 };

struct MxGroups {
    int layout;                     // MxLayout
    int num_groups;
    const int32_t* off_dev;         // device offsets (num_groups + 1), or null
    int32_t off[kMaxGroups + 1];    // host offsets (used when off_dev is null)
    int rows_total;                 // grouped: off[num_groups] must equal this
    int b_group_rows;               // row groups: B rows per group
    int kb_atoms_a, kb_atoms_b;     // atoms per 128-row block along K, of A and of B
    int out_rows;                   // token groups: output rows per group
    int kb_cap;                     // token groups: padded K-blocks the operands hold
    // dense and row groups: 1 when B's codes are stored [K x N] per group
    // (N contiguous; group g's rows start at g * K) and reach the tensor core
    // MN-major; its scale atoms keep the [N x K] layout
    int b_mn;
};

// out (BF16) or out_f32 (FP32, when not null) [M x N] (M = the output rows:
// all tokens for row groups, groups x out_rows for token groups); map_out
// (nullable): the output as boxes of 32 rows x 64 bytes with the 64-byte
// swizzle, through which whole 32-row boxes are stored with TMA. K: the
// contraction of one group (kMxDense, kMxRowGroups); unused for token groups.
// grp: the group layout; max_tiles: an upper bound on the output tiles, which
// sizes the persistent grid.
cudaError_t launch_mx_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap* map_out,
                           const uint8_t* sfa, const uint8_t* sfb, int M, int N, int K, uint16_t* out,
                           float* out_f32, const MxGroups& grp, int64_t max_tiles, uint64_t wait_limit_ns,
                           unsigned int* status, int num_sms, cudaStream_t stream);

// Groups of a grouped packing: device offsets, or host offsets.
struct PackGroups {
    int num_groups;
    int rows_total;                 // off[num_groups] must equal this
    const int32_t* off_dev;         // device offsets (num_groups + 1), or null
    int32_t off[kMaxGroups + 1];    // host offsets (used when off_dev is null)
};

// The exponent bytes of row-wise (1x128) power-of-two scales of grouped rows
// [rows x K] into the MX scale atoms in the groups' tile layout (the A
// operand of a grouped MX Fprop / Dgrad): scale of (row r, K-block b) at
// scales[r + b * kb_stride]; atoms of tile t at [t][K/128]; tiles_cap: the
// tile count the atom buffer holds.
cudaError_t launch_pack_ue8m0_grouped(const float* scales, int64_t K, int64_t kb_stride, const PackGroups& pg,
                                      int64_t tiles_cap, uint8_t* atoms, unsigned int* status, int num_sms,
                                      cudaStream_t stream);

// Exponent bytes of power-of-two block scales into the MX scale atoms of an
// operand [rows x K] (mx.cu); non-representable scales record
// FP8BS_ERR_DEVICE in *status and write 255.
cudaError_t launch_pack_ue8m0(const float* scales, int64_t rows, int64_t K, int row_block, int64_t row_stride,
                              int64_t kb_stride, uint8_t* atoms, unsigned int* status, int num_sms,
                              cudaStream_t stream);

cudaError_t launch_selftest_wait(unsigned int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace fp8bs
