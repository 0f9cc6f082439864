/*
 * fp8bs.h -- C ABI of the GB300 (sm_103a) fine-grained FP8 linear-layer library.
 *
 * The library implements the data path of a linear layer under the
 * DeepSeek-V3 FP8 training recipe:
 *   - dynamic absmax quantization to E4M3 with fp32 scales, in 1x128 tiles
 *     (activations, gradients), 128x128 tiles (weights) and a transposed 128x1
 *     re-tiling of saved operands for the weight gradient;
 *   - the three E4M3 GEMMs of a linear (Fprop Y = X W, Dgrad dX = dY W^T,
 *     Wgrad dW = dY^T X), each promoting its per-128-K partial sums to fp32
 *     scaled by s_a * s_b, with BF16 (Y, dX) or FP32 (dW) output;
 *   - a grouped variant of the GEMMs for MoE experts.
 * Sources for the definitions:
 *   [P1] "scratch: the backward pass, unrolled" (deepseek-v3.ezyang.com),
 *        section "What is asserted, and from where", bullets 1-2 and
 *        "Where casts are drawn".
 *   [P2] "FP8 动态量化里的 partial sum 漂移" (foosynaptic DeepSeek tech notes),
 *        section 3 (fine-grained scale and FP32 promotion table) and
 *        section 5 (promotion every N_c = 128).
 *   [P3] TransformerEngine PR #3573, "Changes" (E4M3 bound 448) and the
 *        all-zero-gradient test patterns.
 *   [P4] prime-rl PR #4073, quantization-conventions table, row
 *        "Negative zero" (E4M3 -0 is 0x80, kept apart from +0 = 0x00).
 *
 * Common conventions
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference after the call returns. Its own device memory is a
 *     status word, the fixed array of fp8_block_gemm_splitk_noalloc, and the
 *     stream-K workspaces of Fprop / Dgrad (one 128 x 256 fp32 tile and one
 *     flag per SM, about 20 MB on a GB300): one per stream that runs a
 *     stream-K GEMM eagerly (up to eight per device, each allocated by the
 *     first such GEMM on its stream; beyond eight, GEMMs on further streams
 *     run without stream-K), and one shared by every stream-K GEMM captured
 *     into a CUDA graph, allocated with the device's set-up by the first call
 *     on the device. Make that first call, and the first Fprop / Dgrad on a
 *     stream, before any stream capture begins. Graphs holding stream-K
 *     GEMMs share their workspace: do not replay two of them concurrently.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream). The returned status covers argument
 *     validation and launch errors only. Errors detected on the device (a
 *     bounded pipeline wait that gave up) are recorded in a per-device status
 *     word read by fp8bs_device_status(), fp8bs_last_device_status(stream) or
 *     fp8bs_copy_device_status().
 *   - Matrices are row-major. "ld" arguments are row strides in elements.
 *   - BF16 data is passed as `const void*` (IEEE bfloat16 bit patterns), E4M3
 *     payloads as `uint8_t*` (OCP E4M3, "fn" variant: max 448, no infinities).
 *   - Quantization: for a tile with values v (fp32 from BF16 or from a
 *     dequantized E4M3 stash): amax = max |v|; s = amax / 448 (IEEE fp32
 *     division) or s = 1 when amax = 0; q = E4M3_RN_satfinite(fp32(v / s)),
 *     ties to even, saturating at +-448, a zero result keeps the sign of v.
 *     Results are bit-identical to the CPU oracle of this repository.
 *   - Pointers must be 16-byte aligned (FP8BS_ERR_ALIGN otherwise).
 *   - Inputs must be finite; NaN/Inf inputs give unspecified payloads.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8BS_API __attribute__((visibility("default")))
#else
#define FP8BS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_ARG = 1,          /* null pointer, negative size or bad enum value */
    FP8BS_ERR_ALIGN = 2,        /* pointer not 16-byte aligned or stride not a multiple of 16 bytes */
    FP8BS_ERR_SHAPE = 3,        /* size outside the documented constraints */
    FP8BS_ERR_LAUNCH = 4,       /* CUDA reported an error launching the kernel */
    FP8BS_ERR_TIMEOUT = 5,      /* device: a bounded pipeline wait gave up (kernel returned early) */
    FP8BS_ERR_UNSUPPORTED = 6,  /* device is not sm_103a-capable, or a driver entry point is missing */
    FP8BS_ERR_DEVICE = 7        /* device: a kernel's own consistency check failed */
} fp8bs_status;

typedef enum {
    FP8BS_SRC_BF16 = 0,         /* requant source is BF16 ("mode B") */
    FP8BS_SRC_E4M3 = 1          /* requant source is an E4M3 stash with 1x128 scales ("mode Q") */
} fp8bs_src_mode;

typedef enum {
    FP8BS_OP_FPROP = 0,
    FP8BS_OP_DGRAD = 1,
    FP8BS_OP_WGRAD = 2,
    FP8BS_OP_FPROP_WKN = 3      /* Fprop with W's codes as stored, [K x N] (see fp8_block_gemm_fprop_wkn) */
} fp8bs_op;

/* Largest number of groups (experts) accepted by the grouped entry points. */
#define FP8BS_MAX_GROUPS 256

/* ------------------------------------------------------------------------ */
/* Helpers (host only, no device work)                                       */
/* ------------------------------------------------------------------------ */

/* Human-readable name of a status code (static string). */
FP8BS_API const char* fp8bs_status_str(fp8bs_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
FP8BS_API int fp8bs_version(void);

/* Row stride of a 1x128 scale array: `rows` rounded up to a multiple of 4
 * (so that every tile row of scales starts on a 16-byte boundary). */
FP8BS_API int64_t fp8bs_scale_ld(int64_t rows);

/* Token count of the transposed 128x1 output: each group's token count
 * rounded up to a multiple of 128, summed. With group_offsets_host == NULL
 * (or groups == 0) the whole `rows` is one group. Returns -1 for invalid
 * offsets. */
FP8BS_API int64_t fp8bs_padded_tokens(int64_t rows, const int32_t* group_offsets_host, int32_t groups);

/* The largest value fp8bs_padded_tokens can take for `groups` groups holding
 * `rows` tokens in total, whatever the split: with k = min(groups, rows)
 * (the most groups that can be non-empty), 128 * floor((rows + 127 k) / 128),
 * and rows rounded up to 128 when k <= 1. The token length of the transposed
 * outputs of the _dev casts and of grouped Wgrad operands with device offsets.
 * Returns -1 for rows < 0 or groups outside [0, FP8BS_MAX_GROUPS]. */
FP8BS_API int64_t fp8bs_padded_tokens_max(int64_t rows, int32_t groups);

/* ------------------------------------------------------------------------ */
/* S1. 1x128 activation / gradient quantizer                                 */
/* [P1] bullet 1 (1x128 activation tiles) and bullet 2 (dY is quantized to    */
/* E4M3 before Dgrad and Wgrad); [P2] section 3 row (a).                      */
/* ------------------------------------------------------------------------ */
/* x       : BF16 [rows x cols], row stride ldx (ldx >= cols, ldx % 8 == 0).
 * q       : E4M3 [rows x cols], dense (row stride cols).
 * scales  : fp32 [ceil(cols/128) x fp8bs_scale_ld(rows)], tile-major: the
 *           scale of row r, column tile t is scales[t * fp8bs_scale_ld(rows) + r].
 *           The padding entries (r >= rows) are not written.
 * Tiles cover columns [128 t, min(128 t + 128, cols)); a ragged last tile
 * takes the absmax over its valid columns.
 * Constraints: rows >= 0, cols > 0, cols % 16 == 0 (FP8BS_ERR_SHAPE). */
FP8BS_API fp8bs_status fp8_quant_1x128(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                             uint8_t* q, float* scales, void* stream);

/* ------------------------------------------------------------------------ */
/* S2. 128x128 weight quantizer                                              */
/* [P1] bullet 1 (128x128 weight tiles); [P2] section 3 row (a).              */
/* ------------------------------------------------------------------------ */
/* w       : BF16 [batch x rows x cols]; matrix b starts at w + b * rows * ldw,
 *           row stride ldw (ldw >= cols, ldw % 8 == 0). For a layer weight
 *           W [K x N] (Y = X W), rows = K and cols = N; batch > 1 stacks the
 *           weights of several experts.
 * q       : E4M3 [batch x rows x cols], dense. This orientation is the Dgrad operand.
 * qT      : optional (may be NULL) E4M3 [batch x cols x rows], dense: the byte
 *           transpose of each matrix of q. This K-contiguous orientation is the
 *           Fprop operand. Because the tiles are square, the transpose needs no
 *           requantization.
 * scales  : fp32 [batch x ceil(rows/128) x ceil(cols/128)], row-major, shared by
 *           q and qT.
 * Constraints: batch >= 1, rows > 0, cols > 0, rows % 16 == 0, cols % 16 == 0. */
FP8BS_API fp8bs_status fp8_quant_128x128(const void* w, int64_t batch, int64_t rows, int64_t cols,
                               int64_t ldw, uint8_t* q, uint8_t* qT, float* scales,
                               void* stream);

/* ------------------------------------------------------------------------ */
/* S3. 128x1 transposed requantization for the weight gradient               */
/* [P1] bullet 2 (Wgrad takes its transposed operands re-tiled 128x1 from    */
/* what the forward saved) and "Where casts are drawn" (a small requant box   */
/* on the stash edge; backward vector kernels emit dY in both orientations).  */
/* ------------------------------------------------------------------------ */
/* Re-tiles a token-major tensor [rows x cols] (rows = tokens) into 128-token
 * x 1-channel tiles and writes the payload transposed (tokens contiguous).
 * src_mode FP8BS_SRC_BF16: src is BF16 [rows x cols], dense, src_scales NULL.
 * src_mode FP8BS_SRC_E4M3: src is the E4M3 stash [rows x cols] written by
 *           fp8_quant_1x128, src_scales its 1x128 scales (layout as above);
 *           each element is decoded as fp32(dec(q) * s) before requantizing.
 * group_offsets_host: optional HOST array of groups + 1 int32 row offsets
 *           (offsets[0] = 0, non-decreasing, offsets[groups] = rows). Each
 *           group's token tiles start at its own first row; a group's last
 *           tile may be ragged. NULL (or groups == 0) means one group.
 * qT      : E4M3 [cols x Mpad], Mpad = fp8bs_padded_tokens(rows, offsets, groups).
 *           Group g occupies padded columns [P_g, P_g + 128 * ceil(T_g / 128))
 *           with P_g the sum of the earlier groups' padded counts; the padding
 *           bytes are written as 0x00.
 * scalesT : fp32 [Mpad/128 x cols]; row j holds the scales of padded token tile j.
 * Constraints: rows >= 0, cols > 0, cols % 16 == 0, groups <= FP8BS_MAX_GROUPS. */
FP8BS_API fp8bs_status fp8_requant_128x1_T(int src_mode, const void* src, const float* src_scales,
                                 int64_t rows, int64_t cols,
                                 const int32_t* group_offsets_host, int32_t groups,
                                 uint8_t* qT, float* scalesT, void* stream);

/* Dual-orientation cast of one BF16 tensor in a single read: the    */
/* 1x128 cast of fp8_quant_1x128 and the 128x1 transposed cast of            */
/* fp8_requant_128x1_T (FP8BS_SRC_BF16), both outputs byte-identical to the  */
/* two separate calls. [P1] "What is asserted, and from where": the output   */
/* gradient is quantized once in both tile orientations (row-wise for Dgrad, */
/* column-wise for Wgrad); [P3] "Performance" measures the separate casts as */
/* an extra read of the gradient, which this call removes.                   */
/* x        : BF16 [rows x cols], dense (row stride = cols), cols % 16 == 0.  */
/* group_offsets_host, groups : as for fp8_requant_128x1_T (NULL/0 = dense);  */
/*            the 1x128 outputs do not depend on the grouping.               */
/* q, scales: as fp8_quant_1x128 (E4M3 [rows x cols]; fp32 tile-major        */
/*            [cols/128 x fp8bs_scale_ld(rows)]).                             */
/* qT, scalesT : as fp8_requant_128x1_T.                                      */
/* Errors as for those two calls.                                             */
FP8BS_API fp8bs_status fp8_quant_dual(const void* x, int64_t rows, int64_t cols,
                                      const int32_t* group_offsets_host, int32_t groups,
                                      uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                      void* stream);

/* Scale rule options for the four quantizers above. The pages name  */
/* the conventions without fixing every detail ([P4] conventions table, rows */
/* "Weight floors", "Two-stage weights", "Activation floors", "Compact       */
/* formats"); the reading implemented here:                                   */
/*   a = max(amax, amax_floor);                                               */
/*   s = a / 448 in fp32, or 1 when a == 0 and no scale floor is set;         */
/*   s = max(s, scale_floor);                                                 */
/*   FP8BS_SCALE_UE8M0: s = the smallest power of two >= s (an exponent byte; */
/*   amax / s stays <= 448, and above 224 for a non-floored tile).            */
/* Scales are still stored as fp32 values (the Hopper container); GEMMs take  */
/* them unchanged. The default (NULL, or rule FP8BS_SCALE_FP32 with zero      */
/* floors) is the plain rule of the calls above.                              */
enum { FP8BS_SCALE_FP32 = 0, FP8BS_SCALE_UE8M0 = 1 };
typedef struct {
    int32_t rule;          /* FP8BS_SCALE_FP32 or FP8BS_SCALE_UE8M0 */
    float amax_floor;      /* >= 0 (0: none) */
    float scale_floor;     /* >= 0 (0: none) */
} fp8bs_scale_opts;

/* The calls above with a scale rule; opts == NULL is the default rule.       */
/* Invalid options (unknown rule, negative or non-finite floors) return       */
/* FP8BS_ERR_ARG.                                                             */
FP8BS_API fp8bs_status fp8_quant_1x128_opts(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                            uint8_t* q, float* scales, const fp8bs_scale_opts* opts,
                                            void* stream);
FP8BS_API fp8bs_status fp8_quant_128x128_opts(const void* w, int64_t batch, int64_t rows, int64_t cols,
                                              int64_t ldw, uint8_t* q, uint8_t* qT, float* scales,
                                              const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_requant_128x1_T_opts(int src_mode, const void* src, const float* src_scales,
                                                int64_t rows, int64_t cols,
                                                const int32_t* group_offsets_host, int32_t groups,
                                                uint8_t* qT, float* scalesT,
                                                const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_opts(const void* x, int64_t rows, int64_t cols,
                                           const int32_t* group_offsets_host, int32_t groups,
                                           uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                           const fp8bs_scale_opts* opts, void* stream);

/* The forward activation cast and its Wgrad requant in one pass: the 1x128  */
/* cast of fp8_quant_1x128 and the 128x1 transposed requant of that E4M3     */
/* result (fp8_requant_128x1_T with FP8BS_SRC_E4M3 on q, scales), both       */
/* outputs byte-identical to those two calls in sequence. [P1] bullet 2 and  */
/* "Where casts are drawn": Wgrad's transposed activation operand is a       */
/* requant of the E4M3 stash the forward saved; this call produces it while  */
/* the forward cast still holds the tile, saving a second read of the stash  */
/* and a launch, at the cost of keeping qT from the forward on.              */
/* Arguments, layouts, constraints and errors as for fp8_quant_dual.         */
FP8BS_API fp8bs_status fp8_quant_dual_stash(const void* x, int64_t rows, int64_t cols,
                                            const int32_t* group_offsets_host, int32_t groups,
                                            uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                            void* stream);
/* The same with a scale rule (see fp8bs_scale_opts); both casts use it.      */
FP8BS_API fp8bs_status fp8_quant_dual_stash_opts(const void* x, int64_t rows, int64_t cols,
                                                 const int32_t* group_offsets_host, int32_t groups,
                                                 uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                                 const fp8bs_scale_opts* opts, void* stream);

/* The transposed cast, the dual cast and the fused forward cast (above) with
 * DEVICE group offsets: offsets_dev (4-byte aligned, groups + 1 entries,
 * 1 <= groups <= FP8BS_MAX_GROUPS) is read by the kernel when it runs, so it
 * may come from earlier device work on the same stream and the call may be
 * captured in a CUDA graph. The outputs are laid out as with host offsets
 * except that qT is [cols x Mcap] and scalesT [Mcap/128 x cols] with
 * Mcap = fp8bs_padded_tokens_max(rows, groups): group g still starts at the
 * padded column P_g (the sum of the earlier groups' padded counts); columns
 * past the groups' padded total are not written. Invalid device offsets
 * (offsets[0] != 0, a decrease, a total other than rows) record
 * FP8BS_ERR_DEVICE in the device status word and nothing is written. opts as
 * for the _opts calls (NULL: the plain rule). */
FP8BS_API fp8bs_status fp8_requant_128x1_T_dev(int src_mode, const void* src, const float* src_scales,
                                               int64_t rows, int64_t cols, const int32_t* offsets_dev,
                                               int32_t groups, uint8_t* qT, float* scalesT,
                                               const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_dev(const void* x, int64_t rows, int64_t cols, const int32_t* offsets_dev,
                                          int32_t groups, uint8_t* q, float* scales, uint8_t* qT,
                                          float* scalesT, const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_stash_dev(const void* x, int64_t rows, int64_t cols,
                                                const int32_t* offsets_dev, int32_t groups, uint8_t* q,
                                                float* scales, uint8_t* qT, float* scalesT,
                                                const fp8bs_scale_opts* opts, void* stream);


/* Stochastic rounding. The 1x128 and 128x128 casts above with the   */
/* E4M3 rounding step made stochastic under a stateless (seed, salt,         */
/* element) contract ([P4] "SR agreement": a stateless seed / salt / counter */
/* scheme with a lower / upper-magnitude rule; [P4] "Remaining differences"  */
/* and the PR text name a Philox helper). The pages do not print the         */
/* contract's layout; this library's reading:                               */
/*   word(idx) = word idx % 4 of Philox4x32-10 (Salmon et al., SC 2011) with */
/*               key (seed & 0xffffffff, seed >> 32) and counter            */
/*               (idx / 4 low 32 bits, idx / 4 high 32 bits, salt, 0),      */
/*               idx = the element's linear index in the logical tensor     */
/*               (row * cols + col; for batched weights,                    */
/*               b * rows * cols + row * cols + col);                       */
/*   x = fp32(v / s) as in the round-to-nearest cast; with L <= |x| < U the  */
/*   neighbouring E4M3 magnitudes, F = floor(2^20 (|x| - L) / (U - L));      */
/*   the code is U if F > (word >> 12), else L; |x| >= 448 gives 448; the    */
/*   sign (and a signed zero) is x's.                                         */
/* Results depend only on (input, seed, salt), not on the launch or device.  */
/* Scales are computed exactly as in the round-to-nearest cast (opts as      */
/* above, NULL = default rule); the transposed qT of the 128x128 cast is the */
/* transpose of the stochastically rounded q.                                */
FP8BS_API fp8bs_status fp8_quant_1x128_sr(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                          uint8_t* q, float* scales, uint64_t seed, uint32_t salt,
                                          const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_128x128_sr(const void* w, int64_t batch, int64_t rows, int64_t cols,
                                            int64_t ldw, uint8_t* q, uint8_t* qT, float* scales,
                                            uint64_t seed, uint32_t salt,
                                            const fp8bs_scale_opts* opts, void* stream);

/* The transposed casts with stochastic rounding, under the same contract:  */
/* element (r, c) of the source tensor [rows x cols] takes word(r * cols + c)*/
/* (the padding tokens of qT stay 0x00).                                     */
/* fp8_requant_128x1_T_sr: fp8_requant_128x1_T with (seed, salt).            */
/* fp8_quant_dual_sr / fp8_quant_dual_stash_sr: the 1x128 part is            */
/* fp8_quant_1x128_sr with (seed, salt); the transposed part uses            */
/* (seed, salt + 1), from the BF16 values (dual) or from the stochastically  */
/* rounded 1x128 result (stash), so each output is byte-identical to the     */
/* corresponding separate calls. Arguments otherwise as the calls without    */
/* _sr (opts: scale rule, NULL = default).                                    */
FP8BS_API fp8bs_status fp8_requant_128x1_T_sr(int src_mode, const void* src, const float* src_scales,
                                              int64_t rows, int64_t cols,
                                              const int32_t* group_offsets_host, int32_t groups,
                                              uint8_t* qT, float* scalesT, uint64_t seed, uint32_t salt,
                                              const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_sr(const void* x, int64_t rows, int64_t cols,
                                         const int32_t* group_offsets_host, int32_t groups,
                                         uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                         uint64_t seed, uint32_t salt, const fp8bs_scale_opts* opts,
                                         void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_stash_sr(const void* x, int64_t rows, int64_t cols,
                                               const int32_t* group_offsets_host, int32_t groups,
                                               uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                               uint64_t seed, uint32_t salt, const fp8bs_scale_opts* opts,
                                               void* stream);

/* ------------------------------------------------------------------------ */
/* S4-S6. Block-scaled E4M3 GEMMs with per-128-K fp32 promotion              */
/* [P1] bullet 1 (all three GEMMs E4M3; BF16 activations and input grads,     */
/* FP32 weight grads); [P2] section 3 rows (a)-(b) and section 5: the tensor  */
/* core accumulates 128 elements of K, the partial is scaled by s_a * s_b and */
/* added to an fp32 accumulator, and the next 128 start from zero.            */
/* The tensor-core partial over one 128-K block and the fp32 accumulation     */
/* order are implementation details; results agree with the oracle within     */
/* |d| <= 2e-3 * sum_k |a_k b_k| + 1e-6 (dequantized operands), plus one BF16 */
/* rounding step for BF16 outputs.                                            */
/* Fprop and Dgrad run stream-K when their output tiles would fill the last   */
/* round of the persistent grid (one CTA per SM) below 90%: each CTA takes    */
/* the same number of K-blocks, and a tile cut between two CTAs is summed in  */
/* two fp32 parts, through a workspace private to the call's stream. Results */
/* are deterministic for a given GPU (they depend on its SM count only       */
/* through that summation order). A GEMM that gave up                        */
/* (FP8BS_ERR_TIMEOUT) may leave stream-K state behind: the status reset of   */
/* fp8bs_device_status / fp8bs_last_device_status / fp8bs_copy_device_status  */
/* clears it, and must come before the next GEMM on that device.             */
/* ------------------------------------------------------------------------ */

/* Fprop: Y[i,j] = sum_b s_x[i,b] * s_w[b, j/128] * P_b[i,j].
 * xq  : E4M3 [M x K] (fp8_quant_1x128 of X), sx its scales.
 * wqT : E4M3 [N x K], the qT output of fp8_quant_128x128 on W [K x N].
 * sw  : fp32 [K/128 x N/128] (the scales of that call).
 * y   : BF16 [M x N], dense, overwritten.
 * Constraints: M >= 0, K > 0, N > 0, K % 128 == 0, N % 128 == 0. */
FP8BS_API fp8bs_status fp8_block_gemm_fprop(const uint8_t* xq, const float* sx,
                                  const uint8_t* wqT, const float* sw,
                                  int64_t M, int64_t N, int64_t K, void* y, void* stream);

/* Fprop on W's codes in their own orientation: the same result as
 * fp8_block_gemm_fprop (bit for bit: the tensor core sees the same operand
 * values), with B read from the q output of fp8_quant_128x128 on W [K x N]
 * instead of its byte transpose. The tensor core takes this operand
 * MN-major (N contiguous in shared memory), so a weight cast feeding only
 * Fprop and Dgrad can skip qT (NULL) and write 3 bytes per element instead
 * of 4: Fprop and Dgrad then read the same codes.
 * wq : E4M3 [K x N], the q output of fp8_quant_128x128 on W [K x N].
 * Other arguments and constraints as for fp8_block_gemm_fprop. */
FP8BS_API fp8bs_status fp8_block_gemm_fprop_wkn(const uint8_t* xq, const float* sx,
                                      const uint8_t* wq, const float* sw,
                                      int64_t M, int64_t N, int64_t K, void* y, void* stream);

/* Dgrad: dX[i,k] = sum_b s_dy[i,b] * s_w[k/128, b] * P_b[i,k], contraction
 * over the layer's N outputs.
 * dyq : E4M3 [M x N] (fp8_quant_1x128 of dY), sdy its scales.
 * wq  : E4M3 [K x N], the q output of fp8_quant_128x128 on W [K x N].
 * sw  : fp32 [K/128 x N/128].
 * dx  : BF16 [M x K], dense, overwritten.
 * Constraints: M >= 0, K % 128 == 0, N % 128 == 0, K, N > 0. */
FP8BS_API fp8bs_status fp8_block_gemm_dgrad(const uint8_t* dyq, const float* sdy,
                                  const uint8_t* wq, const float* sw,
                                  int64_t M, int64_t N, int64_t K, void* dx, void* stream);

/* Wgrad: dW[n,k] = sum_b s_dyT[b,n] * s_xT[b,k] * P_b[n,k], contraction over
 * T (padded) tokens, on the outputs of fp8_requant_128x1_T.
 * dyqT : E4M3 [N x T], sdyT fp32 [T/128 x N].
 * xqT  : E4M3 [K x T], sxT  fp32 [T/128 x K].
 * dw   : FP32 [N x K], dense. accumulate = 0 overwrites, 1 adds into dw.
 * Constraints: T >= 0, T % 128 == 0, N % 128 == 0, K % 128 == 0, N, K > 0.
 * With T == 0 the result is zero (dw is zeroed unless accumulate). */
FP8BS_API fp8bs_status fp8_block_gemm_wgrad(const uint8_t* dyqT, const float* sdyT,
                                  const uint8_t* xqT, const float* sxT,
                                  int64_t T, int64_t N, int64_t K, float* dw,
                                  int accumulate, void* stream);

/* Split-K Fprop / Dgrad, for outputs too small to occupy the GPU (few      */
/* output tiles, long contraction; e.g. 256 x 256 outputs with K = 65536).   */
/* The contraction's 128-blocks are cut into `splits` contiguous ranges (at  */
/* most one range per block). Each range is computed exactly like the unsplit */
/* GEMM ([P2] section 5: per-block partials scaled by s_a * s_b, added in     */
/* fp32); the ranges' fp32 sums are then added in range order and rounded to */
/* BF16 once. The pages' promotion recipe fixes the per-block scaling, not    */
/* the fp32 addition order, so the result differs from the unsplit call only  */
/* by fp32 rounding and stays within the tolerance above. Deterministic.      */
/*                                                                           */
/* op        : FP8BS_OP_FPROP, FP8BS_OP_FPROP_WKN or FP8BS_OP_DGRAD; a, sa, */
/*             b, sb, M, N, K, out as for fp8_block_gemm_fprop (a = xq,       */
/*             b = wqT), fp8_block_gemm_fprop_wkn (a = xq, b = wq) or         */
/*             fp8_block_gemm_dgrad (a = dyq, b = wq).                        */
/* splits    : >= 1; values above the number of 128-blocks are clamped.      */
/* workspace : caller-owned device buffer of at least                        */
/*             fp8bs_splitk_workspace_size(op, M, N, K, splits) bytes,        */
/*             16-byte aligned (may be NULL when that size is 0). Contents on */
/*             entry are ignored and undefined afterwards; it must not be     */
/*             used by anything else until the call has completed on stream.  */
/* Errors: FP8BS_ERR_ARG (bad op, splits < 1, NULL or too small workspace),   */
/* FP8BS_ERR_SHAPE / FP8BS_ERR_ALIGN as for the unsplit calls.                */
/* fp8bs_splitk_workspace_size: the ranges actually used (ceil(blocks /       */
/* ceil(blocks / splits))) x one 128 x 256 fp32 slot per 128 x 256 output     */
/* tile, in bytes; 0 when no split happens or the arguments are invalid.     */
FP8BS_API size_t fp8bs_splitk_workspace_size(int op, int64_t M, int64_t N, int64_t K, int32_t splits);

/* A split count for this device: about one range per idle SM when the       */
/* output has fewer tiles than half the SMs and the contraction has at least  */
/* 16 128-blocks, keeping at least four 128-blocks per range; 1 (no split)    */
/* otherwise (below that the extra reduction pass costs more than it saves). */
/* Uses the current device.                                                   */
FP8BS_API int32_t fp8bs_splitk_default_splits(int op, int64_t M, int64_t N, int64_t K);

FP8BS_API fp8bs_status fp8_block_gemm_splitk(int op, const uint8_t* a, const float* sa,
                                   const uint8_t* b, const float* sb,
                                   int64_t M, int64_t N, int64_t K, int32_t splits,
                                   void* out, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Split-K without a caller workspace. No counterpart in the pages          */
/* ([P1]-[P4]): it exists for callers that cannot allocate device memory     */
/* (an allocator-free runtime, a loop that must not call cudaMalloc because  */
/* it can synchronize the device, a plugin without a memory pool). Same       */
/* arguments and result as fp8_block_gemm_splitk; the range sums go to a     */
/* fixed array of FP8BS_NOALLOC_SCRATCH_BYTES compiled into the library, and */
/* the call allocates nothing.                                                */
/* - Requests needing more than FP8BS_NOALLOC_SCRATCH_BYTES                   */
/*   (fp8bs_splitk_workspace_size(op, M, N, K, splits)) return               */
/*   FP8BS_ERR_SHAPE before any work; lower `splits` or use                  */
/*   fp8_block_gemm_splitk with a workspace.                                  */
/* - The first call on each device (with that device current) does a one-    */
/*   time set-up (it looks up the array's device address; under lazy module  */
/*   loading this is also when the array is placed on the device); make that  */
/*   first call before any stream capture begins.                             */
/* - Every call must be made with the device of `stream` current             */
/*   (FP8BS_ERR_ARG otherwise), like the set-up call.                         */
/* - The array is device memory held on every device where the library's     */
/*   module is loaded, by every process that loads the library, whether or   */
/*   not it calls this entry point, until the process exits.                 */
/* - The looked-up address does not survive cudaDeviceReset; do not call this */
/*   entry point on a device after resetting it.                             */
/* - One array serves all calls on a device: calls whose executions overlap   */
/*   (different streams without ordering, several host threads) race on it    */
/*   and give undefined results. Serialize them (one stream, or events).      */
/* - Nothing in the array needs to start at zero.                             */
#define FP8BS_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

FP8BS_API fp8bs_status fp8_block_gemm_splitk_noalloc(int op, const uint8_t* a, const float* sa,
                                           const uint8_t* b, const float* sb,
                                           int64_t M, int64_t N, int64_t K, int32_t splits,
                                           void* out, void* stream);

/* MXFP8, the format TransformerEngine's pages benchmark on B300    */
/* ([P3] "Changes" and "Performance": MXFP8 operands for dgrad): OCP MX v1.0 */
/* blocks of 32 elements along K with one 8-bit exponent scale              */
/* X = 2^(E - 127) each, E4M3 elements, and the block scaling applied by the */
/* tensor core. Scale choice (a reading; the pages do not print it): X = the */
/* smallest power of two >= fp32(amax / 448), X = 1 for an all-zero block;   */
/* q = E4M3_RN(v / X), an exact division.                                     */
/*                                                                           */
/* Scale atoms: for R rows (padded up to a multiple of 128) and K columns    */
/* (K % 128 == 0), atom (r/128, k/128) is 512 contiguous bytes ordered       */
/* [R/128][K/128]; the byte of row m = r % 128 = m0 + 32 m1 (m0 < 32) and    */
/* 32-block j = (k/32) % 4 is at 16 m0 + 4 m1 + j. Padding rows hold 127.    */
FP8BS_API int64_t fp8bs_mx_scale_bytes(int64_t rows, int64_t cols);

/* x: BF16 [rows x cols] dense, cols % 128 == 0. q: E4M3 [rows x cols].      */
/* scale_atoms: fp8bs_mx_scale_bytes(rows, cols) bytes, 16-byte aligned.     */
FP8BS_API fp8bs_status fp8_mx_quant_1x32(const void* x, int64_t rows, int64_t cols, uint8_t* q,
                                         uint8_t* scale_atoms, void* stream);

/* out[i, j] = sum_k A[i, k] B[j, k] (dequantized by the block scales), fp32 */
/* accumulation over all of K, BF16 output [M x N]. A: [M x K] with its      */
/* atoms (fp8_mx_quant_1x32 of the activations), B: [N x K] with its atoms   */
/* (fp8_mx_quant_1x32 of the other operand with K contiguous, e.g. W^T for   */
/* Fprop). K % 128 == 0, N % 256 == 0. No per-128-K promotion: this is the   */
/* MX recipe, not the one above.                                              */
FP8BS_API fp8bs_status fp8_mx_gemm(const uint8_t* a, const uint8_t* a_scale_atoms,
                                   const uint8_t* b, const uint8_t* b_scale_atoms,
                                   int64_t M, int64_t N, int64_t K, void* out, void* stream);

/* The same GEMM (BF16 output) with B's codes [K x N], N contiguous (W as    */
/* the 128x128 cast stores it, the q output of fp8_quant_128x128_packed),    */
/* read MN-major by the tensor core; b_scale_atoms keep the [N x K] layout   */
/* (atoms_wT of that cast). Equal to fp8_mx_gemm on the byte transpose.      */
FP8BS_API fp8bs_status fp8_mx_gemm_wkn(const uint8_t* a, const uint8_t* a_scale_atoms,
                                       const uint8_t* b, const uint8_t* b_scale_atoms,
                                       int64_t M, int64_t N, int64_t K, void* out, void* stream);

/* The same GEMM with FP32 output [M x N] (the Wgrad form: dW = dY^T X with   */
/* A = the transposed cast of dY and B = the transposed cast of X).          */
FP8BS_API fp8bs_status fp8_mx_gemm_f32(const uint8_t* a, const uint8_t* a_scale_atoms,
                                       const uint8_t* b, const uint8_t* b_scale_atoms,
                                       int64_t M, int64_t N, int64_t K, float* out, void* stream);

/* For experts: the MX GEMMs above applied to each group     */
/* (expert) g, with the group offsets of fp8_block_gemm_grouped (exactly one */
/* of offsets_dev / offsets_host; rows = the total token rows). The MoE form */
/* is the grouped path of TransformerEngine PR #3573 ("Changes": grouped     */
/* predicates and per-group paths; "Performance": MXFP8 at the DeepSeek-V3   */
/* expert shapes).                                                           */
/* op = FP8BS_OP_FPROP: a = Xq [rows x K]; b = stacked W^T codes            */
/*   [groups x N x K]; out = Y BF16 [rows x N].                              */
/* op = FP8BS_OP_FPROP_WKN: as FP8BS_OP_FPROP with b = stacked W codes       */
/*   [groups x K x N] (read MN-major, as in fp8_mx_gemm_wkn); b_scale_atoms  */
/*   as for FP8BS_OP_FPROP.                                                  */
/* op = FP8BS_OP_DGRAD (contraction N, output width K): a = dYq [rows x N];  */
/*   b = stacked W codes [groups x K x N]; out = dX BF16 [rows x K].         */
/*   Fprop / Dgrad a_scale_atoms: the atoms of A in the groups' tile layout: */
/*   group g's rows [offsets[g], offsets[g+1]) form ceil(n_g / 128) tiles of */
/*   128 rows, numbered over the groups in order (tile t = tiles of earlier  */
/*   groups + row / 128); tile t's atoms are [t][contraction/128][512]       */
/*   (fp8_pack_ue8m0_grouped writes them); rows of a group's last tile past  */
/*   its end are ignored. fp8bs_mx_scale_bytes(Tpad, contraction) bytes with */
/*   Tpad = fp8bs_padded_tokens(rows, offsets_host, groups), or with device  */
/*   offsets fp8bs_padded_tokens_max(rows, groups). b_scale_atoms: per group */
/*   fp8bs_mx_scale_bytes(width, contraction) bytes, laid end to end.        */
/* op = FP8BS_OP_WGRAD: a = dY^T codes [N x Tpad], b = X^T codes [K x Tpad]  */
/*   over the padded token layout of the grouped transposed casts (Tpad as   */
/*   above), with their atoms (fp8bs_mx_scale_bytes(N, Tpad) and             */
/*   (K, Tpad) bytes); group g contracts over its own 128-token blocks;      */
/*   out = dW FP32 [groups x N x K] (an empty group's dW is zero). With      */
/*   device offsets the transposed casts write only the actual padded        */
/*   tokens: give the scales past them a power of two (e.g. 1) before they   */
/*   are packed with fp8_pack_ue8m0, or the packing records FP8BS_ERR_DEVICE. */
/* Constraints: 1 <= groups <= FP8BS_MAX_GROUPS; the contraction a multiple  */
/* of 128, the output width (N for Fprop, K for Dgrad and Wgrad) a multiple  */
/* of 256; 16-byte aligned buffers. Invalid device offsets record            */
/* FP8BS_ERR_DEVICE and the kernel writes nothing.                           */
FP8BS_API fp8bs_status fp8_mx_gemm_grouped(int op, int32_t groups, const int32_t* offsets_dev,
                                           const int32_t* offsets_host, int64_t rows, const uint8_t* a,
                                           const uint8_t* a_scale_atoms, const uint8_t* b,
                                           const uint8_t* b_scale_atoms, int64_t N, int64_t K, void* out,
                                           void* stream);

/* Transposed MXFP8 cast: the fp8_mx_quant_1x32 cast of x^T, i.e. blocks of  */
/* 32 consecutive rows (tokens) of x. It gives the operands whose contraction */
/* runs along x's rows: dY^T and X^T for Wgrad, W^T (from W [K x N]) for      */
/* Fprop.                                                                     */
/* x       : BF16 [rows x cols], dense, cols % 16 == 0.                       */
/* qT      : E4M3 [cols x Mpad], Mpad = 128 * ceil(rows / 128); the padding   */
/*           tokens are written as 0x00.                                      */
/* scale_atoms : fp8bs_mx_scale_bytes(cols, Mpad) bytes, the atoms of qT (a   */
/*           [cols x Mpad] matrix), padding rows 127.                          */
/* The result is byte-identical to fp8_mx_quant_1x32 of the zero-padded       */
/* transpose.                                                                 */
FP8BS_API fp8bs_status fp8_mx_quant_1x32_T(const void* x, int64_t rows, int64_t cols, uint8_t* qT,
                                           uint8_t* scale_atoms, void* stream);

/* The packed Blackwell scale layout for power-of-two scales ([P4]  */
/* conventions table, row "Compact formats": fp32 scale containers on Hopper, */
/* packed exponent bytes on Blackwell, packed at the GEMM boundary). Writes   */
/* the exponent byte E of each fp32 scale s = 2^(E - 127) of a block-scaled   */
/* operand into the scale atoms of fp8_mx_gemm (layout above), the scale of   */
/* each 128-element K-block repeated over its four 32-element blocks, so that */
/* fp8_mx_gemm / fp8_mx_gemm_f32 compute the 1x128 / 128x128 recipe's GEMM    */
/* with the tensor core applying the scales (exact for power-of-two scales:   */
/* only the fp32 summation order differs from the promoted GEMMs above).      */
/* Scales come from the quantizers with FP8BS_SCALE_UE8M0.                    */
/* The operand is [rows x K], K contiguous, K % 128 == 0 (the contraction).   */
/* The scale of (row r, K-block b) is                                          */
/*   scales[(r / row_block) * row_stride + b * kb_stride], row_block 1 or 128: */
/*   1x128 scales (S1 layout):      row_block 1,   row_stride 1,             */
/*                                  kb_stride = fp8bs_scale_ld(rows);         */
/*   128x1 transposed scales (S3):  row_block 1,   row_stride 1,             */
/*                                  kb_stride = the operand's rows;           */
/*   W^T [N x K] from S2 scales:    row_block 128, row_stride 1,             */
/*                                  kb_stride = N / 128;                     */
/*   W [K x N] (Dgrad's B, contraction N): row_block 128,                     */
/*                                  row_stride = N / 128, kb_stride 1.        */
/* The caller's scale array must hold every index above. scale_atoms:         */
/* fp8bs_mx_scale_bytes(rows, K) bytes, 16-byte aligned; padding rows are     */
/* written as 127 (scale 1). A scale that is not a power of two in            */
/* [2^-127, 2^127] has no exponent byte: its bytes are written as 255 and     */
/* FP8BS_ERR_DEVICE is recorded in the device status word.                    */
FP8BS_API fp8bs_status fp8_pack_ue8m0(const float* scales, int64_t rows, int64_t K, int32_t row_block,
                                      int64_t row_stride, int64_t kb_stride, uint8_t* scale_atoms,
                                      void* stream);

/* For experts: fp8_pack_ue8m0 for the grouped rows of a 1x128-cast   */
/* operand [rows x K] (the A of a grouped Fprop or Dgrad), into the groups'  */
/* tile layout that fp8_mx_gemm_grouped reads: the scale of (row r, K-block  */
/* b) is scales[r + b * kb_stride] (the S1 layout: kb_stride =               */
/* fp8bs_scale_ld(rows)); row l of group g goes to row l % 128 of tile       */
/* (tiles of the groups before g) + l / 128. Rows of a group's last tile    */
/* past its end are written as 127 (scale 1). Offsets as in                  */
/* fp8_block_gemm_grouped (exactly one of offsets_dev / offsets_host);       */
/* scale_atoms: fp8bs_mx_scale_bytes(Tpad, K) bytes, 16-byte aligned (Tpad   */
/* as in fp8_mx_gemm_grouped). A scale without an exponent byte, or invalid  */
/* device offsets, record FP8BS_ERR_DEVICE.                                  */
FP8BS_API fp8bs_status fp8_pack_ue8m0_grouped(const float* scales, int64_t rows, int64_t K, int64_t kb_stride,
                                              int32_t groups, const int32_t* offsets_dev,
                                              const int32_t* offsets_host, uint8_t* scale_atoms, void* stream);

/* The casts with their scales already packed. The same casts as   */
/* fp8_quant_128x128_opts, fp8_quant_dual_opts and fp8_quant_dual_stash_opts */
/* under the UE8M0 rule (opts->rule must be FP8BS_SCALE_UE8M0, else          */
/* FP8BS_ERR_ARG), which in the same pass also write the exponent bytes of  */
/* their scales into the MX scale atoms of the GEMM operands they feed,      */
/* byte-identical to fp8_pack_ue8m0 of the fp32 scales they return (so the  */
/* MX GEMMs can follow directly, with no packing launch in between).         */
/*   fp8_quant_128x128_packed: W [rows x cols] per batch entry, rows and     */
/*     cols multiples of 128 (else FP8BS_ERR_SHAPE); qT optional (NULL when  */
/*     Fprop reads q through fp8_mx_gemm_wkn); atoms_wT: the atoms of        */
/*     W^T [cols x rows] (Fprop's B), atoms_w: those of W [rows x cols]      */
/*     with the contraction along cols (Dgrad's B); each                     */
/*     fp8bs_mx_scale_bytes(cols, rows) bytes per batch entry, entries       */
/*     consecutive.                                                          */
/*   fp8_quant_dual_packed / fp8_quant_dual_stash_packed: dense x (the      */
/*     _grouped forms below take expert groups), cols % 128 == 0; q_atoms:  */
/*     the atoms of q [rows x cols]                                          */
/*     (fp8bs_mx_scale_bytes(rows, cols) bytes, padding rows 127); qT_atoms: */
/*     those of qT [cols x Mpad] (fp8bs_mx_scale_bytes(cols, Mpad) bytes).   */
/* Atom pointers 16-byte aligned. A scale without an exponent byte (below    */
/* 2^-127, from a tile of tiny values) gets 255 and records FP8BS_ERR_DEVICE */
/* in the device status word, as fp8_pack_ue8m0 does.                        */
FP8BS_API fp8bs_status fp8_quant_128x128_packed(const void* w, int64_t batch, int64_t rows, int64_t cols,
                                                int64_t ldw, uint8_t* q, uint8_t* qT, float* scales,
                                                uint8_t* atoms_wT, uint8_t* atoms_w,
                                                const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_packed(const void* x, int64_t rows, int64_t cols, uint8_t* q,
                                             float* scales, uint8_t* qT, float* scalesT, uint8_t* q_atoms,
                                             uint8_t* qT_atoms, const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_stash_packed(const void* x, int64_t rows, int64_t cols, uint8_t* q,
                                                   float* scales, uint8_t* qT, float* scalesT, uint8_t* q_atoms,
                                                   uint8_t* qT_atoms, const fp8bs_scale_opts* opts,
                                                   void* stream);

/* The same two casts for expert groups (the MoE A and dY casts), with the   */
/* group offsets of fp8_block_gemm_grouped (exactly one of offsets_dev /     */
/* offsets_host, groups + 1 entries): q and scales as fp8_quant_1x128, qT   */
/* and scalesT as the grouped fp8_requant_128x1_T ([cols x Mpad], each group */
/* padded to 128 tokens; with device offsets Mpad is                        */
/* fp8bs_padded_tokens_max(rows, groups) and only the groups' padded tokens */
/* are written). q_atoms: the atoms of q in the groups' tile layout that     */
/* fp8_pack_ue8m0_grouped writes (fp8bs_mx_scale_bytes(Mpad, cols) bytes);  */
/* qT_atoms: those of qT [cols x Mpad] (fp8bs_mx_scale_bytes(cols, Mpad)     */
/* bytes). Byte-identical to the grouped casts followed by                  */
/* fp8_pack_ue8m0_grouped of scales and fp8_pack_ue8m0 of scalesT over the   */
/* groups' padded tokens; atoms of tiles past those tokens are not written. */
FP8BS_API fp8bs_status fp8_quant_dual_packed_grouped(const void* x, int64_t rows, int64_t cols,
                                                     const int32_t* offsets_dev, const int32_t* offsets_host,
                                                     int32_t groups, uint8_t* q, float* scales, uint8_t* qT,
                                                     float* scalesT, uint8_t* q_atoms, uint8_t* qT_atoms,
                                                     const fp8bs_scale_opts* opts, void* stream);
FP8BS_API fp8bs_status fp8_quant_dual_stash_packed_grouped(const void* x, int64_t rows, int64_t cols,
                                                           const int32_t* offsets_dev, const int32_t* offsets_host,
                                                           int32_t groups, uint8_t* q, float* scales, uint8_t* qT,
                                                           float* scalesT, uint8_t* q_atoms, uint8_t* qT_atoms,
                                                           const fp8bs_scale_opts* opts, void* stream);

/* ------------------------------------------------------------------------ */
/* S7. Grouped (MoE expert) GEMMs                                             */
/* The dense definitions above applied to each group (expert) g, whose token  */
/* rows are [offsets[g], offsets[g+1]) (int32, groups + 1 entries,            */
/* offsets[0] = 0, non-decreasing, offsets[groups] = rows). Empty groups are  */
/* allowed: they produce no rows (Fprop, Dgrad) or a zero weight gradient     */
/* (Wgrad). [P1] bullet 1 (the same recipe for every linear); the MoE form is */
/* the grouped-GEMM path of TransformerEngine PR #3573 ("Changes": grouped    */
/* predicates and per-group paths) and prime-rl PR #4073 ("Tests": grouped    */
/* operators with empty experts).                                             */
/* ------------------------------------------------------------------------ */
/* offsets_dev / offsets_host: exactly one is non-NULL (FP8BS_ERR_ARG otherwise).
 *   offsets_host: a HOST array; the call plans the exact tile grid on the host.
 *   offsets_dev : a DEVICE array (4-byte aligned) that the kernel reads when it
 *     runs, so the offsets may be produced on the device by earlier work on the
 *     same stream (a router) and the call can be captured in a CUDA graph whose
 *     routing changes between replays. The grid then covers the largest tile
 *     count any split of `rows` can need; invalid device offsets (offsets[0] != 0,
 *     a decrease, a total other than rows) record FP8BS_ERR_DEVICE in the device
 *     status word and the kernel writes nothing.
 * rows: total token rows M (the A rows for Fprop / Dgrad; the tokens the
 *   transposed casts were given for Wgrad).
 * op = FP8BS_OP_FPROP:
 *   a  = Xq [M x K], sa its 1x128 scales;
 *   b  = stacked WqT [groups x N x K], sb = stacked sw [groups x K/128 x N/128];
 *   out = Y BF16 [M x N].
 * op = FP8BS_OP_FPROP_WKN: as FP8BS_OP_FPROP with
 *   b  = stacked Wq [groups x K x N] (the q output of the batched cast, the
 *        same codes Dgrad reads), taken MN-major as in fp8_block_gemm_fprop_wkn.
 * op = FP8BS_OP_DGRAD (N is the contraction, K the output width):
 *   a  = dYq [M x N], sa its 1x128 scales;
 *   b  = stacked Wq [groups x K x N], sb = stacked sw [groups x K/128 x N/128];
 *   out = dX BF16 [M x K].
 * op = FP8BS_OP_WGRAD:
 *   a  = dYqT [N x Mpad], sa = sdyT [Mpad/128 x N], b = XqT [K x Mpad],
 *   sb = sxT [Mpad/128 x K] from the transposed casts with the same offsets:
 *   Mpad = fp8bs_padded_tokens(rows, offsets_host, groups) with host offsets,
 *   fp8bs_padded_tokens_max(rows, groups) with device offsets (the layout of
 *   the _dev casts);
 *   out = dW FP32 [groups x N x K]; accumulate as in fp8_block_gemm_wgrad.
 * Constraints: 1 <= groups <= FP8BS_MAX_GROUPS, N % 128 == 0, K % 128 == 0. */
FP8BS_API fp8bs_status fp8_block_gemm_grouped(int op, int32_t groups, const int32_t* offsets_dev,
                                              const int32_t* offsets_host, int64_t rows,
                                              const uint8_t* a, const float* sa,
                                              const uint8_t* b, const float* sb,
                                              int64_t N, int64_t K, void* out, int accumulate,
                                              void* stream);

/* ------------------------------------------------------------------------ */
/* Device status and failure detection                                       */
/* ------------------------------------------------------------------------ */

/* The device status word: one per device, holding the first device-side error
 * (FP8BS_ERR_TIMEOUT, FP8BS_ERR_DEVICE) any kernel of this library recorded on
 * that device since the last reset; FP8BS_OK (0) if none. */

/* Synchronizes the current device, then returns the status word. reset != 0
 * clears it. */
FP8BS_API fp8bs_status fp8bs_device_status(int reset);

/* Stream-ordered read: enqueues a copy of the status word on `stream` (and,
 * with reset != 0, its clearing after the copy), waits for that stream only
 * (cudaStreamSynchronize, not the whole device) and returns the value, i.e.
 * the status as of all work issued earlier on `stream`. Work on other streams
 * keeps running. Not for use while `stream` is being captured. */
FP8BS_API fp8bs_status fp8bs_last_device_status(void* stream, int reset);

/* Asynchronous form for graphs and pipelines: enqueues on `stream` a 4-byte
 * device-to-device copy of the status word into `dst` (a caller-owned DEVICE
 * word, 4-byte aligned) and, with reset != 0, its clearing. Never waits; may
 * be captured in a CUDA graph. */
FP8BS_API fp8bs_status fp8bs_copy_device_status(unsigned int* dst, int reset, void* stream);

/* Upper bound, in nanoseconds, on any single pipeline wait inside the GEMM
 * kernels (default 2e9). A wait that exceeds it records FP8BS_ERR_TIMEOUT,
 * the kernel drains its in-flight copies and returns. Host-global setting. */
FP8BS_API void fp8bs_set_wait_limit_ns(uint64_t ns);

/* Launches one CTA that waits on a barrier nothing will arrive on, bounded
 * by limit_ns; the wait gives up, records FP8BS_ERR_TIMEOUT in the device
 * status word and the kernel returns. Exercises the timeout path without a
 * fault; the context stays usable. */
FP8BS_API fp8bs_status fp8bs_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Runs fp8_block_gemm_fprop on the caller's operands (same arguments and
 * checks; K >= 384, so that a tile needs a tensor-memory buffer a second
 * time) with every wait bounded by limit_ns and with the promotion epilogue
 * holding on to the buffers it has read: the MMA thread's wait for a buffer
 * to come back can only give up. The GEMM then records FP8BS_ERR_TIMEOUT in
 * the device status word, stops issuing, lets its copies and MMAs drain,
 * frees its tensor memory and returns; y holds partial results. This
 * exercises the timeout path of a real GEMM without a fault; the context
 * stays usable. Test hook: not part of the computation. */
FP8BS_API fp8bs_status fp8bs_selftest_gemm_timeout(const uint8_t* xq, const float* sx, const uint8_t* wqT,
                                                   const float* sw, int64_t M, int64_t N, int64_t K, void* y,
                                                   uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
