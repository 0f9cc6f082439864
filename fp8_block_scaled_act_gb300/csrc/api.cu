// api.cu -- the extern "C" entry points declared in fp8bs.h: argument
// validation, per-device setup, TMA tensor maps and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "fp8bs.h"
#include "internal.h"

namespace fp8bs {
namespace {

// Device-side status word: the first error a kernel records (0 = none).
__device__ unsigned int g_device_status;

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::atomic<bool> ready{false};
    bool supported = false;
    int num_sms = 0;
    unsigned int* status = nullptr;
    // stream-K GEMM workspaces, one per stream that has run a stream-K GEMM
    // on this device (so that GEMMs on different streams never share one):
    // one partial 128 x 256 fp32 tile and one flag per SM each
    struct SkSlot {
        cudaStream_t stream = nullptr;
        float* ws = nullptr;
        unsigned int* flags = nullptr;
    };
    static constexpr int kSkSlots = 8;
    SkSlot sk[kSkSlots];
    int sk_used = 0;
    // the workspace of GEMMs captured into CUDA graphs (a capturing stream
    // cannot allocate); allocated with the device's set-up
    SkSlot sk_graph;
};

// One stream-K workspace (a partial tile and a flag per SM); false if the
// allocation failed.
bool alloc_stream_k(DeviceState& st, DeviceState::SkSlot& sl, cudaStream_t stream)
{
    void* ws = nullptr;
    void* fl = nullptr;
    const size_t ws_bytes = static_cast<size_t>(st.num_sms) * kBM * kBN * sizeof(float);
    if (cudaMalloc(&ws, ws_bytes) != cudaSuccess || cudaMalloc(&fl, st.num_sms * sizeof(unsigned int)) != cudaSuccess ||
        cudaMemset(fl, 0, st.num_sms * sizeof(unsigned int)) != cudaSuccess) {
        if (ws) cudaFree(ws);
        if (fl) cudaFree(fl);
        cudaGetLastError();
        return false;
    }
    sl.stream = stream;
    sl.ws = static_cast<float*>(ws);
    sl.flags = static_cast<unsigned int*>(fl);
    return true;
}

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device setup on first use: capability check, SM count, the address of
// the status word. Runs once per device (it makes CUDA runtime calls that a
// stream capture would reject, so the first call on a device should come
// before any capture).
fp8bs_status device_state(DeviceState** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8BS_ERR_UNSUPPORTED;
    DeviceState& st = g_devices[dev];
    if (st.ready.load(std::memory_order_acquire)) {   // set-up done: no lock
        if (!st.supported || !g_encode) return FP8BS_ERR_UNSUPPORTED;
        *out = &st;
        return FP8BS_OK;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!st.ready.load(std::memory_order_relaxed)) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FP8BS_ERR_UNSUPPORTED;
        st.supported = (prop.major == 10 && prop.minor == 3);
        st.num_sms = prop.multiProcessorCount;
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return FP8BS_ERR_UNSUPPORTED;
        st.status = static_cast<unsigned int*>(ptr);
        if (st.supported) alloc_stream_k(st, st.sk_graph, nullptr);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) == cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        st.ready.store(true, std::memory_order_release);
    }
    if (!st.supported || !g_encode) return FP8BS_ERR_UNSUPPORTED;
    *out = &st;
    return FP8BS_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The MXFP8 GEMM with BF16 (out_bf16) or FP32 (out_f32) output (defined
// after the extern "C" wrappers).
fp8bs_status mx_gemm_common(const uint8_t* a, const uint8_t* a_scale_atoms, const uint8_t* b,
                            const uint8_t* b_scale_atoms, int64_t M, int64_t N, int64_t K, uint16_t* out_bf16,
                            float* out_f32, void* stream, bool b_mn = false);
fp8bs_status mx_gemm_grouped(int op, int32_t groups, const int32_t* offsets_dev, const int32_t* offsets_host,
                             int64_t rows, const uint8_t* a, const uint8_t* a_atoms, const uint8_t* b,
                             const uint8_t* b_atoms, int64_t N, int64_t K, void* out, void* stream);

// The quantizer entry points with an optional stochastic-rounding key
// (defined after the extern "C" wrappers).
fp8bs_status quant_1x128_common(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                float* scales, const fp8bs_scale_opts* opts, const SrParams* sr, void* stream);
fp8bs_status quant_128x128_common(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ldw,
                                  uint8_t* q, uint8_t* qT, float* scales, const fp8bs_scale_opts* opts,
                                  const SrParams* sr, void* stream, uint8_t* atoms_wT, uint8_t* atoms_w);

// Public scale options -> kernel rule; false for invalid options.
bool to_rule(const fp8bs_scale_opts* o, ScaleRule* r)
{
    r->ue8m0 = 0;
    r->amax_floor = 0.0f;
    r->scale_floor = 0.0f;
    if (!o) return true;
    if (o->rule != FP8BS_SCALE_FP32 && o->rule != FP8BS_SCALE_UE8M0) return false;
    if (!(o->amax_floor >= 0.0f && o->amax_floor <= 3.0e38f)) return false;     // also rejects NaN
    if (!(o->scale_floor >= 0.0f && o->scale_floor <= 3.0e38f)) return false;
    r->ue8m0 = o->rule == FP8BS_SCALE_UE8M0 ? 1 : 0;
    r->amax_floor = o->amax_floor;
    r->scale_floor = o->scale_floor;
    return true;
}

inline fp8bs_status launch_status(cudaError_t e) { return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH; }

// 2D E4M3 tensor map over a row-major [outer x inner] byte matrix, box
// [box_outer x 128 bytes], 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_outer)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {128u, box_outer};
    const cuuint32_t estr[2] = {1u, 1u};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over a BF16 GEMM output [rows x cols] (row-major, 16-byte aligned
// rows) for the epilogue's TMA stores: box of 64 columns x 32 rows, 128-byte
// swizzle (the layout the epilogue writes into shared memory).
bool make_out_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64u, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over a BF16 cast source [rows x cols] with row pitch `row_bytes`
// (a multiple of 16): box of 64 columns x box_rows rows, 128-byte swizzle,
// zero fill out of bounds.
bool make_src_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                  uint32_t box_rows)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {64u, box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor-map cache. Encoding a map is a driver call of a microsecond or
// two; an eager caller repeats the same few (pointer, shape) pairs, so each
// host thread keeps a small direct-mapped cache of encoded maps keyed by the
// device and every argument of the encoding. A hit copies the 128-byte map.
struct MapKey {
    int dev;
    int kind;   // 0: E4M3 operand map, 1: BF16 output map, 2: BF16 cast source map,
                // 3: batched BF16 weights, 4: batched E4M3 weight codes
    const void* base;
    uint64_t inner, outer, row_bytes;
    uint32_t box_outer;
    uint64_t depth = 1;   // batch entries (three-dimensional maps)
    bool operator==(const MapKey& o) const
    {
        return dev == o.dev && kind == o.kind && base == o.base && inner == o.inner && outer == o.outer &&
               row_bytes == o.row_bytes && box_outer == o.box_outer && depth == o.depth;
    }
};

struct MapSlot {
    bool used = false;
    MapKey key;
    CUtensorMap map;
};

constexpr int kMapSlots = 64;
thread_local MapSlot t_maps[kMapSlots];

MapSlot& map_slot(const MapKey& k)
{
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) >> 4;
    h ^= k.inner * 0x9E3779B97F4A7C15ull ^ k.outer * 0xC2B2AE3D27D4EB4Full ^ k.row_bytes * 0x165667B19E3779F9ull;
    h ^= (static_cast<uint64_t>(k.box_outer) << 32) ^ (static_cast<uint64_t>(k.dev) << 8) ^ k.kind;
    h ^= k.depth * 0x27D4EB2F165667C5ull;
    h ^= h >> 29;
    return t_maps[h % kMapSlots];
}

bool cached_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                uint32_t box_outer)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const MapKey k{dev, 0, base, inner, outer, row_bytes, box_outer};
    MapSlot& sl = map_slot(k);
    if (sl.used && sl.key == k) {
        *m = sl.map;
        return true;
    }
    if (!make_map(m, base, inner, outer, row_bytes, box_outer)) return false;
    sl.used = true;
    sl.key = k;
    sl.map = *m;
    return true;
}

bool cached_out_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const MapKey k{dev, 1, base, cols, rows, cols * 2, 32u};
    MapSlot& sl = map_slot(k);
    if (sl.used && sl.key == k) {
        *m = sl.map;
        return true;
    }
    if (!make_out_map(m, base, cols, rows)) return false;
    sl.used = true;
    sl.key = k;
    sl.map = *m;
    return true;
}

bool cached_src_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_rows = 32u)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const MapKey k{dev, 2, base, cols, rows, row_bytes, box_rows};
    MapSlot& sl = map_slot(k);
    if (sl.used && sl.key == k) {
        *m = sl.map;
        return true;
    }
    if (!make_src_map(m, base, cols, rows, row_bytes, box_rows)) return false;
    sl.used = true;
    sl.key = k;
    sl.map = *m;
    return true;
}

// 3D map over batched weights [batch][rows][cols] (BF16, row pitch
// row_bytes; or E4M3 codes, dense) with boxes of one batch entry: box_cols
// columns x 128 rows, 128-byte swizzle, zero fill out of bounds (so a box
// never reaches into the next batch entry).
bool cached_batch_map(CUtensorMap* m, bool bf16, const void* base, uint64_t cols, uint64_t rows, uint64_t batch,
                      uint64_t row_bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    MapKey k{dev, bf16 ? 3 : 4, base, cols, rows, row_bytes, 128u};
    k.depth = batch;
    MapSlot& sl = map_slot(k);
    if (sl.used && sl.key == k) {
        *m = sl.map;
        return true;
    }
    const cuuint64_t dims[3] = {cols, rows, batch};
    const cuuint64_t strides[2] = {row_bytes, row_bytes * rows};
    const cuuint32_t box[3] = {bf16 ? 64u : 128u, 128u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    if (g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base),
                 dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    sl.used = true;
    sl.key = k;
    sl.map = *m;
    return true;
}

// The stream-K workspace for a GEMM on `stream`: a capturing stream gets the
// device's graph workspace; any other stream its own, allocated by its first
// stream-K GEMM. Null when none can be had (the table is full or the
// allocation failed): the GEMM then runs without stream-K.
DeviceState::SkSlot* stream_k_slot(DeviceState* st, cudaStream_t stream)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cap != cudaStreamCaptureStatusNone) return st->sk_graph.ws ? &st->sk_graph : nullptr;
    for (int i = 0; i < st->sk_used; ++i)
        if (st->sk[i].stream == stream) return &st->sk[i];
    if (st->sk_used == DeviceState::kSkSlots) return nullptr;
    if (!alloc_stream_k(*st, st->sk[st->sk_used], stream)) return nullptr;
    return &st->sk[st->sk_used++];
}

// Clears the stream-K flags of every workspace of this device (a GEMM that
// gave up may have left a published partial unconsumed).
cudaError_t clear_stream_k_flags(DeviceState* st, cudaStream_t stream, bool async)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    const size_t n = st->num_sms * sizeof(unsigned int);
    for (int i = -1; i < st->sk_used; ++i) {
        unsigned int* f = i < 0 ? st->sk_graph.flags : st->sk[i].flags;
        if (!f) continue;
        const cudaError_t e = async ? cudaMemsetAsync(f, 0, n, stream) : cudaMemset(f, 0, n);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

void init_params(GemmParams& p, DeviceState* st, int n_cols)
{
    std::memset(&p, 0, sizeof(p));
    p.n_cols = n_cols;
    p.n_tiles = (n_cols + kBN - 1) / kBN;
    p.splits = 1;
    p.kb_per_split = 1 << 30;
    p.wait_limit_ns = g_wait_limit_ns;
    p.status = st->status;
}

// Validates group offsets (host array of groups + 1 entries).
bool valid_offsets(const int32_t* off, int32_t groups)
{
    if (!off || groups < 1 || groups > kMaxGroups || off[0] != 0) return false;
    for (int g = 0; g < groups; ++g)
        if (off[g + 1] < off[g]) return false;
    return true;
}

int64_t padded_tokens(int64_t rows, const int32_t* off, int32_t groups)
{
    if (!off || groups == 0) return (rows + 127) / 128 * 128;
    int64_t tot = 0;
    for (int g = 0; g < groups; ++g) tot += (static_cast<int64_t>(off[g + 1] - off[g]) + 127) / 128 * 128;
    return tot;
}

// Upper bound on the padded token count of `groups` groups holding `rows`
// tokens in total: at most k = min(groups, rows) groups are non-empty and
// sum_g ceil(T_g / 128) <= floor((rows + 127 k) / 128).
int64_t padded_tokens_max(int64_t rows, int32_t groups)
{
    const int64_t k = groups < rows ? groups : rows;
    if (k <= 1) return (rows + 127) / 128 * 128;
    return (rows + 127 * k) / 128 * 128;
}

// Fprop / Dgrad, dense or grouped. For Fprop the contraction length is K and
// the output width N; for Dgrad they are N and K. `contr` and `width` are
// those two; b rows per group = width.
// Split-K shape: with `splits` requested over nkb K-blocks, each range takes
// kps = ceil(nkb / splits) blocks and `used` = ceil(nkb / kps) ranges are
// non-empty.
void splitk_shape(int64_t nkb, int64_t splits, int& used, int& kps)
{
    if (splits > nkb) splits = nkb;
    if (splits < 1) splits = 1;
    kps = static_cast<int>((nkb + splits - 1) / splits);
    used = static_cast<int>((nkb + kps - 1) / kps);
}

// The ops of the row-wise GEMM (Fprop in either B layout, Dgrad).
bool rowwise_op(int op)
{
    return op == FP8BS_OP_FPROP || op == FP8BS_OP_FPROP_WKN || op == FP8BS_OP_DGRAD;
}

// Group offsets of a call: exactly one of host (planned on the host) and
// dev (read by the kernel) is set; `rows` is the total token count.
struct Offsets {
    const int32_t* host;
    const int32_t* dev;
    int32_t groups;
    int64_t rows;
};

void copy_offsets(GemmParams& p, const Offsets& o)
{
    p.num_groups = o.groups;
    if (o.dev) {
        p.off_dev = o.dev;
    } else {
        for (int g = 0; g <= o.groups; ++g) p.off[g] = o.host[g];
    }
}

// Fprop / Dgrad, dense or grouped; with splits > 1 (dense only) the
// K-blocks of every tile are cut into ranges whose fp32 sums go to the
// workspace `ws`, followed by the reduction kernel.
// op: FP8BS_OP_FPROP (b = W^T codes [N x K]), FP8BS_OP_FPROP_WKN (b = W codes
// [K x N], read MN-major) or FP8BS_OP_DGRAD (b = W codes [K x N]).
fp8bs_status run_rowwise_gemm(int op, const Offsets& o, const uint8_t* a, const float* sa, const uint8_t* b,
                              const float* sb, int64_t N, int64_t K, void* out, void* stream, int32_t splits = 1,
                              float* ws = nullptr, uint64_t selftest_limit_ns = 0)
{
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    const bool dgrad = op == FP8BS_OP_DGRAD;
    const bool b_mn = op == FP8BS_OP_FPROP_WKN;
    const int64_t contr = dgrad ? N : K;
    const int64_t width = dgrad ? K : N;
    const int64_t M = o.rows;
    if (M == 0) return FP8BS_OK;
    if (M > 0x7FFFFFFF - kBM * static_cast<int64_t>(o.groups) || width * o.groups > 0x7FFFFFFF ||
        contr > 0x7FFFFFFF || (b_mn && contr * o.groups > 0x7FFFFFFF))   // MN-major B rows: contr x groups
        return FP8BS_ERR_SHAPE;

    GemmParams p;
    init_params(p, st, static_cast<int>(width));
    p.layout = kRowGroups;
    copy_offsets(p, o);
    p.kblocks = static_cast<int>(contr / kBK);
    p.b_group_rows = static_cast<int>(b_mn ? contr : width);
    p.b_mn = b_mn ? 1 : 0;
    p.rows_total = static_cast<int>(M);
    p.sb_group_stride = (K / 128) * (N / 128);
    // tiles: exact from host offsets, else the bound over any split of M rows
    int64_t row_tiles = 0;
    if (o.host) {
        for (int g = 0; g < o.groups; ++g) row_tiles += (o.host[g + 1] - o.host[g] + kBM - 1) / kBM;
    } else {
        row_tiles = padded_tokens_max(M, o.groups) / kBM;
    }
    p.sa = sa;
    p.sa_ld = fp8bs_scale_ld(M);
    p.sa_rows = static_cast<int>(p.sa_ld);
    p.sb = sb;
    // sw is [K/128 x N/128]: Fprop walks K-blocks along its rows, Dgrad along its columns
    p.sb_kstride = dgrad ? 1 : N / 128;
    p.sb_cstride = dgrad ? N / 128 : 1;
    p.out = out;
    p.out_ld = width;
    p.accumulate = 0;
    if (selftest_limit_ns != 0) {   // fp8bs_selftest_gemm_timeout
        p.hold_release = 1;
        p.wait_limit_ns = selftest_limit_ns;
    }
    int used = 1, kps = 1 << 30;
    if (splits > 1 && o.groups == 1) splitk_shape(contr / kBK, splits, used, kps);
    if (used > 1) {
        if (!ws) return FP8BS_ERR_ARG;
        p.splits = used;
        p.kb_per_split = kps;
        p.ws = ws;
        p.ws_split_stride = splitk_tile_floats(M, width);
    }

    CUtensorMap ma, mb, mo;
    std::memset(&mo, 0, sizeof(mo));
    if (!cached_map(&ma, a, contr, M, contr, kBM)) return FP8BS_ERR_ARG;
    // B: [width x contr] K-major boxes of 256 rows, or [contr x width]
    // (MN-major) boxes of 128 K rows x 128 columns
    if (b_mn ? !cached_map(&mb, b, width, contr * o.groups, width, kBK)
             : !cached_map(&mb, b, contr, width * o.groups, contr, kBN))
        return FP8BS_ERR_ARG;
    if (used <= 1) {
        if (!cached_out_map(&mo, out, width, M)) return FP8BS_ERR_ARG;
        p.tma_store = 1;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int64_t max_units = row_tiles * p.n_tiles * p.splits;
    // Stream-K when the tiles fill the persistent grid's last round poorly
    // (one group with host offsets, no split-K): every CTA then takes the
    // same number of K-blocks, and a tile cut between two CTAs is finished
    // by the first of them.
    if (used <= 1 && o.groups == 1 && o.host && selftest_limit_ns == 0 && max_units > st->num_sms &&
        max_units * p.kblocks < 0x7FFFFFFF - 2 * static_cast<int64_t>(st->num_sms) * p.kblocks) {
        const int64_t grid = st->num_sms;
        const int64_t rounds = (max_units + grid - 1) / grid;
        DeviceState::SkSlot* sl = nullptr;
        if (static_cast<double>(max_units) < 0.9 * static_cast<double>(rounds * grid) &&
            (sl = stream_k_slot(st, cs)) != nullptr) {
            const int64_t total = max_units * p.kblocks;
            p.sk_len = static_cast<int>((total + grid - 1) / grid);   // >= p.kblocks since max_units > grid
            // a range of sk_len K-blocks touches at most this many tiles
            p.sk_units = (p.sk_len + p.kblocks - 1) / p.kblocks + 1;
            p.sk_ws = sl->ws;
            p.sk_flags = sl->flags;
            max_units = grid;
        }
    }
    const fp8bs_status r =
        launch_status(launch_gemm(GemmKind::kBlockScaleBf16, ma, mb, mo, p, max_units, st->num_sms, cs));
    if (r != FP8BS_OK || used <= 1) return r;
    return launch_status(
        launch_splitk_reduce(ws, used, M, width, static_cast<uint16_t*>(out), st->num_sms, cs));
}

// Wgrad, dense (one group over all T tokens) or grouped (padded segments,
// T = the padded token count of the operands).
fp8bs_status run_wgrad(const Offsets& o, int64_t T, const uint8_t* a, const float* sa, const uint8_t* b,
                       const float* sb, int64_t N, int64_t K, float* out, int accumulate, void* stream)
{
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    if (N > 0x7FFFFFFF || K > 0x7FFFFFFF || T > 0x7FFFFFFF || N * K * o.groups > (int64_t(1) << 62))
        return FP8BS_ERR_SHAPE;
    if (T == 0) {
        if (accumulate) return FP8BS_OK;
        return launch_status(cudaMemsetAsync(out, 0, sizeof(float) * N * K * o.groups,
                                             static_cast<cudaStream_t>(stream)));
    }
    GemmParams p;
    init_params(p, st, static_cast<int>(K));
    p.layout = kTokenGroups;
    copy_offsets(p, o);
    p.out_rows = static_cast<int>(N);
    p.tcap = static_cast<int>(T);
    p.out_group_stride = N * K;
    p.sa = sa;
    p.sa_ld = N;
    p.sa_rows = static_cast<int>(N);
    p.sb = sb;
    p.sb_kstride = K;
    p.sb_cstride = 1;
    p.out = out;
    p.out_ld = K;
    p.accumulate = accumulate ? 1 : 0;

    // Wgrad stores its FP32 tile from registers (a TMA store through shared
    // memory measured slower), so its output map stays unused
    CUtensorMap ma, mb, mo;
    std::memset(&mo, 0, sizeof(mo));
    if (!cached_map(&ma, a, T, N, T, kBM) || !cached_map(&mb, b, T, K, T, kBN)) return FP8BS_ERR_ARG;
    const int64_t max_units = static_cast<int64_t>(o.groups) * (N / kBM) * p.n_tiles;
    return launch_status(launch_gemm(GemmKind::kVectorScaleF32, ma, mb, mo, p, max_units, st->num_sms,
                                     static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" {

const char* fp8bs_status_str(fp8bs_status s)
{
    switch (s) {
    case FP8BS_OK: return "ok";
    case FP8BS_ERR_ARG: return "invalid argument";
    case FP8BS_ERR_ALIGN: return "misaligned pointer or stride";
    case FP8BS_ERR_SHAPE: return "unsupported shape";
    case FP8BS_ERR_LAUNCH: return "kernel launch failed";
    case FP8BS_ERR_TIMEOUT: return "device wait timed out";
    case FP8BS_ERR_UNSUPPORTED: return "unsupported device (needs sm_103a)";
    case FP8BS_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

int fp8bs_version(void) { return 100; }

int64_t fp8bs_scale_ld(int64_t rows) { return rows <= 0 ? 0 : (rows + 3) / 4 * 4; }

int64_t fp8bs_padded_tokens(int64_t rows, const int32_t* group_offsets_host, int32_t groups)
{
    if (rows < 0) return -1;
    if (group_offsets_host && groups > 0) {
        if (!valid_offsets(group_offsets_host, groups) || group_offsets_host[groups] != rows) return -1;
    }
    return padded_tokens(rows, group_offsets_host, groups);
}

fp8bs_status fp8_quant_1x128(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                             float* scales, void* stream)
{
    return fp8_quant_1x128_opts(x, rows, cols, ldx, q, scales, nullptr, stream);
}

fp8bs_status fp8_quant_1x128_opts(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                  float* scales, const fp8bs_scale_opts* opts, void* stream)
{
    return quant_1x128_common(x, rows, cols, ldx, q, scales, opts, nullptr, stream);
}

fp8bs_status fp8_quant_1x128_sr(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                float* scales, uint64_t seed, uint32_t salt, const fp8bs_scale_opts* opts,
                                void* stream)
{
    const SrParams sr{seed, salt};
    return quant_1x128_common(x, rows, cols, ldx, q, scales, opts, &sr, stream);
}

}  // extern "C"

namespace fp8bs {
namespace {

fp8bs_status quant_1x128_common(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                float* scales, const fp8bs_scale_opts* opts, const SrParams* sr, void* stream)
{
    ScaleRule rule;
    if (!to_rule(opts, &rule)) return FP8BS_ERR_ARG;
    if (rows < 0 || cols <= 0 || ldx < cols) return FP8BS_ERR_ARG;
    if (cols % 16 != 0) return FP8BS_ERR_SHAPE;
    if (rows == 0) return FP8BS_OK;
    if (!x || !q || !scales) return FP8BS_ERR_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || ldx % 8 != 0) return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    if (!sr && rows <= 0x7FFFFFFF && cols <= 0x7FFFFFFF) {
        // round to nearest: the TMA-fed kernel (codes leave through a byte
        // map with a box of 32 rows x 128 columns)
        CUtensorMap map_x, map_q;
        if (!cached_src_map(&map_x, x, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(ldx) * 2) ||
            !cached_map(&map_q, q, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                        static_cast<uint64_t>(cols), 32u))
            return FP8BS_ERR_LAUNCH;
        return launch_status(launch_quant_1x128_stream(map_x, map_q, rows, cols, scales, fp8bs_scale_ld(rows),
                                                       rule, g_wait_limit_ns, st->status, st->num_sms,
                                                       static_cast<cudaStream_t>(stream)));
    }
    return launch_status(launch_quant_1x128(static_cast<const uint16_t*>(x), rows, cols, ldx, q,
                                            scales, fp8bs_scale_ld(rows), rule, sr, st->num_sms,
                                            static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace fp8bs

extern "C" {

fp8bs_status fp8_quant_128x128(const void* w, int64_t batch, int64_t rows, int64_t cols,
                               int64_t ldw, uint8_t* q, uint8_t* qT, float* scales, void* stream)
{
    return fp8_quant_128x128_opts(w, batch, rows, cols, ldw, q, qT, scales, nullptr, stream);
}

fp8bs_status fp8_quant_128x128_opts(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ldw,
                                    uint8_t* q, uint8_t* qT, float* scales, const fp8bs_scale_opts* opts,
                                    void* stream)
{
    return quant_128x128_common(w, batch, rows, cols, ldw, q, qT, scales, opts, nullptr, stream, nullptr, nullptr);
}

fp8bs_status fp8_quant_128x128_sr(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ldw,
                                  uint8_t* q, uint8_t* qT, float* scales, uint64_t seed, uint32_t salt,
                                  const fp8bs_scale_opts* opts, void* stream)
{
    const SrParams sr{seed, salt};
    return quant_128x128_common(w, batch, rows, cols, ldw, q, qT, scales, opts, &sr, stream, nullptr, nullptr);
}

}  // extern "C"

namespace fp8bs {
namespace {

fp8bs_status quant_128x128_common(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ldw,
                                  uint8_t* q, uint8_t* qT, float* scales, const fp8bs_scale_opts* opts,
                                  const SrParams* sr, void* stream, uint8_t* atoms_wT, uint8_t* atoms_w)
{
    ScaleRule rule;
    if (!to_rule(opts, &rule)) return FP8BS_ERR_ARG;
    if (batch < 1 || rows <= 0 || cols <= 0 || ldw < cols) return FP8BS_ERR_ARG;
    if (rows % 16 != 0 || cols % 16 != 0) return FP8BS_ERR_SHAPE;
    if (!w || !q || !scales) return FP8BS_ERR_ARG;
    if (!aligned16(w) || !aligned16(q) || (qT && !aligned16(qT)) || ldw % 8 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    if (!sr) {
        // round to nearest: the TMA-fed tile kernel
        CUtensorMap map_w, map_q;
        if (!cached_batch_map(&map_w, true, w, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                              static_cast<uint64_t>(batch), static_cast<uint64_t>(ldw) * 2) ||
            !cached_batch_map(&map_q, false, q, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                              static_cast<uint64_t>(batch), static_cast<uint64_t>(cols)))
            return FP8BS_ERR_LAUNCH;
        return launch_status(launch_wcast_tile(map_w, map_q, batch, rows, cols, qT, scales, rule, atoms_wT, atoms_w,
                                               st->status, g_wait_limit_ns, st->num_sms,
                                               static_cast<cudaStream_t>(stream)));
    }
    return launch_status(launch_quant_128x128(static_cast<const uint16_t*>(w), batch, rows, cols, ldw, q, qT,
                                              scales, rule, sr, static_cast<cudaStream_t>(stream), atoms_wT,
                                              atoms_w, st->status));
}

}  // namespace
}  // namespace fp8bs

extern "C" {

}  // extern "C"

namespace fp8bs {
namespace {

// The 128x1 transposed cast (S3), optionally with the same pass's 1x128 cast
// of a BF16 source (q, q_scales non-null).
fp8bs_status requant_common(int src_mode, const void* src, const float* src_scales, int64_t rows, int64_t cols,
                            const int32_t* group_offsets_host, int32_t groups, uint8_t* qT, float* scalesT,
                            uint8_t* q, float* q_scales, const fp8bs_scale_opts* opts, void* stream,
                            bool stash = false, const SrParams* sr = nullptr, uint8_t* q_atoms = nullptr,
                            uint8_t* qT_atoms = nullptr, const int32_t* offsets_dev = nullptr)
{
    ScaleRule rule;
    if (!to_rule(opts, &rule)) return FP8BS_ERR_ARG;
    if (src_mode != FP8BS_SRC_BF16 && src_mode != FP8BS_SRC_E4M3) return FP8BS_ERR_ARG;
    if (rows < 0 || cols <= 0 || groups < 0) return FP8BS_ERR_ARG;
    if (cols % 16 != 0) return FP8BS_ERR_SHAPE;
    if (rows > 0x7FFFFFFF) return FP8BS_ERR_SHAPE;
    if (offsets_dev && (group_offsets_host || groups < 1 || groups > kMaxGroups)) return FP8BS_ERR_ARG;
    if (offsets_dev && (reinterpret_cast<uintptr_t>(offsets_dev) & 3u) != 0) return FP8BS_ERR_ALIGN;
    const bool grouped = group_offsets_host && groups > 0;
    if (grouped && (!valid_offsets(group_offsets_host, groups) || group_offsets_host[groups] != rows))
        return FP8BS_ERR_ARG;
    const int64_t mpad = offsets_dev ? padded_tokens_max(rows, groups)
                                     : padded_tokens(rows, grouped ? group_offsets_host : nullptr, grouped ? groups : 0);
    if (mpad == 0) return FP8BS_OK;
    if (!src || !qT || !scalesT || (src_mode == FP8BS_SRC_E4M3 && !src_scales)) return FP8BS_ERR_ARG;
    if (!aligned16(src) || !aligned16(qT) || !aligned16(scalesT) ||
        (src_scales && !aligned16(src_scales)) || (q && !aligned16(q)) || (q_scales && !aligned16(q_scales)))
        return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;

    RequantParams p;
    std::memset(&p, 0, sizeof(p));
    p.mode = src_mode;
    p.src = src;
    p.src_scales = src_scales;
    p.src_scale_ld = fp8bs_scale_ld(rows);
    p.rows = rows;
    p.cols = cols;
    p.qT = qT;
    p.scT = scalesT;
    p.mpad = mpad;
    p.q = q;
    p.q_scales = q_scales;
    p.q_scale_ld = fp8bs_scale_ld(rows);
    p.stash = stash ? 1 : 0;
    p.rule = rule;
    p.q_atoms = q_atoms;
    p.qT_atoms = qT_atoms;
    p.status = st->status;
    if (sr) {
        // the 1x128 part of a dual cast takes (seed, salt), the transposed
        // part (seed, salt + 1); a plain requant's transposed cast (seed, salt)
        p.sr = 1;
        p.sr_seed = sr->seed;
        p.sr_salt_rows = sr->salt;
        p.sr_salt_cols = q ? sr->salt + 1u : sr->salt;
    }
    if (offsets_dev) {
        p.num_groups = groups;
        p.off_dev = offsets_dev;
    } else if (grouped) {
        p.num_groups = groups;
        int tiles = 0;
        for (int g = 0; g <= groups; ++g) p.off[g] = group_offsets_host[g];
        for (int g = 0; g < groups; ++g) {
            p.tile_start[g] = tiles;
            tiles += (group_offsets_host[g + 1] - group_offsets_host[g] + 127) / 128;
        }
        p.tile_start[groups] = tiles;
    } else {
        p.num_groups = 1;
        p.off[0] = 0;
        p.off[1] = static_cast<int32_t>(rows);
        p.tile_start[0] = 0;
        p.tile_start[1] = static_cast<int32_t>(mpad / 128);
    }
    if (q && q_scales && src_mode == FP8BS_SRC_BF16 && !sr) {
        // round to nearest, dense or grouped: the TMA-fed tile kernel
        CUtensorMap map_x, map_q;
        if (!cached_src_map(&map_x, src, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(cols) * 2, 128u) ||
            !cached_map(&map_q, q, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                        static_cast<uint64_t>(cols), 128u))
            return FP8BS_ERR_LAUNCH;
        return launch_status(
            launch_dual_tile(map_x, map_q, p, g_wait_limit_ns, st->num_sms, static_cast<cudaStream_t>(stream)));
    }
    return launch_status(launch_requant_128x1_T(p, static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace fp8bs

extern "C" {

fp8bs_status fp8_requant_128x1_T(int src_mode, const void* src, const float* src_scales,
                                 int64_t rows, int64_t cols, const int32_t* group_offsets_host,
                                 int32_t groups, uint8_t* qT, float* scalesT, void* stream)
{
    return requant_common(src_mode, src, src_scales, rows, cols, group_offsets_host, groups, qT, scalesT,
                          nullptr, nullptr, nullptr, stream);
}

fp8bs_status fp8_requant_128x1_T_opts(int src_mode, const void* src, const float* src_scales, int64_t rows,
                                      int64_t cols, const int32_t* group_offsets_host, int32_t groups,
                                      uint8_t* qT, float* scalesT, const fp8bs_scale_opts* opts, void* stream)
{
    return requant_common(src_mode, src, src_scales, rows, cols, group_offsets_host, groups, qT, scalesT,
                          nullptr, nullptr, opts, stream);
}

fp8bs_status fp8_quant_dual(const void* x, int64_t rows, int64_t cols, const int32_t* group_offsets_host,
                            int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                            void* stream)
{
    return fp8_quant_dual_opts(x, rows, cols, group_offsets_host, groups, q, scales, qT, scalesT, nullptr, stream);
}

fp8bs_status fp8_quant_dual_opts(const void* x, int64_t rows, int64_t cols, const int32_t* group_offsets_host,
                                 int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                 const fp8bs_scale_opts* opts, void* stream)
{
    if (rows > 0 && (!q || !scales)) return FP8BS_ERR_ARG;
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, group_offsets_host, groups, qT, scalesT, q,
                          scales, opts, stream);
}

fp8bs_status fp8_quant_dual_stash(const void* x, int64_t rows, int64_t cols, const int32_t* group_offsets_host,
                                  int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                  void* stream)
{
    return fp8_quant_dual_stash_opts(x, rows, cols, group_offsets_host, groups, q, scales, qT, scalesT, nullptr,
                                     stream);
}

fp8bs_status fp8_quant_dual_stash_opts(const void* x, int64_t rows, int64_t cols, const int32_t* group_offsets_host,
                                       int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                       const fp8bs_scale_opts* opts, void* stream)
{
    if (rows > 0 && (!q || !scales)) return FP8BS_ERR_ARG;
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, group_offsets_host, groups, qT, scalesT, q,
                          scales, opts, stream, true);
}

fp8bs_status fp8_requant_128x1_T_dev(int src_mode, const void* src, const float* src_scales, int64_t rows,
                                     int64_t cols, const int32_t* offsets_dev, int32_t groups, uint8_t* qT,
                                     float* scalesT, const fp8bs_scale_opts* opts, void* stream)
{
    if (!offsets_dev) return FP8BS_ERR_ARG;
    return requant_common(src_mode, src, src_scales, rows, cols, nullptr, groups, qT, scalesT, nullptr, nullptr,
                          opts, stream, false, nullptr, nullptr, nullptr, offsets_dev);
}

fp8bs_status fp8_quant_dual_dev(const void* x, int64_t rows, int64_t cols, const int32_t* offsets_dev,
                                int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                const fp8bs_scale_opts* opts, void* stream)
{
    if (!offsets_dev) return FP8BS_ERR_ARG;
    if (rows > 0 && (!q || !scales)) return FP8BS_ERR_ARG;
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, nullptr, groups, qT, scalesT, q, scales, opts,
                          stream, false, nullptr, nullptr, nullptr, offsets_dev);
}

fp8bs_status fp8_quant_dual_stash_dev(const void* x, int64_t rows, int64_t cols, const int32_t* offsets_dev,
                                      int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                      const fp8bs_scale_opts* opts, void* stream)
{
    if (!offsets_dev) return FP8BS_ERR_ARG;
    if (rows > 0 && (!q || !scales)) return FP8BS_ERR_ARG;
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, nullptr, groups, qT, scalesT, q, scales, opts,
                          stream, true, nullptr, nullptr, nullptr, offsets_dev);
}

fp8bs_status fp8_quant_dual_packed(const void* x, int64_t rows, int64_t cols, uint8_t* q, float* scales,
                                   uint8_t* qT, float* scalesT, uint8_t* q_atoms, uint8_t* qT_atoms,
                                   const fp8bs_scale_opts* opts, void* stream)
{
    if (!opts || opts->rule != FP8BS_SCALE_UE8M0) return FP8BS_ERR_ARG;
    if (cols % 128 != 0) return FP8BS_ERR_SHAPE;
    if (rows > 0 && (!q || !scales || !q_atoms || !qT_atoms)) return FP8BS_ERR_ARG;
    if ((q_atoms && !aligned16(q_atoms)) || (qT_atoms && !aligned16(qT_atoms))) return FP8BS_ERR_ALIGN;
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, nullptr, 0, qT, scalesT, q, scales, opts, stream,
                          false, nullptr, q_atoms, qT_atoms);
}

fp8bs_status fp8_quant_dual_stash_packed(const void* x, int64_t rows, int64_t cols, uint8_t* q, float* scales,
                                         uint8_t* qT, float* scalesT, uint8_t* q_atoms, uint8_t* qT_atoms,
                                         const fp8bs_scale_opts* opts, void* stream)
{
    if (!opts || opts->rule != FP8BS_SCALE_UE8M0) return FP8BS_ERR_ARG;
    if (cols % 128 != 0) return FP8BS_ERR_SHAPE;
    if (rows > 0 && (!q || !scales || !q_atoms || !qT_atoms)) return FP8BS_ERR_ARG;
    if ((q_atoms && !aligned16(q_atoms)) || (qT_atoms && !aligned16(qT_atoms))) return FP8BS_ERR_ALIGN;
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, nullptr, 0, qT, scalesT, q, scales, opts, stream,
                          true, nullptr, q_atoms, qT_atoms);
}

// The grouped forms: the tile kernel writes each block's exponent bytes into
// the atoms of the groups' tile layout (q: padded token tile rt, K-block ct)
// and of qT [cols x Mpad] (channel tile ct, token tile rt).
static fp8bs_status dual_packed_grouped(bool stash, const void* x, int64_t rows, int64_t cols,
                                        const int32_t* offsets_dev, const int32_t* offsets_host, int32_t groups,
                                        uint8_t* q, float* scales, uint8_t* qT, float* scalesT, uint8_t* q_atoms,
                                        uint8_t* qT_atoms, const fp8bs_scale_opts* opts, void* stream)
{
    if (!opts || opts->rule != FP8BS_SCALE_UE8M0) return FP8BS_ERR_ARG;
    if (cols % 128 != 0) return FP8BS_ERR_SHAPE;
    if ((offsets_dev == nullptr) == (offsets_host == nullptr) || groups < 1) return FP8BS_ERR_ARG;
    if (rows > 0 && (!q || !scales || !q_atoms || !qT_atoms)) return FP8BS_ERR_ARG;
    if ((q_atoms && !aligned16(q_atoms)) || (qT_atoms && !aligned16(qT_atoms))) return FP8BS_ERR_ALIGN;
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, offsets_host, groups, qT, scalesT, q, scales, opts,
                          stream, stash, nullptr, q_atoms, qT_atoms, offsets_dev);
}

fp8bs_status fp8_quant_dual_packed_grouped(const void* x, int64_t rows, int64_t cols, const int32_t* offsets_dev,
                                           const int32_t* offsets_host, int32_t groups, uint8_t* q, float* scales,
                                           uint8_t* qT, float* scalesT, uint8_t* q_atoms, uint8_t* qT_atoms,
                                           const fp8bs_scale_opts* opts, void* stream)
{
    return dual_packed_grouped(false, x, rows, cols, offsets_dev, offsets_host, groups, q, scales, qT, scalesT,
                               q_atoms, qT_atoms, opts, stream);
}

fp8bs_status fp8_quant_dual_stash_packed_grouped(const void* x, int64_t rows, int64_t cols,
                                                 const int32_t* offsets_dev, const int32_t* offsets_host,
                                                 int32_t groups, uint8_t* q, float* scales, uint8_t* qT,
                                                 float* scalesT, uint8_t* q_atoms, uint8_t* qT_atoms,
                                                 const fp8bs_scale_opts* opts, void* stream)
{
    return dual_packed_grouped(true, x, rows, cols, offsets_dev, offsets_host, groups, q, scales, qT, scalesT,
                               q_atoms, qT_atoms, opts, stream);
}

fp8bs_status fp8_quant_128x128_packed(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ldw,
                                      uint8_t* q, uint8_t* qT, float* scales, uint8_t* atoms_wT, uint8_t* atoms_w,
                                      const fp8bs_scale_opts* opts, void* stream)
{
    if (!opts || opts->rule != FP8BS_SCALE_UE8M0) return FP8BS_ERR_ARG;
    if (rows % 128 != 0 || cols % 128 != 0) return FP8BS_ERR_SHAPE;
    if (!atoms_wT || !atoms_w) return FP8BS_ERR_ARG;
    if (!aligned16(atoms_wT) || !aligned16(atoms_w)) return FP8BS_ERR_ALIGN;
    return quant_128x128_common(w, batch, rows, cols, ldw, q, qT, scales, opts, nullptr, stream, atoms_wT, atoms_w);
}

fp8bs_status fp8_requant_128x1_T_sr(int src_mode, const void* src, const float* src_scales, int64_t rows,
                                    int64_t cols, const int32_t* group_offsets_host, int32_t groups, uint8_t* qT,
                                    float* scalesT, uint64_t seed, uint32_t salt, const fp8bs_scale_opts* opts,
                                    void* stream)
{
    const SrParams sr{seed, salt};
    return requant_common(src_mode, src, src_scales, rows, cols, group_offsets_host, groups, qT, scalesT, nullptr,
                          nullptr, opts, stream, false, &sr);
}

fp8bs_status fp8_quant_dual_sr(const void* x, int64_t rows, int64_t cols, const int32_t* group_offsets_host,
                               int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT, uint64_t seed,
                               uint32_t salt, const fp8bs_scale_opts* opts, void* stream)
{
    if (rows > 0 && (!q || !scales)) return FP8BS_ERR_ARG;
    const SrParams sr{seed, salt};
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, group_offsets_host, groups, qT, scalesT, q,
                          scales, opts, stream, false, &sr);
}

fp8bs_status fp8_quant_dual_stash_sr(const void* x, int64_t rows, int64_t cols, const int32_t* group_offsets_host,
                                     int32_t groups, uint8_t* q, float* scales, uint8_t* qT, float* scalesT,
                                     uint64_t seed, uint32_t salt, const fp8bs_scale_opts* opts, void* stream)
{
    if (rows > 0 && (!q || !scales)) return FP8BS_ERR_ARG;
    const SrParams sr{seed, salt};
    return requant_common(FP8BS_SRC_BF16, x, nullptr, rows, cols, group_offsets_host, groups, qT, scalesT, q,
                          scales, opts, stream, true, &sr);
}

fp8bs_status fp8_block_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wqT,
                                  const float* sw, int64_t M, int64_t N, int64_t K, void* y,
                                  void* stream)
{
    if (M < 0 || N <= 0 || K <= 0) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || N % 128 != 0 || M > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!xq || !sx || !wqT || !sw || !y) return FP8BS_ERR_ARG;
    if (!aligned16(xq) || !aligned16(sx) || !aligned16(wqT) || !aligned16(sw) || !aligned16(y))
        return FP8BS_ERR_ALIGN;
    const int32_t off[2] = {0, static_cast<int32_t>(M)};
    return run_rowwise_gemm(FP8BS_OP_FPROP, Offsets{off, nullptr, 1, M}, xq, sx, wqT, sw, N, K, y, stream);
}

fp8bs_status fp8_block_gemm_fprop_wkn(const uint8_t* xq, const float* sx, const uint8_t* wq,
                                      const float* sw, int64_t M, int64_t N, int64_t K, void* y,
                                      void* stream)
{
    if (M < 0 || N <= 0 || K <= 0) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || N % 128 != 0 || M > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!xq || !sx || !wq || !sw || !y) return FP8BS_ERR_ARG;
    if (!aligned16(xq) || !aligned16(sx) || !aligned16(wq) || !aligned16(sw) || !aligned16(y))
        return FP8BS_ERR_ALIGN;
    const int32_t off[2] = {0, static_cast<int32_t>(M)};
    return run_rowwise_gemm(FP8BS_OP_FPROP_WKN, Offsets{off, nullptr, 1, M}, xq, sx, wq, sw, N, K, y, stream);
}

fp8bs_status fp8_block_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wq,
                                  const float* sw, int64_t M, int64_t N, int64_t K, void* dx,
                                  void* stream)
{
    if (M < 0 || N <= 0 || K <= 0) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || N % 128 != 0 || M > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!dyq || !sdy || !wq || !sw || !dx) return FP8BS_ERR_ARG;
    if (!aligned16(dyq) || !aligned16(sdy) || !aligned16(wq) || !aligned16(sw) || !aligned16(dx))
        return FP8BS_ERR_ALIGN;
    const int32_t off[2] = {0, static_cast<int32_t>(M)};
    return run_rowwise_gemm(FP8BS_OP_DGRAD, Offsets{off, nullptr, 1, M}, dyq, sdy, wq, sw, N, K, dx, stream);
}

int64_t fp8bs_mx_scale_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols < 0 || cols % 128 != 0) return -1;
    return (rows + 127) / 128 * (cols / 128) * 512;
}

fp8bs_status fp8_pack_ue8m0(const float* scales, int64_t rows, int64_t K, int32_t row_block,
                            int64_t row_stride, int64_t kb_stride, uint8_t* scale_atoms, void* stream)
{
    if (rows < 0 || K <= 0 || row_stride < 0 || kb_stride < 0) return FP8BS_ERR_ARG;
    if (row_block != 1 && row_block != 128) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || rows > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (rows == 0) return FP8BS_OK;
    if (!scales || !scale_atoms) return FP8BS_ERR_ARG;
    if (!aligned16(scale_atoms) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0) return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    return launch_status(launch_pack_ue8m0(scales, rows, K, row_block, row_stride, kb_stride, scale_atoms,
                                           st->status, st->num_sms, static_cast<cudaStream_t>(stream)));
}

fp8bs_status fp8_mx_quant_1x32(const void* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* scale_atoms,
                               void* stream)
{
    if (rows < 0 || cols <= 0) return FP8BS_ERR_ARG;
    if (cols % 128 != 0 || rows > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (rows == 0) return FP8BS_OK;
    if (!x || !q || !scale_atoms) return FP8BS_ERR_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scale_atoms)) return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    return launch_status(launch_mx_quant_1x32(static_cast<const uint16_t*>(x), rows, cols, q, scale_atoms,
                                              st->num_sms, static_cast<cudaStream_t>(stream)));
}

fp8bs_status fp8_mx_quant_1x32_T(const void* x, int64_t rows, int64_t cols, uint8_t* qT, uint8_t* scale_atoms,
                                 void* stream)
{
    if (rows < 0 || cols <= 0) return FP8BS_ERR_ARG;
    if (cols % 16 != 0 || rows > 0x7FFFFF00 || cols > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (rows == 0) return FP8BS_OK;
    if (!x || !qT || !scale_atoms) return FP8BS_ERR_ARG;
    if (!aligned16(x) || !aligned16(qT) || !aligned16(scale_atoms)) return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    return launch_status(launch_mx_quant_1x32_T(static_cast<const uint16_t*>(x), rows, cols, qT, scale_atoms,
                                                static_cast<cudaStream_t>(stream)));
}

fp8bs_status fp8_mx_gemm(const uint8_t* a, const uint8_t* a_scale_atoms, const uint8_t* b,
                         const uint8_t* b_scale_atoms, int64_t M, int64_t N, int64_t K, void* out, void* stream)
{
    return mx_gemm_common(a, a_scale_atoms, b, b_scale_atoms, M, N, K, static_cast<uint16_t*>(out), nullptr,
                          stream);
}

fp8bs_status fp8_mx_gemm_wkn(const uint8_t* a, const uint8_t* a_scale_atoms, const uint8_t* b,
                             const uint8_t* b_scale_atoms, int64_t M, int64_t N, int64_t K, void* out,
                             void* stream)
{
    return mx_gemm_common(a, a_scale_atoms, b, b_scale_atoms, M, N, K, static_cast<uint16_t*>(out), nullptr,
                          stream, true);
}

fp8bs_status fp8_mx_gemm_f32(const uint8_t* a, const uint8_t* a_scale_atoms, const uint8_t* b,
                             const uint8_t* b_scale_atoms, int64_t M, int64_t N, int64_t K, float* out,
                             void* stream)
{
    return mx_gemm_common(a, a_scale_atoms, b, b_scale_atoms, M, N, K, nullptr, out, stream);
}

fp8bs_status fp8_mx_gemm_grouped(int op, int32_t groups, const int32_t* offsets_dev, const int32_t* offsets_host,
                                 int64_t rows, const uint8_t* a, const uint8_t* a_scale_atoms, const uint8_t* b,
                                 const uint8_t* b_scale_atoms, int64_t N, int64_t K, void* out, void* stream)
{
    return mx_gemm_grouped(op, groups, offsets_dev, offsets_host, rows, a, a_scale_atoms, b, b_scale_atoms, N, K,
                           out, stream);
}

fp8bs_status fp8_pack_ue8m0_grouped(const float* scales, int64_t rows, int64_t K, int64_t kb_stride,
                                    int32_t groups, const int32_t* offsets_dev, const int32_t* offsets_host,
                                    uint8_t* scale_atoms, void* stream)
{
    if (rows < 0 || K <= 0 || kb_stride < 0 || groups < 1 || groups > kMaxGroups) return FP8BS_ERR_ARG;
    if ((offsets_dev == nullptr) == (offsets_host == nullptr)) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || rows > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (offsets_dev && (reinterpret_cast<uintptr_t>(offsets_dev) & 3u) != 0) return FP8BS_ERR_ALIGN;
    if (offsets_host && (!valid_offsets(offsets_host, groups) || offsets_host[groups] != rows))
        return FP8BS_ERR_ARG;
    const int64_t tiles = (offsets_dev ? padded_tokens_max(rows, groups) : padded_tokens(rows, offsets_host, groups)) / 128;
    if (tiles == 0) return FP8BS_OK;
    if (!scales || !scale_atoms) return FP8BS_ERR_ARG;
    if (!aligned16(scale_atoms) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0) return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    PackGroups pg;
    std::memset(&pg, 0, sizeof(pg));
    pg.num_groups = groups;
    pg.rows_total = static_cast<int>(rows);
    pg.off_dev = offsets_dev;
    if (offsets_host)
        for (int g = 0; g <= groups; ++g) pg.off[g] = offsets_host[g];
    return launch_status(launch_pack_ue8m0_grouped(scales, K, kb_stride, pg, tiles, scale_atoms, st->status,
                                                   st->num_sms, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace fp8bs {
namespace {

// The MX GEMM's output [rows x cols] (BF16 or FP32) as boxes of 32 rows x
// 64 bytes (32 BF16 or 16 FP32 columns), 64-byte swizzle.
bool make_mx_out_map(CUtensorMap* m, void* out, int64_t cols, int64_t rows, bool f32)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * (f32 ? 4 : 2)};
    const cuuint32_t box[2] = {f32 ? 16u : 32u, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    return g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// b_mn: B's codes are [K x N] (read MN-major) instead of [N x K].
fp8bs_status mx_gemm_common(const uint8_t* a, const uint8_t* a_scale_atoms, const uint8_t* b,
                            const uint8_t* b_scale_atoms, int64_t M, int64_t N, int64_t K, uint16_t* out_bf16,
                            float* out_f32, void* stream, bool b_mn)
{
    void* out = out_bf16 ? static_cast<void*>(out_bf16) : static_cast<void*>(out_f32);
    if (M < 0 || N <= 0 || K <= 0) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || N % 256 != 0 || M > 0x7FFFFF00 || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!a || !a_scale_atoms || !b || !b_scale_atoms || !out) return FP8BS_ERR_ARG;
    if (!aligned16(a) || !aligned16(a_scale_atoms) || !aligned16(b) || !aligned16(b_scale_atoms) ||
        !aligned16(out))
        return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    CUtensorMap ma, mb, mo;
    if (!make_map(&ma, a, K, M, K, kBM)) return FP8BS_ERR_ARG;
    if (b_mn ? !make_map(&mb, b, N, K, N, kBK) : !make_map(&mb, b, K, N, K, kBN)) return FP8BS_ERR_ARG;
    if (!make_mx_out_map(&mo, out, N, M, out_bf16 == nullptr)) return FP8BS_ERR_ARG;
    MxGroups grp;
    std::memset(&grp, 0, sizeof(grp));
    grp.layout = kMxDense;
    grp.b_mn = b_mn ? 1 : 0;
    grp.kb_atoms_a = grp.kb_atoms_b = static_cast<int>(K / 128);
    const int64_t tiles = ((M + kBM - 1) / kBM) * (N / kBN);
    return launch_status(launch_mx_gemm(ma, mb, &mo, a_scale_atoms, b_scale_atoms,
                                        static_cast<int>(M),
                                        static_cast<int>(N), static_cast<int>(K), out_bf16, out_f32,
                                        grp, tiles, g_wait_limit_ns, st->status, st->num_sms,
                                        static_cast<cudaStream_t>(stream)));
}

// Grouped MX GEMM (see fp8_mx_gemm_grouped in fp8bs.h).
fp8bs_status mx_gemm_grouped(int op, int32_t groups, const int32_t* offsets_dev, const int32_t* offsets_host,
                             int64_t rows, const uint8_t* a, const uint8_t* a_atoms, const uint8_t* b,
                             const uint8_t* b_atoms, int64_t N, int64_t K, void* out, void* stream)
{
    if (!rowwise_op(op) && op != FP8BS_OP_WGRAD) return FP8BS_ERR_ARG;
    if (groups < 1 || groups > kMaxGroups || rows < 0 || N <= 0 || K <= 0) return FP8BS_ERR_ARG;
    if ((offsets_dev == nullptr) == (offsets_host == nullptr)) return FP8BS_ERR_ARG;
    if (offsets_dev && (reinterpret_cast<uintptr_t>(offsets_dev) & 3u) != 0) return FP8BS_ERR_ALIGN;
    if (offsets_host && (!valid_offsets(offsets_host, groups) || offsets_host[groups] != rows))
        return FP8BS_ERR_ARG;
    // contraction and output width of one group
    const bool b_mn = op == FP8BS_OP_FPROP_WKN;
    const int64_t contr = op == FP8BS_OP_DGRAD ? N : K;
    const int64_t width = op == FP8BS_OP_DGRAD ? K : N;
    if (contr % 128 != 0 || width % 256 != 0 || rows > 0x7FFFFF00 || contr > 0x7FFFFFFF ||
        width * groups > 0x7FFFFFFF || N * groups > 0x7FFFFFFF || (b_mn && contr * groups > 0x7FFFFFFF))
        return FP8BS_ERR_SHAPE;
    if (!out) return FP8BS_ERR_ARG;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int64_t tpad = offsets_dev ? padded_tokens_max(rows, groups) : padded_tokens(rows, offsets_host, groups);
    if (op == FP8BS_OP_WGRAD && tpad == 0) {   // no tokens: every group's dW is zero
        if (!aligned16(out)) return FP8BS_ERR_ALIGN;
        return launch_status(cudaMemsetAsync(out, 0, sizeof(float) * groups * N * K, cs));
    }
    if (op != FP8BS_OP_WGRAD && rows == 0) return FP8BS_OK;
    if (!a || !a_atoms || !b || !b_atoms) return FP8BS_ERR_ARG;
    if (!aligned16(a) || !aligned16(a_atoms) || !aligned16(b) || !aligned16(b_atoms) || !aligned16(out))
        return FP8BS_ERR_ALIGN;
    MxGroups grp;
    std::memset(&grp, 0, sizeof(grp));
    grp.num_groups = groups;
    grp.off_dev = offsets_dev;
    if (offsets_host)
        for (int g = 0; g <= groups; ++g) grp.off[g] = offsets_host[g];
    grp.rows_total = static_cast<int>(rows);
    CUtensorMap ma, mb, mo;
    if (op == FP8BS_OP_WGRAD) {
        // a = dY^T [N x Tpad], b = X^T [K x Tpad]; out FP32 [groups x N x K]
        if (tpad > 0x7FFFFFFF) return FP8BS_ERR_SHAPE;
        if (!make_map(&ma, a, tpad, N, tpad, kBM) || !make_map(&mb, b, tpad, K, tpad, kBN) ||
            !make_mx_out_map(&mo, out, K, groups * N, true))
            return FP8BS_ERR_ARG;
        grp.layout = kMxTokenGroups;
        grp.out_rows = static_cast<int>(N);
        grp.kb_atoms_a = grp.kb_atoms_b = static_cast<int>(tpad / 128);
        grp.kb_cap = static_cast<int>(tpad / 128);
        const int64_t tiles = static_cast<int64_t>(groups) * (N / kBM) * (K / kBN);
        return launch_status(launch_mx_gemm(ma, mb, &mo, a_atoms, b_atoms, static_cast<int>(groups * N),
                                            static_cast<int>(K), 0, nullptr, static_cast<float*>(out), grp, tiles,
                                            g_wait_limit_ns, st->status, st->num_sms, cs));
    }
    // Fprop: a = Xq [rows x K], b = stacked WqT [groups x N x K] (or, for
    // FP8BS_OP_FPROP_WKN, stacked Wq [groups x K x N] read MN-major); Dgrad:
    // a = dYq [rows x N], b = stacked Wq [groups x K x N]; out BF16 [rows x width]
    if (!make_map(&ma, a, contr, rows, contr, kBM) ||
        (b_mn ? !make_map(&mb, b, width, contr * groups, width, kBK)
              : !make_map(&mb, b, contr, width * groups, contr, kBN)) ||
        !make_mx_out_map(&mo, out, width, rows, false))
        return FP8BS_ERR_ARG;
    grp.layout = kMxRowGroups;
    grp.b_mn = b_mn ? 1 : 0;
    grp.b_group_rows = static_cast<int>(width);
    grp.kb_atoms_a = grp.kb_atoms_b = static_cast<int>(contr / 128);
    const int64_t mtiles = tpad / 128;
    return launch_status(launch_mx_gemm(ma, mb, &mo, a_atoms, b_atoms, static_cast<int>(rows),
                                        static_cast<int>(width), static_cast<int>(contr),
                                        static_cast<uint16_t*>(out), nullptr, grp, mtiles * (width / kBN),
                                        g_wait_limit_ns, st->status, st->num_sms, cs));
}

}  // namespace
}  // namespace fp8bs

extern "C" {

size_t fp8bs_splitk_workspace_size(int op, int64_t M, int64_t N, int64_t K, int32_t splits)
{
    if (!rowwise_op(op) || M <= 0 || N <= 0 || K <= 0 || splits <= 1)
        return 0;
    const int64_t contr = op == FP8BS_OP_DGRAD ? N : K;
    const int64_t width = op == FP8BS_OP_DGRAD ? K : N;
    if (contr % 128 != 0) return 0;
    int used = 1, kps = 1;
    splitk_shape(contr / 128, splits, used, kps);
    if (used <= 1) return 0;
    return static_cast<size_t>(used) * static_cast<size_t>(splitk_tile_floats(M, width)) * sizeof(float);
}

int32_t fp8bs_splitk_default_splits(int op, int64_t M, int64_t N, int64_t K)
{
    if (!rowwise_op(op) || M <= 0 || N <= 0 || K <= 0) return 1;
    DeviceState* st = nullptr;
    if (device_state(&st) != FP8BS_OK) return 1;
    const int64_t contr = op == FP8BS_OP_DGRAD ? N : K;
    const int64_t width = op == FP8BS_OP_DGRAD ? K : N;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((width + kBN - 1) / kBN);
    const int64_t nkb = contr / kBK;
    // enough tiles to occupy the SMs, or too little K to be worth splitting
    if (tiles * 2 > st->num_sms || nkb < 16) return 1;
    int64_t sp = st->num_sms / tiles;
    if (sp > nkb / 4) sp = nkb / 4;   // at least four K-blocks per range
    return sp < 1 ? 1 : static_cast<int32_t>(sp);
}

fp8bs_status fp8_block_gemm_splitk(int op, const uint8_t* a, const float* sa, const uint8_t* b,
                                   const float* sb, int64_t M, int64_t N, int64_t K, int32_t splits,
                                   void* out, void* workspace, size_t workspace_bytes, void* stream)
{
    if (!rowwise_op(op)) return FP8BS_ERR_ARG;
    if (M < 0 || N <= 0 || K <= 0 || splits < 1) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || N % 128 != 0 || M > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!a || !sa || !b || !sb || !out) return FP8BS_ERR_ARG;
    if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(out))
        return FP8BS_ERR_ALIGN;
    const size_t need = fp8bs_splitk_workspace_size(op, M, N, K, splits);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return FP8BS_ERR_ARG;
        if (!aligned16(workspace)) return FP8BS_ERR_ALIGN;
    }
    const int32_t off[2] = {0, static_cast<int32_t>(M)};
    return run_rowwise_gemm(op, Offsets{off, nullptr, 1, M}, a, sa, b, sb, N, K, out, stream,
                            need > 0 ? splits : 1, static_cast<float*>(workspace));
}

fp8bs_status fp8_block_gemm_wgrad(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT,
                                  const float* sxT, int64_t T, int64_t N, int64_t K, float* dw,
                                  int accumulate, void* stream)
{
    if (T < 0 || N <= 0 || K <= 0) return FP8BS_ERR_ARG;
    if (T % 128 != 0 || N % 128 != 0 || K % 128 != 0) return FP8BS_ERR_SHAPE;
    if (!dw) return FP8BS_ERR_ARG;
    if (T > 0 && (!dyqT || !sdyT || !xqT || !sxT)) return FP8BS_ERR_ARG;
    if (!aligned16(dw) || (T > 0 && (!aligned16(dyqT) || !aligned16(sdyT) || !aligned16(xqT) ||
                                     !aligned16(sxT))))
        return FP8BS_ERR_ALIGN;
    const int32_t off[2] = {0, static_cast<int32_t>(T)};
    return run_wgrad(Offsets{off, nullptr, 1, T}, T, dyqT, sdyT, xqT, sxT, N, K, dw, accumulate, stream);
}

fp8bs_status fp8_block_gemm_grouped(int op, int32_t groups, const int32_t* offsets_dev,
                                    const int32_t* offsets_host, int64_t rows, const uint8_t* a,
                                    const float* sa, const uint8_t* b, const float* sb, int64_t N, int64_t K,
                                    void* out, int accumulate, void* stream)
{
    if (!rowwise_op(op) && op != FP8BS_OP_WGRAD) return FP8BS_ERR_ARG;
    if (groups < 1 || groups > kMaxGroups || rows < 0) return FP8BS_ERR_ARG;
    if ((offsets_dev == nullptr) == (offsets_host == nullptr)) return FP8BS_ERR_ARG;   // exactly one
    if (offsets_host && (!valid_offsets(offsets_host, groups) || offsets_host[groups] != rows)) return FP8BS_ERR_ARG;
    if (offsets_dev && (reinterpret_cast<uintptr_t>(offsets_dev) & 3u) != 0) return FP8BS_ERR_ALIGN;
    if (N <= 0 || K <= 0) return FP8BS_ERR_ARG;
    if (N % 128 != 0 || K % 128 != 0) return FP8BS_ERR_SHAPE;
    if (rows > 0x7FFFFF00) return FP8BS_ERR_SHAPE;
    if (!out) return FP8BS_ERR_ARG;
    const Offsets o{offsets_host, offsets_dev, groups, rows};
    if (op == FP8BS_OP_WGRAD) {
        const int64_t T = offsets_host ? padded_tokens(rows, offsets_host, groups) : padded_tokens_max(rows, groups);
        if (T > 0 && (!a || !sa || !b || !sb)) return FP8BS_ERR_ARG;
        if (!aligned16(out) || (T > 0 && (!aligned16(a) || !aligned16(sa) || !aligned16(b) ||
                                          !aligned16(sb))))
            return FP8BS_ERR_ALIGN;
        return run_wgrad(o, T, a, sa, b, sb, N, K, static_cast<float*>(out), accumulate, stream);
    }
    if (rows == 0) return FP8BS_OK;
    if (!a || !sa || !b || !sb) return FP8BS_ERR_ARG;
    if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(out))
        return FP8BS_ERR_ALIGN;
    return run_rowwise_gemm(op, o, a, sa, b, sb, N, K, out, stream);
}

int64_t fp8bs_padded_tokens_max(int64_t rows, int32_t groups)
{
    if (rows < 0 || groups < 0 || groups > kMaxGroups) return -1;
    return padded_tokens_max(rows, groups);
}

fp8bs_status fp8bs_device_status(int reset)
{
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    if (cudaDeviceSynchronize() != cudaSuccess) return FP8BS_ERR_LAUNCH;
    unsigned int v = 0;
    if (cudaMemcpy(&v, st->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    if (reset) {
        const unsigned int zero = 0;
        if (cudaMemcpy(st->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return FP8BS_ERR_LAUNCH;
        // a GEMM that gave up may have left stream-K partials unconsumed
        if (clear_stream_k_flags(st, nullptr, false) != cudaSuccess) return FP8BS_ERR_LAUNCH;
    }
    return static_cast<fp8bs_status>(v);
}

fp8bs_status fp8bs_last_device_status(void* stream, int reset)
{
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaMemcpyAsync(&v, st->status, sizeof(v), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    if (reset && cudaMemsetAsync(st->status, 0, sizeof(unsigned int), cs) != cudaSuccess) return FP8BS_ERR_LAUNCH;
    if (reset && clear_stream_k_flags(st, cs, true) != cudaSuccess) return FP8BS_ERR_LAUNCH;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return FP8BS_ERR_LAUNCH;
    return static_cast<fp8bs_status>(v);
}

fp8bs_status fp8bs_copy_device_status(unsigned int* dst, int reset, void* stream)
{
    if (!dst) return FP8BS_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(dst) & 3u) != 0) return FP8BS_ERR_ALIGN;
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dst, st->status, sizeof(unsigned int), cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    if (reset && cudaMemsetAsync(st->status, 0, sizeof(unsigned int), cs) != cudaSuccess) return FP8BS_ERR_LAUNCH;
    if (reset && clear_stream_k_flags(st, cs, true) != cudaSuccess) return FP8BS_ERR_LAUNCH;
    return FP8BS_OK;
}

void fp8bs_set_wait_limit_ns(uint64_t ns)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    g_wait_limit_ns = ns;
}

fp8bs_status fp8bs_selftest_wait_timeout(uint64_t limit_ns, void* stream)
{
    DeviceState* st = nullptr;
    fp8bs_status s = device_state(&st);
    if (s != FP8BS_OK) return s;
    return launch_status(launch_selftest_wait(st->status, limit_ns, static_cast<cudaStream_t>(stream)));
}

fp8bs_status fp8bs_selftest_gemm_timeout(const uint8_t* xq, const float* sx, const uint8_t* wqT, const float* sw,
                                         int64_t M, int64_t N, int64_t K, void* y, uint64_t limit_ns, void* stream)
{
    if (M <= 0 || N <= 0 || K <= 0 || limit_ns == 0) return FP8BS_ERR_ARG;
    if (K % 128 != 0 || N % 128 != 0 || M > 0x7FFFFF00 || K < 3 * 128) return FP8BS_ERR_SHAPE;
    if (!xq || !sx || !wqT || !sw || !y) return FP8BS_ERR_ARG;
    if (!aligned16(xq) || !aligned16(sx) || !aligned16(wqT) || !aligned16(sw) || !aligned16(y))
        return FP8BS_ERR_ALIGN;
    const int32_t off[2] = {0, static_cast<int32_t>(M)};
    return run_rowwise_gemm(FP8BS_OP_FPROP, Offsets{off, nullptr, 1, M}, xq, sx, wqT, sw, N, K, y, stream, 1, nullptr,
                            limit_ns);
}

}  // extern "C"
