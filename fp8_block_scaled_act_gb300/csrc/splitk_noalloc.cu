// splitk_noalloc.cu -- split-K Fprop / Dgrad whose workspace is a fixed
// array compiled into the library, for callers that must not allocate.
//
// fp8_block_gemm_splitk takes its fp32 range sums in a caller workspace.
// Some callers cannot provide one: code that runs where allocating device
// memory is not allowed or not wanted (an allocator-free runtime, a hot loop
// that must not call cudaMalloc because it can synchronize the device, a
// plugin that owns no memory pool). This entry point uses the static
// scratch array below instead and makes no allocation of any kind.
//
// Set-up: the first call on each device (with that device current) looks up
// the array's device address with cudaGetSymbolAddress and keeps it; later
// calls on that device reuse it. With lazy module loading that lookup is also
// when the library's module, and with it the array, is loaded onto the
// device, so make that first call before any stream capture begins. The
// array is device memory that every process loading the library holds on
// each device where the module is loaded, whether or not it calls this entry
// point. Every call must be made with the device of `stream` current (the
// call checks this and returns FP8BS_ERR_ARG otherwise). The kept address
// does not survive cudaDeviceReset: a process that resets a device must not
// call this entry point on it afterwards.
//
// Limits and sharing: the scratch holds kScratchBytes (32 MiB); a request
// whose fp8bs_splitk_workspace_size exceeds that is rejected with
// FP8BS_ERR_SHAPE before any work. One array serves every call in the
// process on a device, so two calls whose executions overlap (issued on
// different streams without ordering, or from several host threads) race on
// it and both results are undefined; serialize them (one stream, or events).
// Nothing in the scratch needs to start at zero: every element the
// reduction reads was written by the same call's GEMM.
#include <cuda_runtime.h>

#include <mutex>

#include "fp8bs.h"

namespace {

constexpr size_t kScratchBytes = FP8BS_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) unsigned char g_splitk_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
fp8bs_status scratch_pointer(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8BS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_splitk_scratch) != cudaSuccess || !ptr) return FP8BS_ERR_UNSUPPORTED;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return FP8BS_OK;
}

}  // namespace

extern "C" {

fp8bs_status fp8_block_gemm_splitk_noalloc(int op, const uint8_t* a, const float* sa, const uint8_t* b,
                                           const float* sb, int64_t M, int64_t N, int64_t K, int32_t splits,
                                           void* out, void* stream)
{
    if (op != FP8BS_OP_FPROP && op != FP8BS_OP_FPROP_WKN && op != FP8BS_OP_DGRAD) return FP8BS_ERR_ARG;
    if (M < 0 || N <= 0 || K <= 0 || splits < 1) return FP8BS_ERR_ARG;
    if (fp8bs_splitk_workspace_size(op, M, N, K, splits) > kScratchBytes) return FP8BS_ERR_SHAPE;
    if (stream) {
        // the scratch address is the current device's: the stream must belong to it
        int cur = 0, sdev = 0;
        if (cudaGetDevice(&cur) != cudaSuccess ||
            cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
            return FP8BS_ERR_ARG;
        if (sdev != cur) return FP8BS_ERR_ARG;
    }
    void* scratch = nullptr;
    const fp8bs_status s = scratch_pointer(&scratch);
    if (s != FP8BS_OK) return s;
    return fp8_block_gemm_splitk(op, a, sa, b, sb, M, N, K, splits, out, scratch, kScratchBytes, stream);
}

}  // extern "C"
