// fa_noalloc.cu -- split-KV forward for callers that cannot allocate device
// memory.
//
// fa_fwd_splitkv needs a workspace for its per-range partial results, and
// the caller normally provides it.  Some callers cannot call cudaMalloc or an
// allocator at all, for instance:
//   - code running inside a framework's allocation-free region;
//   - plugins that are handed only input and output buffers;
//   - real-time loops where an allocation could block or fragment memory.
// For them, this file owns a fixed scratch array in device global memory, and
// fa_fwd_splitkv_noalloc uses it as that workspace.
//
// In host code the name of a __device__ array stands for a host-side shadow,
// not a device address, so the address the kernels get comes from
// cudaGetSymbolAddress.  This is done once per device, with that device
// current, on the first call made on it.
#include "fa.h"

#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

// The scratch every call shares.  A device holds it from the time this
// library's code is loaded there (under lazy module loading, the first call of
// the entry point at the latest) until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device and kept for the life of the process (a cudaDeviceReset, which may
// move the array, is not followed: the header says so).
fa_status scratch_on_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V, void *O,
                                            float *LSE, int B, int H, int N, int D, int causal,
                                            float scale, const int32_t *kv_len, int num_splits,
                                            void *stream)
{
    if (B < 0 || H < 0 || N < 0 || D <= 0 || num_splits < 0 || num_splits > FA_MAX_SPLITS)
        return FA_ERR_INVALID_ARG;
    if ((long long)B * H * N == 0) return FA_OK;
    if (num_splits == 0) num_splits = fa_fwd_splitkv_auto_splits(B, H, N, D);
    const size_t need = fa_fwd_splitkv_workspace_bytes(B, H, N, D, num_splits);
    if (need == 0 || need > (size_t)FA_NOALLOC_SCRATCH_BYTES)
        return FA_ERR_UNSUPPORTED;   // the problem needs more scratch than the fixed array holds
    void *scratch = nullptr;
    const fa_status st = scratch_on_current_device(&scratch);
    if (st != FA_OK) return st;
    // The partial results are fully rewritten before the merge reads them, so
    // whatever an earlier call left in the scratch does not matter.
    return fa_fwd_splitkv(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, num_splits, scratch,
                          (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}
