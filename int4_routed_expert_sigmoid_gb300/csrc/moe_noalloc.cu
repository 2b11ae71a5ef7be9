// moe_noalloc.cu -- moe_expert_ffn_int4_noalloc: the expert FFN with its scratch
// in memory this library reserves when it is loaded, for callers that cannot
// allocate device memory themselves.
//
// Who needs it: a caller that runs inside a host framework which owns every
// byte of device memory and forbids other allocations, or a caller on a
// latency-critical path that cannot afford cudaMalloc/cudaFree (both may
// synchronise the device).  Such a caller can still pass its inputs and
// outputs, but cannot provide the FFN's workspace.
//
// How: the workspace is a file-scope __device__ array of kNoAllocScratchBytes
// (8 MiB) that every GPU which loads the library holds until the process
// exits.  In host code the array's name is only a host-side stand-in, so the
// device address is looked up once per device (cudaGetSymbolAddress, with that
// device current) on the first call made on that device, and cached.  That
// first call on a device should come before any stream capture.  Nothing here
// calls cudaMalloc, cudaFree or an allocating library routine.
//
// Sharing: every call on a device uses the same array, which keeps the last
// call's contents.  The FFN fully writes its scratch before reading it, so
// nothing has to start at zero.  Calls that overlap on the GPU (different
// streams, or different host threads without ordering) race on the array.
#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_ffn_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_ffn_scratch on the current device (looked up once).
int scratch_on_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ffn_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_expert_ffn_int4_noalloc(const float *x, const moe_layer_int4 *w,
                                           const int32_t *offsets, const int32_t *sorted_pair,
                                           const int32_t *uniq, const int32_t *n_uniq, int T, int k,
                                           int mode, float *y_pair, float *y_shared, int32_t *err,
                                           void *stream)
{
    if (w == nullptr || T < 1 || k < 1)
        return MOE_ERR_INVALID_ARG;
    const size_t need = moe_ffn_workspace_bytes(T, k, w->d, w->f, mode);
    if (need == 0)
        return MOE_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes)
        return MOE_ERR_WORKSPACE;   // this batch needs more scratch than the reserved array
    void *scratch = nullptr;
    const int rc = scratch_on_current_device(&scratch);
    if (rc != MOE_OK)
        return rc;
    return moe_expert_ffn_int4(x, w, offsets, sorted_pair, uniq, n_uniq, T, k, mode, y_pair,
                               y_shared, scratch, kNoAllocScratchBytes, err, stream);
}
