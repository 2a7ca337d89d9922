// ulysses_attn_bwd_noalloc: the attention backward for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a
// custom allocator's own callbacks, in a process whose memory pool is fixed
// up front and may not grow, in a plugin given only the tensors it works on,
// or on a real-time path that must not take the allocator's locks.  Such a
// caller can pass its inputs and outputs but cannot provide the fp32 scratch
// ulysses_attn_bwd takes as `workspace`.
//
// Here that scratch is one file-scope device array of a fixed size.  Any GPU
// that loads this part of the library holds it until the process exits.  Its
// device address is looked up once per device with cudaGetSymbolAddress (the
// array's name in host code is only a host-side stand-in).  The runtime loads
// device code lazily, so that lookup, on the first call on each device, is
// what loads this module and makes the driver reserve the array: a caller
// that cannot afford the reservation inside its restricted context makes its
// first call on each device outside it, and before any stream capture.  The
// address is the current device's, so the stream and every pointer must
// belong to the current device.  Every call shares the array and it keeps the
// previous call's contents; the backward rewrites or clears every byte it
// reads before reading it.  Calls that overlap on the GPU (different streams,
// or threads without ordering) race on the array and must not be issued.
#include <ulysses.h>

#include <mutex>

#include "uly_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, or nullptr.
void *noalloc_scratch()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess)
            return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" {

uly_status ulysses_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                                    const void *dout, void *dq, void *dk, void *dv, int64_t B, int64_t N,
                                    int32_t Hq_local, int32_t Hkv_local, int32_t d, int32_t num_shards,
                                    int32_t causal, const int32_t *cu_seqlens_host, int32_t num_docs,
                                    float softmax_scale, uly_dtype dtype, void *stream)
{
    ULY_NVTX_RANGE();
    const size_t need = ulysses_attn_workspace_size(B, N, Hq_local, Hkv_local, d, num_shards,
                                                    cu_seqlens_host ? num_docs : 0, 1, dtype);
    if (need == 0)
        return ULY_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes)
        return ULY_ERR_SCRATCH_LIMIT;
    void *scratch = noalloc_scratch();
    if (scratch == nullptr)
        return ULY_ERR_CUDA;
    return ulysses_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, N, Hq_local, Hkv_local, d, num_shards, causal,
                            cu_seqlens_host, num_docs, softmax_scale, dtype, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
