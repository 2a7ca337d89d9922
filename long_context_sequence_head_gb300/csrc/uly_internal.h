// Internal declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "uly_ptx.cuh"

namespace uly {

// cuTensorMapEncodeTiled, resolved through the runtime once per process.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Device status word of the current device (2 x u32: flags, first site).
unsigned *device_status_ptr();
uint64_t wait_limit_ns();
int num_sms();

inline WaitCfg wait_cfg() { return WaitCfg{device_status_ptr(), wait_limit_ns()}; }

// ---------------------------------------------------------------- swap
// seq layout [P][B][N/P][H][d] <-> head layout [P][B][N][H/P][d].
cudaError_t launch_swap(bool to_head, const void *src, void *dst, int64_t B, int64_t N, int H, int d, int P,
                        int esize, cudaStream_t stream);

// ----------------------------------------------------------- attention
struct AttnShape {
    int64_t SB;      // num_shards * B (independent (shard, batch) problems)
    int64_t N;       // tokens
    int Hq, Hkv, d;  // per shard
    int causal;
    const int32_t *cu_dev;  // device cu_seqlens [num_docs+1] or nullptr
    int num_docs;
    float scale;      // softmax scale
};

cudaError_t launch_attn_fwd_f32(const AttnShape &s, const float *q, const float *k, const float *v, float *o,
                                float *lse, cudaStream_t stream);
cudaError_t launch_attn_bwd_f32(const AttnShape &s, const float *q, const float *k, const float *v,
                                const float *o, const float *lse, const float *dout, float *dq, float *dk,
                                float *dv, float *ws_D, cudaStream_t stream);

cudaError_t launch_attn_fwd_bf16(const AttnShape &s, const void *q, const void *k, const void *v, void *o,
                                 float *lse, cudaStream_t stream);

// bf16 backward scratch (fp32): lse2/D [SB][Hq][Npad], dq_acc [SB][Hq][Npad][d]
struct BwdScratch {
    float *lse2;
    float *D;
    float *dq_acc;
    int64_t Npad;
};
cudaError_t launch_attn_bwd_bf16(const AttnShape &s, const void *q, const void *k, const void *v, const void *o,
                                 const float *lse, const void *dout, void *dq, void *dk, void *dv,
                                 const BwdScratch &scr, cudaStream_t stream);

cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream);

}  // namespace uly
