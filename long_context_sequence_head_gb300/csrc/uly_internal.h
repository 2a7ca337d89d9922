// Internal declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "uly_ptx.cuh"

namespace uly {

// cuTensorMapEncodeTiled, resolved through the runtime once per process.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// An NVTX push/pop range around one call of the C ABI, named after the call,
// so that profilers can attribute kernels to it.  NVTX 3 is header-only: with
// no tool attached a push or pop is a check of a null function pointer.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define ULY_NVTX_RANGE() const ::uly::NvtxRange uly_nvtx_range_(__func__)

// Device status word of the current device (2 x u32: flags, first site).
unsigned *device_status_ptr();
uint64_t wait_limit_ns();
int num_sms();

// Rows [lo, hi) of the document holding token i (the whole sequence without documents).
inline void doc_range_host(const int32_t *cu, int num_docs, int64_t N, int64_t i, int64_t &lo, int64_t &hi)
{
    lo = 0;
    hi = N;
    if (cu == nullptr || num_docs <= 0)
        return;
    int a = 0, b = num_docs;
    while (b - a > 1) {
        const int m = (a + b) >> 1;
        if (static_cast<int64_t>(cu[m]) <= i)
            a = m;
        else
            b = m;
    }
    lo = cu[a];
    hi = cu[a + 1];
}

// The 128-row tiles of a packed-document sequence in the order the bf16
// kernels walk them, longest walk first, so that no long walk is left to run
// on alone at the end of a launch (with documents the walk length follows a
// tile's place in its document, not its index).  Forward (bwd = false): query
// tiles, walk = the key tiles their rows may attend to, ties with the later
// tile first.  Backward: key tiles, walk = the query tiles that may attend to
// them, ties with the earlier tile first.  out: ceil(N/128) entries.
inline void tile_order_host(bool bwd, int64_t N, int causal, const int32_t *cu, int num_docs, int32_t *out)
{
    const int n = static_cast<int>((N + 127) / 128);
    std::vector<int64_t> walk(n);
    for (int t = 0; t < n; ++t) {
        const int64_t a = static_cast<int64_t>(t) * 128, b = std::min<int64_t>(a + 127, N - 1);
        int64_t lo_a, hi_a, lo_b, hi_b;
        doc_range_host(cu, num_docs, N, a, lo_a, hi_a);
        doc_range_host(cu, num_docs, N, b, lo_b, hi_b);
        const int64_t lo = (bwd && causal) ? a : lo_a;
        const int64_t hi = (!bwd && causal) ? b + 1 : hi_b;
        walk[t] = (hi - 1) / 128 - lo / 128 + 1;
        out[t] = bwd ? t : n - 1 - t;
    }
    std::stable_sort(out, out + n, [&](int32_t x, int32_t y) { return walk[x] > walk[y]; });
}

// Problems interleaved per group of the grid: the fewest that make a group's
// work per SM at least 1.5 times the longest single work unit, so that the
// last group's longest units do not run on alone at the end of the launch.
inline int group_for(int64_t work_per_problem, int64_t longest_unit, int64_t nprob)
{
    if (work_per_problem <= 0)
        return 1;
    int64_t g = (3 * longest_unit * num_sms() + 2 * work_per_problem - 1) / (2 * work_per_problem);
    if (g > nprob)
        g = nprob;
    return g < 1 ? 1 : static_cast<int>(g);
}

inline WaitCfg wait_cfg() { return WaitCfg{device_status_ptr(), wait_limit_ns()}; }

// ---------------------------------------------------------------- swap
// seq layout [P][B][N/P][H][d] <-> head layout [P][B][N][H/P][d].
cudaError_t launch_swap(bool to_head, const void *src, void *dst, int64_t B, int64_t N, int H, int d, int P,
                        int esize, cudaStream_t stream);

// Up to kSwapMaxBatch tensors with common B, N, d, P and element size in one
// launch; each has its own head count and direction.
constexpr int kSwapMaxBatch = 4;
struct SwapDesc {
    const void *src;
    void *dst;
    int H;
    int to_head;
};
cudaError_t launch_swap_batch(const SwapDesc *descs, int n, int64_t B, int64_t N, int d, int P, int esize,
                              cudaStream_t stream);

// ----------------------------------------------------------- attention
// Where the rows of an attention tensor live.
//   head layout (seq == 0): [S][B][N][H][d], shard-major, what the swap writes;
//   seq layout  (seq == 1): [P][B][N/P][P*H][d], the sequence-sharded buffer
//     before the swap: head shard r of local head h is global head r*H + h,
//     token n sits in sequence shard n / (N/P) at position n % (N/P).
// Row (sb, n, h) with sb = shard*B + batch.
struct RowLayout {
    int seq;
    int B;
    int64_t Np;  // N / P (seq layout)
    int P;       // head shards == sequence shards (seq layout)

    __host__ __device__ int64_t off(int64_t N, int64_t sb, int64_t n, int H, int h, int d) const
    {
        if (!seq)
            return ((sb * N + n) * H + h) * static_cast<int64_t>(d);
        const int64_t r = sb / B, b = sb % B, s = n / Np, t = n % Np;
        return (((s * B + b) * Np + t) * (static_cast<int64_t>(H) * P) + r * H + h) * static_cast<int64_t>(d);
    }
    // coordinates {head, token, batch, outer} of the 5-D tensor map of this
    // layout for a tile of rows starting at token n0 (which never straddles a
    // sequence shard in the seq layout)
    __host__ __device__ void tile(int64_t sb, int64_t n0, int H, int h, int &c1, int &c2, int &c3, int &c4) const
    {
        const int r = static_cast<int>(sb / B), b = static_cast<int>(sb % B);
        c3 = b;
        if (!seq) {
            c1 = h;
            c2 = static_cast<int>(n0);
            c4 = r;
        } else {
            c1 = r * H + h;
            c2 = static_cast<int>(n0 % Np);
            c4 = static_cast<int>(n0 / Np);
        }
    }
};

struct AttnShape {
    int64_t SB;      // num_shards * B (independent (shard, batch) problems)
    int64_t N;       // tokens
    int Hq, Hkv, d;  // per shard
    int causal;
    const int32_t *cu_dev;  // device cu_seqlens [num_docs+1] or nullptr
    const int32_t *cu_host; // the same on the host (valid during the call) or nullptr
    int32_t *order_dev;     // with documents: device room for a 128-row tile order [ceil(N/128)], else nullptr
    int num_docs;
    float scale;      // softmax scale
    RowLayout L;     // where q/k/v/o/dout/dq/dk/dv rows live
    // buffer extents in elements, for the bounds checks of debug builds
    int64_t q_elems;    // q, o, dout, dq
    int64_t kv_elems;   // k, v, dk, dv
    int64_t lse_elems;  // lse (and the per-row fp32 scratch)
    unsigned *status;   // device status word
};

// 5-D bf16 tensor map {d, H, T, B, outer} over a row-major
// [outer][B][T][H][d] buffer, box {64, 1, 128, 1, 1}, 128-byte swizzle.
CUresult make_rows_map_bf16(CUtensorMap *map, const void *base, const AttnShape &s, int H);

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

// ------------------------------------------------------- sharded loss
cudaError_t launch_sharded_ce(const void *logits, const int64_t *labels, void *dlogits, float *shard_loss,
                              int64_t *shard_good, float *total, int64_t B, int64_t N, int64_t V, int P, int esize,
                              void *workspace, cudaStream_t stream);
size_t sharded_ce_workspace(int64_t B, int64_t N, int P);

}  // namespace uly

#include <ulysses.h>

namespace uly {

// Validated attention calls (ulysses_api.cu), shared by the C entry points
// and the ring-attention orchestration.
uly_status attn_fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t N,
                         int32_t Hq_local, int32_t Hkv_local, int32_t d, int32_t num_shards, int32_t causal,
                         const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale, uly_dtype dtype,
                         void *workspace, size_t workspace_bytes, void *stream, RowLayout L);
uly_status attn_bwd_impl(const void *q, const void *k, const void *v, const void *o, const float *lse,
                         const void *dout, void *dq, void *dk, void *dv, int64_t B, int64_t N, int32_t Hq_local,
                         int32_t Hkv_local, int32_t d, int32_t num_shards, int32_t causal,
                         const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale, uly_dtype dtype,
                         void *workspace, size_t workspace_bytes, void *stream, RowLayout L);
RowLayout head_rows(int64_t B, int64_t N, int32_t S);

// ring attention (ring.cu)
size_t ring_workspace_size(int64_t B, int64_t N, int Hq, int Hkv, int d, int P, bool bwd, uly_dtype dt);
uly_status ring_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t N, int Hq,
                    int Hkv, int d, int P, int causal, float scale, uly_dtype dt, void *workspace, size_t ws_bytes,
                    cudaStream_t s);
uly_status ring_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
                    void *dq, void *dk, void *dv, int64_t B, int64_t N, int Hq, int Hkv, int d, int P, int causal,
                    float scale, uly_dtype dt, void *workspace, size_t ws_bytes, cudaStream_t s);

}  // namespace uly
