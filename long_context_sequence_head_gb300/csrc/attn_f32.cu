// fp32 attention forward/backward over Ulysses head shards (SIMT, FFMA).
//
// The correctness path for fp32 inputs: TF32 tensor cores cannot meet a 1e-5
// relative error, so this path uses plain fp32 arithmetic with accurate
// exp/log.  One warp owns one query row (forward, dQ) or one key row (dK, dV);
// each lane holds d/32 consecutive-stride elements of the row and dot
// products are reduced with warp shuffles.
//
// Definitions (blog summary step 4 "Local Attention"; gradients as required
// for training): s_ij = scale <q_i, k_j>, lse_i = ln sum_j exp(s_ij),
// o_i = sum_j exp(s_ij - lse_i) v_j; D_i = <dO_i, O_i>, dS_ij = P_ij
// (<dO_i, v_j> - D_i), dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij
// q_i, dV_j = sum_i P_ij dO_i, with dK/dV summed over the GQA group.
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Document bounds of token i: [lo, hi).  Without documents [0, N).
__device__ __forceinline__ void doc_bounds(const AttnShape &s, int64_t i, int64_t &lo, int64_t &hi)
{
    lo = 0;
    hi = s.N;
    if (s.cu_dev == nullptr)
        return;
    int a = 0, b = s.num_docs;  // find k with cu[k] <= i < cu[k+1]
    while (b - a > 1) {
        const int m = (a + b) >> 1;
        if (static_cast<int64_t>(s.cu_dev[m]) <= i)
            a = m;
        else
            b = m;
    }
    lo = s.cu_dev[a];
    hi = s.cu_dev[a + 1];
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) fwd_f32_kernel(AttnShape s, const float *__restrict__ q,
                                                              const float *__restrict__ k,
                                                              const float *__restrict__ v, float *__restrict__ o,
                                                              float *__restrict__ lse)
{
    constexpr int E = D / 32;
    const int lane = lane_id();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kWarps + warp_id();
    const int h = blockIdx.y;
    const int64_t sb = blockIdx.z;
    if (i >= s.N)
        return;
    const int kvh = h / (s.Hq / s.Hkv);
    const int64_t qoff = s.L.off(s.N, sb, i, s.Hq, h, D);
    if (!ULY_IN_BOUNDS(s.status, qoff, D, s.q_elems, 0x01))
        return;
    const float *qi = q + qoff;
    float qr[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qr[e] = qi[lane + 32 * e];
        acc[e] = 0.f;
    }
    int64_t lo, hi;
    doc_bounds(s, i, lo, hi);
    if (s.causal)
        hi = i + 1;
    float m = -INFINITY, l = 0.f;
    for (int64_t j = lo; j < hi; ++j) {
        const int64_t koff = s.L.off(s.N, sb, j, s.Hkv, kvh, D);
        if (!ULY_IN_BOUNDS(s.status, koff, D, s.kv_elems, 0x02))
            break;
        const float *kj = k + koff;
        const float *vj = v + koff;
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e)
            part = fmaf(qr[e], kj[lane + 32 * e], part);
        const float sc = warp_sum(part) * s.scale;
        const float m_new = fmaxf(m, sc);
        const float alpha = expf(m - m_new);
        const float p = expf(sc - m_new);
        l = l * alpha + p;
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[e] = fmaf(p, vj[lane + 32 * e], acc[e] * alpha);
        m = m_new;
    }
    float *oi = o + qoff;
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e)
        oi[lane + 32 * e] = acc[e] * inv;
    const int64_t li = (sb * s.Hq + h) * s.N + i;
    if (lane == 0 && ULY_IN_BOUNDS(s.status, li, 1, s.lse_elems, 0x03))
        lse[li] = m + logf(l);
}

// D_i = <dO_i, O_i>, stored [SB][Hq][N]
template <int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_pre_f32_kernel(AttnShape s, const float *__restrict__ o,
                                                                  const float *__restrict__ dout,
                                                                  float *__restrict__ Dv)
{
    constexpr int E = D / 32;
    const int lane = lane_id();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kWarps + warp_id();
    const int h = blockIdx.y;
    const int64_t sb = blockIdx.z;
    if (i >= s.N)
        return;
    const int64_t off = s.L.off(s.N, sb, i, s.Hq, h, D);
    const int64_t li = (sb * s.Hq + h) * s.N + i;
    if (!ULY_IN_BOUNDS(s.status, off, D, s.q_elems, 0x04) || !ULY_IN_BOUNDS(s.status, li, 1, s.lse_elems, 0x05))
        return;
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
        part = fmaf(dout[off + lane + 32 * e], o[off + lane + 32 * e], part);
    part = warp_sum(part);
    if (lane == 0)
        Dv[li] = part;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_f32_kernel(AttnShape s, const float *__restrict__ q,
                                                                 const float *__restrict__ k,
                                                                 const float *__restrict__ v,
                                                                 const float *__restrict__ lse,
                                                                 const float *__restrict__ dout,
                                                                 const float *__restrict__ Dv,
                                                                 float *__restrict__ dq)
{
    constexpr int E = D / 32;
    const int lane = lane_id();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kWarps + warp_id();
    const int h = blockIdx.y;
    const int64_t sb = blockIdx.z;
    if (i >= s.N)
        return;
    const int kvh = h / (s.Hq / s.Hkv);
    const int64_t off = s.L.off(s.N, sb, i, s.Hq, h, D);
    if (!ULY_IN_BOUNDS(s.status, off, D, s.q_elems, 0x06) ||
        !ULY_IN_BOUNDS(s.status, (sb * s.Hq + h) * s.N + i, 1, s.lse_elems, 0x07))
        return;
    float qr[E], dor[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qr[e] = q[off + lane + 32 * e];
        dor[e] = dout[off + lane + 32 * e];
        acc[e] = 0.f;
    }
    const float lse_i = lse[(sb * s.Hq + h) * s.N + i];
    const float D_i = Dv[(sb * s.Hq + h) * s.N + i];
    int64_t lo, hi;
    doc_bounds(s, i, lo, hi);
    if (s.causal)
        hi = i + 1;
    for (int64_t j = lo; j < hi; ++j) {
        const int64_t koff = s.L.off(s.N, sb, j, s.Hkv, kvh, D);
        if (!ULY_IN_BOUNDS(s.status, koff, D, s.kv_elems, 0x08))
            break;
        const float *kj = k + koff;
        const float *vj = v + koff;
        float ps = 0.f, pd = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            ps = fmaf(qr[e], kj[lane + 32 * e], ps);
            pd = fmaf(dor[e], vj[lane + 32 * e], pd);
        }
        const float p = expf(warp_sum(ps) * s.scale - lse_i);
        const float dS = p * (warp_sum(pd) - D_i);
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[e] = fmaf(dS, kj[lane + 32 * e], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
        dq[off + lane + 32 * e] = acc[e] * s.scale;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkv_f32_kernel(AttnShape s, const float *__restrict__ q,
                                                                  const float *__restrict__ k,
                                                                  const float *__restrict__ v,
                                                                  const float *__restrict__ lse,
                                                                  const float *__restrict__ dout,
                                                                  const float *__restrict__ Dv,
                                                                  float *__restrict__ dk, float *__restrict__ dv)
{
    constexpr int E = D / 32;
    const int lane = lane_id();
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kWarps + warp_id();
    const int kvh = blockIdx.y;
    const int64_t sb = blockIdx.z;
    if (j >= s.N)
        return;
    const int G = s.Hq / s.Hkv;
    const int64_t off = s.L.off(s.N, sb, j, s.Hkv, kvh, D);
    if (!ULY_IN_BOUNDS(s.status, off, D, s.kv_elems, 0x09))
        return;
    float kr[E], vr[E], ak[E], av[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        kr[e] = k[off + lane + 32 * e];
        vr[e] = v[off + lane + 32 * e];
        ak[e] = 0.f;
        av[e] = 0.f;
    }
    int64_t lo, hi;
    doc_bounds(s, j, lo, hi);
    if (s.causal)
        lo = j;  // rows i >= j attend to key j
    for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
        for (int64_t i = lo; i < hi; ++i) {
            const int64_t qo = s.L.off(s.N, sb, i, s.Hq, h, D);
            if (!ULY_IN_BOUNDS(s.status, qo, D, s.q_elems, 0x0a) ||
                !ULY_IN_BOUNDS(s.status, (sb * s.Hq + h) * s.N + i, 1, s.lse_elems, 0x0b))
                break;
            float ps = 0.f, pd = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ps = fmaf(q[qo + lane + 32 * e], kr[e], ps);
                pd = fmaf(dout[qo + lane + 32 * e], vr[e], pd);
            }
            const float lse_i = lse[(sb * s.Hq + h) * s.N + i];
            const float D_i = Dv[(sb * s.Hq + h) * s.N + i];
            const float p = expf(warp_sum(ps) * s.scale - lse_i);
            const float dS = p * (warp_sum(pd) - D_i);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ak[e] = fmaf(dS, q[qo + lane + 32 * e], ak[e]);
                av[e] = fmaf(p, dout[qo + lane + 32 * e], av[e]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        dk[off + lane + 32 * e] = ak[e] * s.scale;
        dv[off + lane + 32 * e] = av[e];
    }
}

template <int D>
cudaError_t fwd_f32(const AttnShape &s, const float *q, const float *k, const float *v, float *o, float *lse,
                    cudaStream_t st)
{
    dim3 grid(static_cast<unsigned>((s.N + kWarps - 1) / kWarps), s.Hq, static_cast<unsigned>(s.SB));
    fwd_f32_kernel<D><<<grid, kWarps * 32, 0, st>>>(s, q, k, v, o, lse);
    return cudaGetLastError();
}

template <int D>
cudaError_t bwd_f32(const AttnShape &s, const float *q, const float *k, const float *v, const float *o,
                    const float *lse, const float *dout, float *dq, float *dk, float *dv, float *Dv,
                    cudaStream_t st)
{
    const unsigned nb = static_cast<unsigned>((s.N + kWarps - 1) / kWarps);
    bwd_pre_f32_kernel<D><<<dim3(nb, s.Hq, static_cast<unsigned>(s.SB)), kWarps * 32, 0, st>>>(s, o, dout, Dv);
    bwd_dq_f32_kernel<D><<<dim3(nb, s.Hq, static_cast<unsigned>(s.SB)), kWarps * 32, 0, st>>>(s, q, k, v, lse,
                                                                                              dout, Dv, dq);
    bwd_dkv_f32_kernel<D><<<dim3(nb, s.Hkv, static_cast<unsigned>(s.SB)), kWarps * 32, 0, st>>>(s, q, k, v, lse,
                                                                                                dout, Dv, dk, dv);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_f32(const AttnShape &s, const float *q, const float *k, const float *v, float *o,
                                float *lse, cudaStream_t stream)
{
    if (s.d == 64)
        return fwd_f32<64>(s, q, k, v, o, lse, stream);
    if (s.d == 128)
        return fwd_f32<128>(s, q, k, v, o, lse, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_bwd_f32(const AttnShape &s, const float *q, const float *k, const float *v,
                                const float *o, const float *lse, const float *dout, float *dq, float *dk,
                                float *dv, float *ws_D, cudaStream_t stream)
{
    if (s.d == 64)
        return bwd_f32<64>(s, q, k, v, o, lse, dout, dq, dk, dv, ws_D, stream);
    if (s.d == 128)
        return bwd_f32<128>(s, q, k, v, o, lse, dout, dq, dk, dv, ws_D, stream);
    return cudaErrorInvalidValue;
}

}  // namespace uly
