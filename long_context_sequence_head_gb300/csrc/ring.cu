// Ring attention over P virtual ranks, on the attention kernels of this
// library (the pages' alternative to Ulysses: "Sequence Parallelism for
// Long-Context AI Training", "Advanced Scaling: Ring Attention and Ulysses";
// the blog summary's "Comparing Ulysses and Ring Attention" table).
//
// Rank r holds chunk r = tokens [r*N/P, (r+1)*N/P) of Q, K, V for ALL heads
// (no head sharding).  In P steps every query chunk meets every key chunk:
// step k pairs query chunk r with key chunk (r - k) mod P.  Under a causal
// mask step 0 is chunk r against itself (causal inside the chunk) and the
// later steps only keep r >= k (earlier key chunks, unmasked); the
// non-causal case also runs the wrapped pairs r < k.
//
// On one GPU the chunks are the P contiguous shards of the sequence-sharded
// buffer, so "receiving chunk s" is only a pointer offset: each step is one
// launch of the attention kernel over the chunk pairs of that step, with the
// chunks of the query side and the key side addressed from different bases.
//
// Forward: partial (o, lse) per step, folded into the running result by
//   m = max(lse_a, lse_b), w_x = exp(lse_x - m),
//   o = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = m + ln(w_a + w_b).
// Backward: each chunk pair's gradients computed with the FINAL o and lse
// (P_ij = exp(s_ij - lse_i) and D_i = <dO_i, O_i> are global), summed in
// fp32: dQ of chunk r over its key chunks, dK/dV of chunk s over the query
// chunks that saw it.
#include "uly_internal.h"

namespace uly {
namespace {

template <typename T>
__device__ __forceinline__ float ld_f(const T *p);
template <>
__device__ __forceinline__ float ld_f<uint16_t>(const uint16_t *p)
{
    return __uint_as_float(static_cast<uint32_t>(*p) << 16);
}
template <>
__device__ __forceinline__ float ld_f<float>(const float *p)
{
    return *p;
}
template <typename T>
__device__ __forceinline__ T to_t(float v);
template <>
__device__ __forceinline__ uint16_t to_t<uint16_t>(float v)
{
    return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}
template <>
__device__ __forceinline__ float to_t<float>(float v)
{
    return v;
}

// Fold a partial (o_b, lse_b) into the running (o_a, lse_a), one warp per
// (chunk, batch, token, head) row; rows of `nchunks` consecutive chunks.
template <typename T>
__global__ void merge_kernel(T *__restrict__ o_a, float *__restrict__ lse_a, const T *__restrict__ o_b,
                             const float *__restrict__ lse_b, int64_t nchunks, int64_t B, int64_t Np, int H, int d)
{
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rows = nchunks * B * Np * H;
    if (w >= rows)
        return;
    const int h = static_cast<int>(w % H);
    const int64_t t = (w / H) % Np;
    const int64_t cb = w / (H * Np);  // chunk * B + b
    const int64_t li = (cb * H + h) * Np + t;
    const float la = lse_a[li], lb = lse_b[li];
    const float m = fmaxf(la, lb);
    const float wa = __expf(la - m), wb = __expf(lb - m);
    const float inv = 1.f / (wa + wb);
    T *pa = o_a + w * d;
    const T *pb = o_b + w * d;
    for (int c = lane; c < d; c += 32)
        pa[c] = to_t<T>((wa * ld_f<T>(pa + c) + wb * ld_f<T>(pb + c)) * inv);
    if (lane == 0)
        lse_a[li] = m + __logf(wa + wb);
}

template <typename T>
__global__ void accumulate_kernel(float *__restrict__ acc, const T *__restrict__ part, int64_t n)
{
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        acc[i] += ld_f<T>(part + i);
}

template <typename T>
__global__ void store_kernel(T *__restrict__ out, const float *__restrict__ acc, int64_t n)
{
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = to_t<T>(acc[i]);
}

unsigned grid_for(int64_t n)
{
    const int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
    return static_cast<unsigned>(blocks < cap ? blocks : cap);
}

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

struct RingSizes {
    int64_t Np, q_chunk, kv_chunk, lse_chunk;  // elements per chunk
    int es;
};

RingSizes sizes(int64_t B, int64_t N, int Hq, int Hkv, int d, int P, uly_dtype dt)
{
    RingSizes z;
    z.Np = N / P;
    z.q_chunk = B * z.Np * Hq * d;
    z.kv_chunk = B * z.Np * Hkv * d;
    z.lse_chunk = B * Hq * z.Np;
    z.es = dt == ULY_BF16 ? 2 : 4;
    return z;
}

// A step: query chunks [q0, q0+n) meet key chunks [k0, k0+n).
struct Pair {
    int q0, k0, n, causal;
};

int step_pairs(int k, int P, int causal, Pair (&out)[2])
{
    if (k == 0) {
        out[0] = Pair{0, 0, P, causal};
        return 1;
    }
    int cnt = 0;
    out[cnt++] = Pair{k, 0, P - k, 0};                 // key chunk r - k, before the queries
    if (!causal)
        out[cnt++] = Pair{0, P - k, k, 0};             // wrapped: key chunk r - k + P
    return cnt;
}

}  // namespace

size_t ring_workspace_size(int64_t B, int64_t N, int Hq, int Hkv, int d, int P, bool bwd, uly_dtype dt)
{
    const RingSizes z = sizes(B, N, Hq, Hkv, d, P, dt);
    const size_t attn_ws = ulysses_attn_workspace_size(B, z.Np, Hq, Hkv, d, P, 0, bwd ? 1 : 0, dt);
    if (attn_ws == 0)
        return 0;
    if (!bwd)
        return al(attn_ws) + al(P * z.q_chunk * z.es) + al(P * z.lse_chunk * sizeof(float));
    return al(attn_ws) + al(P * z.q_chunk * z.es) + 2 * al(P * z.kv_chunk * z.es) +
           al(P * z.q_chunk * sizeof(float)) + 2 * al(P * z.kv_chunk * sizeof(float));
}

uly_status ring_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t N, int Hq,
                    int Hkv, int d, int P, int causal, float scale, uly_dtype dt, void *workspace, size_t ws_bytes,
                    cudaStream_t s)
{
    const RingSizes z = sizes(B, N, Hq, Hkv, d, P, dt);
    const size_t attn_ws = ulysses_attn_workspace_size(B, z.Np, Hq, Hkv, d, P, 0, 0, dt);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *o_part = ws + al(attn_ws);
    float *lse_part = reinterpret_cast<float *>(ws + al(attn_ws) + al(P * z.q_chunk * z.es));
    const uint8_t *qb = static_cast<const uint8_t *>(q), *kb = static_cast<const uint8_t *>(k),
                  *vb = static_cast<const uint8_t *>(v);
    uint8_t *ob = static_cast<uint8_t *>(o);
    for (int step = 0; step < P; ++step) {
        Pair pairs[2];
        const int np = step_pairs(step, P, causal, pairs);
        for (int pi = 0; pi < np; ++pi) {
            const Pair &pr = pairs[pi];
            // step 0 writes the running result directly; later steps a partial
            void *dst_o = step == 0 ? static_cast<void *>(ob) : o_part;
            float *dst_l = step == 0 ? lse : lse_part;
            uly_status st = attn_fwd_impl(
                qb + pr.q0 * z.q_chunk * z.es, kb + pr.k0 * z.kv_chunk * z.es, vb + pr.k0 * z.kv_chunk * z.es,
                static_cast<uint8_t *>(dst_o) + (step == 0 ? 0 : pr.q0 * z.q_chunk * z.es),
                dst_l + (step == 0 ? 0 : pr.q0 * z.lse_chunk), B, z.Np, Hq, Hkv, d, pr.n, pr.causal, nullptr, 0,
                scale, dt, workspace, attn_ws, s, head_rows(B, z.Np, pr.n));
            if (st != ULY_OK)
                return st;
            if (step == 0)
                continue;
            const int64_t rows = pr.n * B * z.Np * Hq;
            const unsigned blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
            if (dt == ULY_BF16)
                merge_kernel<uint16_t><<<blocks, 256, 0, s>>>(
                    reinterpret_cast<uint16_t *>(ob) + pr.q0 * z.q_chunk, lse + pr.q0 * z.lse_chunk,
                    static_cast<const uint16_t *>(o_part) + pr.q0 * z.q_chunk, lse_part + pr.q0 * z.lse_chunk, pr.n,
                    B, z.Np, Hq, d);
            else
                merge_kernel<float><<<blocks, 256, 0, s>>>(
                    reinterpret_cast<float *>(ob) + pr.q0 * z.q_chunk, lse + pr.q0 * z.lse_chunk,
                    static_cast<const float *>(o_part) + pr.q0 * z.q_chunk, lse_part + pr.q0 * z.lse_chunk, pr.n, B,
                    z.Np, Hq, d);
            if (cudaGetLastError() != cudaSuccess)
                return ULY_ERR_CUDA;
        }
    }
    return ULY_OK;
}

uly_status ring_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
                    void *dq, void *dk, void *dv, int64_t B, int64_t N, int Hq, int Hkv, int d, int P, int causal,
                    float scale, uly_dtype dt, void *workspace, size_t ws_bytes, cudaStream_t s)
{
    const RingSizes z = sizes(B, N, Hq, Hkv, d, P, dt);
    const size_t attn_ws = ulysses_attn_workspace_size(B, z.Np, Hq, Hkv, d, P, 0, 1, dt);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    size_t off = al(attn_ws);
    uint8_t *dq_part = ws + off;
    off += al(P * z.q_chunk * z.es);
    uint8_t *dk_part = ws + off;
    off += al(P * z.kv_chunk * z.es);
    uint8_t *dv_part = ws + off;
    off += al(P * z.kv_chunk * z.es);
    float *dq_acc = reinterpret_cast<float *>(ws + off);
    off += al(P * z.q_chunk * sizeof(float));
    float *dk_acc = reinterpret_cast<float *>(ws + off);
    off += al(P * z.kv_chunk * sizeof(float));
    float *dv_acc = reinterpret_cast<float *>(ws + off);
    if (cudaMemsetAsync(dq_acc, 0, P * z.q_chunk * sizeof(float), s) != cudaSuccess ||
        cudaMemsetAsync(dk_acc, 0, P * z.kv_chunk * sizeof(float), s) != cudaSuccess ||
        cudaMemsetAsync(dv_acc, 0, P * z.kv_chunk * sizeof(float), s) != cudaSuccess)
        return ULY_ERR_CUDA;
    const uint8_t *qb = static_cast<const uint8_t *>(q), *kb = static_cast<const uint8_t *>(k),
                  *vb = static_cast<const uint8_t *>(v), *obp = static_cast<const uint8_t *>(o),
                  *dob = static_cast<const uint8_t *>(dout);
    for (int step = 0; step < P; ++step) {
        Pair pairs[2];
        const int np = step_pairs(step, P, causal, pairs);
        for (int pi = 0; pi < np; ++pi) {
            const Pair &pr = pairs[pi];
            uly_status st = attn_bwd_impl(
                qb + pr.q0 * z.q_chunk * z.es, kb + pr.k0 * z.kv_chunk * z.es, vb + pr.k0 * z.kv_chunk * z.es,
                obp + pr.q0 * z.q_chunk * z.es, lse + pr.q0 * z.lse_chunk, dob + pr.q0 * z.q_chunk * z.es, dq_part,
                dk_part, dv_part, B, z.Np, Hq, Hkv, d, pr.n, pr.causal, nullptr, 0, scale, dt, workspace, attn_ws,
                s, head_rows(B, z.Np, pr.n));
            if (st != ULY_OK)
                return st;
            const int64_t nq = pr.n * z.q_chunk, nkv = pr.n * z.kv_chunk;
            if (dt == ULY_BF16) {
                accumulate_kernel<uint16_t><<<grid_for(nq), 256, 0, s>>>(
                    dq_acc + pr.q0 * z.q_chunk, reinterpret_cast<const uint16_t *>(dq_part), nq);
                accumulate_kernel<uint16_t><<<grid_for(nkv), 256, 0, s>>>(
                    dk_acc + pr.k0 * z.kv_chunk, reinterpret_cast<const uint16_t *>(dk_part), nkv);
                accumulate_kernel<uint16_t><<<grid_for(nkv), 256, 0, s>>>(
                    dv_acc + pr.k0 * z.kv_chunk, reinterpret_cast<const uint16_t *>(dv_part), nkv);
            } else {
                accumulate_kernel<float><<<grid_for(nq), 256, 0, s>>>(dq_acc + pr.q0 * z.q_chunk,
                                                                       reinterpret_cast<const float *>(dq_part), nq);
                accumulate_kernel<float><<<grid_for(nkv), 256, 0, s>>>(dk_acc + pr.k0 * z.kv_chunk,
                                                                        reinterpret_cast<const float *>(dk_part), nkv);
                accumulate_kernel<float><<<grid_for(nkv), 256, 0, s>>>(dv_acc + pr.k0 * z.kv_chunk,
                                                                        reinterpret_cast<const float *>(dv_part), nkv);
            }
            if (cudaGetLastError() != cudaSuccess)
                return ULY_ERR_CUDA;
        }
    }
    const int64_t nq = P * z.q_chunk, nkv = P * z.kv_chunk;
    if (dt == ULY_BF16) {
        store_kernel<uint16_t><<<grid_for(nq), 256, 0, s>>>(static_cast<uint16_t *>(dq), dq_acc, nq);
        store_kernel<uint16_t><<<grid_for(nkv), 256, 0, s>>>(static_cast<uint16_t *>(dk), dk_acc, nkv);
        store_kernel<uint16_t><<<grid_for(nkv), 256, 0, s>>>(static_cast<uint16_t *>(dv), dv_acc, nkv);
    } else {
        store_kernel<float><<<grid_for(nq), 256, 0, s>>>(static_cast<float *>(dq), dq_acc, nq);
        store_kernel<float><<<grid_for(nkv), 256, 0, s>>>(static_cast<float *>(dk), dk_acc, nkv);
        store_kernel<float><<<grid_for(nkv), 256, 0, s>>>(static_cast<float *>(dv), dv_acc, nkv);
    }
    return cudaGetLastError() == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

}  // namespace uly
