// Sequence-parallel loss: labels shifted over the whole sequence before it is
// sharded, per-shard mean cross entropy over the good tokens, and the
// good-token-weighted aggregation across the P shards (Accelerate PR
// "Deepspeed Ulysses/ALST integration", user API step 2; the Transformers
// docs list label shifting and loss aggregation among what the Trainer does
// for SP), plus the gradient of the aggregated loss with respect to the
// logits.
//
//   shifted[b][n] = labels[b][n + 1]  (n < N - 1),  -100 for the last token
//   loss_r  = mean over rank r's good tokens of  lse(logits) - logits[label]
//   total   = sum_r loss_r * good_r / max(sum_r good_r, 1)
//   d total / d logits[row] = (softmax(row) - onehot(label)) / max(T, 1)
//                             for good rows, 0 for ignored rows.
//
// Memory-bound: every kernel streams the logits with 16-byte loads.  Without
// the gradient one CTA per token row computes the row's log-sum-exp online
// (running maximum and rescaled sum) in one pass.  With the gradient the row
// must be seen twice (the normaliser comes before any gradient element), so
// a cluster of C CTAs holds the row on chip instead: each bulk-loads one
// 16-byte-aligned chunk into shared memory (in four pieces, so the reduction
// starts on the first while the rest arrive), the C partial (max, sum) pairs
// are merged through distributed shared memory, and each CTA writes its
// chunk of the gradient from shared memory with coalesced 16-byte stores --
// one HBM read and one write per element.  The shard reductions are deterministic trees, no float atomics.
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int kRowThreads = 256;
constexpr int kIgnore = -100;

// shifted labels (int32) and per-shard good counts; labels out of range are
// reported through the status word and treated as ignored
__global__ void shift_count_kernel(const int64_t *__restrict__ labels, int32_t *__restrict__ shifted,
                                   unsigned long long *__restrict__ good, int64_t B, int64_t N, int64_t Np,
                                   int P, int64_t V, unsigned *status)
{
    const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t rows = B * N;
    int is_good = 0;
    int r = 0;
    if (row < rows) {
        const int64_t t = row % Np;
        const int64_t b = (row / Np) % B;
        r = static_cast<int>(row / (Np * B));
        const int64_t n = static_cast<int64_t>(r) * Np + t;  // position in sequence row b
        int32_t y = kIgnore;
        if (n + 1 < N) {
            const int64_t r2 = (n + 1) / Np, t2 = (n + 1) % Np;
            const int64_t lab = labels[(r2 * B + b) * Np + t2];
            if (lab >= 0 && lab < V)
                y = static_cast<int32_t>(lab);
            else if (lab != kIgnore)
                atomicOr(status, kDevBadArg);
        }
        shifted[row] = y;
        is_good = (y != kIgnore);
    }
    // one atomic per warp and shard (rows of a block may span two shards)
    const unsigned mask = __ballot_sync(0xffffffffu, is_good);
    const int r0 = __shfl_sync(0xffffffffu, r, 0);
    const bool same = __all_sync(0xffffffffu, r == r0 || row >= rows);
    if (same) {
        if ((threadIdx.x & 31) == 0 && mask)
            atomicAdd(&good[r0], static_cast<unsigned long long>(__popc(mask)));
    } else if (is_good) {
        atomicAdd(&good[r], 1ull);
    }
}

struct MS {
    float m, s;  // running maximum (log2 domain) and sum of 2^(x - m)
};

__device__ __forceinline__ MS ms_merge(MS a, MS b)
{
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY)
        return MS{m, 0.f};
    return MS{m, a.s * ex2_approx(a.m - m) + b.s * ex2_approx(b.m - m)};
}

template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&x)[8]);

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t *p, float (&x)[8])
{
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float *p, float (&x)[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}

template <typename T>
__device__ __forceinline__ void store8(T *p, const float (&g)[8]);

template <>
__device__ __forceinline__ void store8<uint16_t>(uint16_t *p, const float (&g)[8])
{
    *reinterpret_cast<uint4 *>(p) =
        make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7]));
}

template <>
__device__ __forceinline__ void store8<float>(float *p, const float (&g)[8])
{
    *reinterpret_cast<float4 *>(p) = make_float4(g[0], g[1], g[2], g[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(g[4], g[5], g[6], g[7]);
}

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<uint16_t>(uint16_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
}
template <>
__device__ __forceinline__ float to_f<float>(float v)
{
    return v;
}

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ uint16_t from_f<uint16_t>(float v)
{
    return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}
template <>
__device__ __forceinline__ float from_f<float>(float v)
{
    return v;
}

// One CTA per token row: log-sum-exp over V, the row's loss, optionally the
// gradient row.  vec: V is a multiple of 8 and rows are 16-byte aligned.
template <typename T, bool kVec>
__global__ void __launch_bounds__(kRowThreads) ce_rows_kernel(const T *__restrict__ logits,
                                                              const int32_t *__restrict__ shifted,
                                                              const unsigned long long *__restrict__ good, int P,
                                                              int64_t V, float *__restrict__ row_loss,
                                                              T *__restrict__ dlogits)
{
    constexpr float kLog2e = 1.4426950408889634f;
    const int64_t row = blockIdx.x;
    const T *x = logits + row * V;
    MS acc{-INFINITY, 0.f};
    if (kVec) {
        for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < V; c += kRowThreads * 8) {
            float v[8];
            load8<T>(x + c, v);
            float vm = v[0];
#pragma unroll
            for (int k = 1; k < 8; ++k)
                vm = fmaxf(vm, v[k]);
            vm *= kLog2e;
            if (vm > acc.m) {
                acc.s = (acc.m == -INFINITY) ? 0.f : acc.s * ex2_approx(acc.m - vm);
                acc.m = vm;
            }
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                s += ex2_approx(fmaf(v[k], kLog2e, -acc.m));
            acc.s += s;
        }
    } else {
        for (int64_t c = threadIdx.x; c < V; c += kRowThreads) {
            const float v = to_f<T>(x[c]) * kLog2e;
            if (v > acc.m) {
                acc.s = (acc.m == -INFINITY) ? 0.f : acc.s * ex2_approx(acc.m - v);
                acc.m = v;
            }
            acc.s += ex2_approx(v - acc.m);
        }
    }
    // block reduction of (max, sum)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MS other{__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.s, o)};
        acc = ms_merge(acc, other);
    }
    __shared__ MS red[kRowThreads / 32];
    __shared__ float lse2_sh;
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        MS t = red[0];
        for (int w = 1; w < kRowThreads / 32; ++w)
            t = ms_merge(t, red[w]);
        const float lse2 = t.m + __log2f(t.s);  // log2 of sum_k 2^(x_k log2 e)
        lse2_sh = lse2;
        const int32_t y = shifted[row];
        row_loss[row] = (y >= 0) ? (lse2 - to_f<T>(x[y]) * kLog2e) * 0.69314718055994530942f : 0.f;
    }
    if (dlogits == nullptr)
        return;
    __syncthreads();
    const float lse2 = lse2_sh;
    const int32_t y = shifted[row];
    unsigned long long T_all = 0;
    for (int r = 0; r < P; ++r)
        T_all += good[r];
    const float inv_t = 1.f / static_cast<float>(T_all > 0 ? T_all : 1ull);
    T *g = dlogits + row * V;
    if (kVec) {
        for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < V; c += kRowThreads * 8) {
            float v[8], o[8];
            load8<T>(x + c, v);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float pk = ex2_approx(fmaf(v[k], kLog2e, -lse2));
                o[k] = (y >= 0) ? (pk - ((c + k) == y ? 1.f : 0.f)) * inv_t : 0.f;
            }
            store8<T>(g + c, o);
        }
    } else {
        for (int64_t c = threadIdx.x; c < V; c += kRowThreads) {
            const float pk = ex2_approx(fmaf(to_f<T>(x[c]), kLog2e, -lse2));
            g[c] = from_f<T>((y >= 0) ? (pk - (c == y ? 1.f : 0.f)) * inv_t : 0.f);
        }
    }
}

// On-chip variant for the gradient: one row per cluster of C CTAs (C = 1, 2,
// 4 or 8).  CTA `rank` holds elements [rank*Vc, rank*Vc + n) of the row.
constexpr int kOnchipMaxChunkBytes = 80 * 1024;  // two CTAs per SM

__device__ __forceinline__ MS ld_cluster_ms(const MS *local, uint32_t cta)
{
    float m, s;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(m), "=f"(s) : "r"(cluster_addr(local, cta))
                 : "memory");
    return MS{m, s};
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float (&x)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void unpack16<uint16_t>(const uint4 &u, float (&x)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &u, float (&x)[4])
{
    x[0] = __uint_as_float(u.x), x[1] = __uint_as_float(u.y), x[2] = __uint_as_float(u.z), x[3] = __uint_as_float(u.w);
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float (&g)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ uint4 pack16<uint16_t>(const float (&g)[8])
{
    return make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]),
                      pack_bf16x2(g[6], g[7]));
}
template <>
__device__ __forceinline__ uint4 pack16<float>(const float (&g)[4])
{
    return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]), __float_as_uint(g[3]));
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) ce_rows_onchip_kernel(const T *__restrict__ logits,
                                                                     const int32_t *__restrict__ shifted,
                                                                     const unsigned long long *__restrict__ good,
                                                                     int P, int64_t V, int64_t Vc, int C,
                                                                     float *__restrict__ row_loss,
                                                                     T *__restrict__ dlogits, WaitCfg w)
{
    constexpr float kLog2e = 1.4426950408889634f;
    constexpr int kPer = 16 / sizeof(T);  // elements per 16-byte vector
    extern __shared__ __align__(128) uint8_t chunk_raw[];
    __shared__ __align__(8) uint64_t bar[4];  // one per quarter of the chunk
    __shared__ __align__(8) MS part;  // this CTA's (max, sum), read by the whole cluster
    __shared__ MS red[kRowThreads / 32];
    __shared__ float lse2_sh;
    const uint32_t rank = cluster_ctarank();
    const int64_t row = blockIdx.x / C;
    const int64_t c0 = static_cast<int64_t>(rank) * Vc;
    const int64_t n = (V - c0 < Vc) ? V - c0 : Vc;  // > 0 and a multiple of kPer (checked at launch)
    uint4 *buf = reinterpret_cast<uint4 *>(chunk_raw);
    const int64_t nv = n / kPer;
    const int64_t sub = (nv + 3) / 4;  // 16-byte vectors per quarter
    if (threadIdx.x == 0) {
        for (int q = 0; q < 4; ++q)
            mbar_init(&bar[q], 1);
        fence_mbar_init();
        for (int q = 0; q < 4; ++q) {
            const int64_t v0 = q * sub, v1 = (q + 1) * sub < nv ? (q + 1) * sub : nv;
            const uint32_t qb = v1 > v0 ? static_cast<uint32_t>((v1 - v0) * 16) : 0u;
            if (qb) {
                mbar_expect_tx(&bar[q], qb);
                bulk_g2s(buf + v0, reinterpret_cast<const uint8_t *>(logits + row * V + c0) + v0 * 16, qb, &bar[q]);
            } else {
                mbar_arrive(&bar[q]);
            }
        }
    }
    __syncthreads();
    bool ok = true;
    // (max, sum of 2^(x log2 e - max)) over the chunk, online
    MS acc{-INFINITY, 0.f};
    for (int q = 0; q < 4 && ok; ++q) {
        ok = mbar_wait(&bar[q], 0, w, 0x91);
        const int64_t v1 = (q + 1) * sub < nv ? (q + 1) * sub : nv;
        for (int64_t i = q * sub + threadIdx.x; ok && i < v1; i += kRowThreads) {
            float v[kPer];
            unpack16<T>(buf[i], v);
            float vm = v[0];
#pragma unroll
            for (int k = 1; k < kPer; ++k)
                vm = fmaxf(vm, v[k]);
            vm *= kLog2e;
            if (vm > acc.m) {
                acc.s = (acc.m == -INFINITY) ? 0.f : acc.s * ex2_approx(acc.m - vm);
                acc.m = vm;
            }
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < kPer; ++k)
                sum += ex2_approx(fmaf(v[k], kLog2e, -acc.m));
            acc.s += sum;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MS other{__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.s, o)};
        acc = ms_merge(acc, other);
    }
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        MS t = red[0];
        for (int k = 1; k < kRowThreads / 32; ++k)
            t = ms_merge(t, red[k]);
        part = t;
    }
    // every CTA's partial is visible cluster-wide after this barrier
    cluster_sync_all();
    if (threadIdx.x == 0) {
        // merged in rank order: every CTA of the row computes the same value
        MS t = ld_cluster_ms(&part, 0);
        for (int r = 1; r < C; ++r)
            t = ms_merge(t, ld_cluster_ms(&part, static_cast<uint32_t>(r)));
        const float lse2 = t.m + __log2f(t.s);
        lse2_sh = lse2;
        if (rank == 0) {
            const int32_t y = shifted[row];
            row_loss[row] = (y >= 0) ? (lse2 - to_f<T>(logits[row * V + y]) * kLog2e) * 0.69314718055994530942f : 0.f;
        }
    }
    __syncthreads();
    const float lse2 = lse2_sh;
    const int32_t y = shifted[row];
    unsigned long long T_all = 0;
    for (int r = 0; r < P; ++r)
        T_all += good[r];
    const float inv_t = 1.f / static_cast<float>(T_all > 0 ? T_all : 1ull);
    if (ok) {
        // the gradient over the chunk, straight from shared memory
        for (int64_t i = threadIdx.x; i < nv; i += kRowThreads) {
            float v[kPer], g[kPer];
            unpack16<T>(buf[i], v);
            const int64_t c = c0 + i * kPer;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const float pk = ex2_approx(fmaf(v[k], kLog2e, -lse2));
                g[k] = (y >= 0) ? (pk - ((c + k) == y ? 1.f : 0.f)) * inv_t : 0.f;
            }
            reinterpret_cast<uint4 *>(dlogits + row * V + c0)[i] = pack16<T>(g);
        }
    }
    // no CTA leaves while another may still read its partial
    cluster_sync_all();
}

// Per shard: deterministic sum of its rows' losses, mean over its good tokens.
__global__ void __launch_bounds__(1024) shard_reduce_kernel(const float *__restrict__ row_loss,
                                                            const unsigned long long *__restrict__ good,
                                                            int64_t rows_per_shard, float *__restrict__ shard_loss,
                                                            int64_t *__restrict__ shard_good)
{
    const int r = blockIdx.x;
    const float *base = row_loss + static_cast<int64_t>(r) * rows_per_shard;
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < rows_per_shard; i += blockDim.x)
        s += base[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    __shared__ double part[32];
    if ((threadIdx.x & 31) == 0)
        part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w)
            t += part[w];
        const unsigned long long gr = good[r];
        shard_loss[r] = gr > 0 ? static_cast<float>(t / static_cast<double>(gr)) : 0.f;
        shard_good[r] = static_cast<int64_t>(gr);
    }
}

// total = sum_r loss_r * good_r / max(sum_r good_r, 1), in the pages' form
__global__ void total_kernel(const float *__restrict__ shard_loss, const int64_t *__restrict__ shard_good, int P,
                             float *__restrict__ total)
{
    double num = 0.0;
    long long den = 0;
    for (int r = 0; r < P; ++r) {
        num += static_cast<double>(shard_loss[r]) * static_cast<double>(shard_good[r]);
        den += shard_good[r];
    }
    *total = static_cast<float>(num / static_cast<double>(den > 1 ? den : 1));
}

template <typename T>
cudaError_t run(const void *logits, const int64_t *labels, void *dlogits, float *shard_loss, int64_t *shard_good,
                float *total, int64_t B, int64_t N, int64_t V, int P, int32_t *shifted, float *row_loss,
                unsigned long long *good, cudaStream_t s)
{
    const int64_t Np = N / P;
    const int64_t rows = B * N;
    cudaError_t e = cudaMemsetAsync(good, 0, sizeof(unsigned long long) * P, s);
    if (e != cudaSuccess)
        return e;
    shift_count_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, s>>>(labels, shifted, good, B, N, Np, P,
                                                                                 V, device_status_ptr());
    const bool vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0) &&
                     (dlogits == nullptr || reinterpret_cast<uintptr_t>(dlogits) % 16 == 0);
    // with the gradient: the smallest cluster whose chunks fit on chip
    int C = 0;
    int64_t Vc = 0;
    if (vec && dlogits != nullptr) {
        constexpr int64_t kPer = 16 / sizeof(T);
        for (int c = 1; c <= 8; c *= 2) {
            const int64_t vc = ((V + c - 1) / c + kPer - 1) / kPer * kPer;
            if (vc * static_cast<int64_t>(sizeof(T)) <= kOnchipMaxChunkBytes && V - (c - 1) * vc > 0) {
                C = c;
                Vc = vc;
                break;
            }
        }
    }
    if (C > 0) {
        const size_t smem = static_cast<size_t>(Vc) * sizeof(T);
        e = cudaFuncSetAttribute(ce_rows_onchip_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(rows * C));
        cfg.blockDim = dim3(kRowThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(C);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, ce_rows_onchip_kernel<T>, static_cast<const T *>(logits),
                               static_cast<const int32_t *>(shifted), static_cast<const unsigned long long *>(good), P,
                               V, Vc, C, row_loss, static_cast<T *>(dlogits), wait_cfg());
        if (e != cudaSuccess)
            return e;
    } else if (vec)
        ce_rows_kernel<T, true><<<static_cast<unsigned>(rows), kRowThreads, 0, s>>>(
            static_cast<const T *>(logits), shifted, good, P, V, row_loss, static_cast<T *>(dlogits));
    else
        ce_rows_kernel<T, false><<<static_cast<unsigned>(rows), kRowThreads, 0, s>>>(
            static_cast<const T *>(logits), shifted, good, P, V, row_loss, static_cast<T *>(dlogits));
    shard_reduce_kernel<<<P, 1024, 0, s>>>(row_loss, good, B * Np, shard_loss, shard_good);
    total_kernel<<<1, 1, 0, s>>>(shard_loss, shard_good, P, total);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sharded_ce(const void *logits, const int64_t *labels, void *dlogits, float *shard_loss,
                              int64_t *shard_good, float *total, int64_t B, int64_t N, int64_t V, int P, int esize,
                              void *workspace, cudaStream_t stream)
{
    // workspace: [256-byte header: good counts] [shifted labels int32 B*N] [row losses fp32 B*N]
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    unsigned long long *good = reinterpret_cast<unsigned long long *>(ws);
    const size_t lab_bytes = (static_cast<size_t>(B) * N * sizeof(int32_t) + 255) & ~size_t(255);
    const size_t head = (static_cast<size_t>(P) * sizeof(unsigned long long) + 255) & ~size_t(255);
    int32_t *shifted = reinterpret_cast<int32_t *>(ws + head);
    float *row_loss = reinterpret_cast<float *>(ws + head + lab_bytes);
    if (esize == 2)
        return run<uint16_t>(logits, labels, dlogits, shard_loss, shard_good, total, B, N, V, P, shifted, row_loss,
                             good, stream);
    return run<float>(logits, labels, dlogits, shard_loss, shard_good, total, B, N, V, P, shifted, row_loss, good,
                      stream);
}

size_t sharded_ce_workspace(int64_t B, int64_t N, int P)
{
    const size_t head = (static_cast<size_t>(P) * sizeof(unsigned long long) + 255) & ~size_t(255);
    const size_t lab_bytes = (static_cast<size_t>(B) * N * sizeof(int32_t) + 255) & ~size_t(255);
    const size_t loss_bytes = (static_cast<size_t>(B) * N * sizeof(float) + 255) & ~size_t(255);
    return head + lab_bytes + loss_bytes;
}

}  // namespace uly
