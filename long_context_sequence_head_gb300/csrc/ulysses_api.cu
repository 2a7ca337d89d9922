// extern "C" entry points declared in include/ulysses.h: host-side
// validation, workspace carving and kernel dispatch.  Nothing here allocates
// device memory; every buffer belongs to the caller.
#include <ulysses.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "uly_internal.h"

namespace {

// Device status word: [0] flags (uly::kDevTimeout | uly::kDevBadArg),
// [1] id of the first wait site that ran out.
__device__ unsigned g_device_status[2];

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int esize_of(uly_dtype dt) { return dt == ULY_BF16 ? 2 : (dt == ULY_FP32 ? 4 : 0); }

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return -1;
    return dev;
}

__global__ void selftest_bounds_kernel(unsigned *status)
{
    // an access of 4 elements at offset 8 of a 4-element buffer: the check
    // fails and reports; nothing is read or written
    if (threadIdx.x == 0 && ULY_IN_BOUNDS(status, 8, 4, 4, 0x7f))
        atomicOr(status, uly::kDevBadArg);  // reached only if the check passed
}

__global__ void selftest_timeout_kernel(uly::WaitCfg w)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0)
        return;
    uly::mbar_init(&bar, 1);
    uly::fence_mbar_init();
    // nothing ever arrives on `bar`: the bounded wait must give up
    uly::mbar_wait(&bar, 0, w, 0x7e);
}

// Workspace layout (every region 256-byte aligned):
//   [0, 256)          reserved
//   cu_seqlens copy   (num_docs + 1) int32, if documents are packed
//   tile order        ceil(N/128) int32, if documents are packed (the bf16
//                     kernels' walk order, longest walks first)
//   bf16 backward     lse2 [SB][Hq][Npad], D [SB][Hq][Npad], dq_acc [SB][Hq][Npad][d]
//   fp32 backward     D [SB][Hq][N]
struct WsLayout {
    size_t cu_off = 0, order_off = 0, lse2_off = 0, D_off = 0, acc_off = 0, total = 0;
    int64_t Npad = 0;
};

WsLayout ws_layout(int64_t B, int64_t N, int Hq, int d, int S, int num_docs, bool bwd, uly_dtype dt)
{
    WsLayout L;
    size_t off = kAlign;
    L.cu_off = off;
    if (num_docs > 0)
        off += align_up(static_cast<size_t>(num_docs + 1) * sizeof(int32_t));
    L.order_off = off;
    if (num_docs > 0)
        off += align_up(static_cast<size_t>((N + 127) / 128) * sizeof(int32_t));
    const int64_t SB = static_cast<int64_t>(S) * B;
    L.Npad = (N + 127) / 128 * 128;
    if (bwd) {
        if (dt == ULY_BF16) {
            const size_t rows = static_cast<size_t>(SB) * Hq * L.Npad;
            L.lse2_off = off;
            off += align_up(rows * sizeof(float));
            L.D_off = off;
            off += align_up(rows * sizeof(float));
            L.acc_off = off;
            off += align_up(rows * d * sizeof(float));
        } else {
            L.D_off = off;
            off += align_up(static_cast<size_t>(SB) * Hq * N * sizeof(float));
        }
    }
    L.total = off;
    return L;
}

// cu_seqlens: none (num_docs = 0), or [0 .. N] non-decreasing over num_docs >= 1 documents.
uly_status check_docs(int64_t N, const int32_t *cu, int32_t num_docs)
{
    if (cu == nullptr)
        return num_docs == 0 ? ULY_OK : ULY_ERR_INVALID_ARG;
    if (num_docs < 1 || cu[0] != 0 || static_cast<int64_t>(cu[num_docs]) != N)
        return ULY_ERR_INVALID_ARG;
    for (int i = 0; i < num_docs; ++i)
        if (cu[i + 1] < cu[i])
            return ULY_ERR_INVALID_ARG;
    return ULY_OK;
}

uly_status check_attn_args(int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d, int32_t S, int32_t causal,
                           const int32_t *cu, int32_t num_docs, uly_dtype dt)
{
    if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || S < 1 || (causal != 0 && causal != 1))
        return ULY_ERR_INVALID_ARG;
    if (Hq % Hkv != 0)
        return ULY_ERR_INVALID_ARG;
    if (d != 64 && d != 128)
        return ULY_ERR_UNSUPPORTED;
    if (esize_of(dt) == 0)
        return ULY_ERR_INVALID_ARG;
    if (dt == ULY_BF16 && d != 128)
        return ULY_ERR_UNSUPPORTED;
    if (N > (int64_t(1) << 30) || static_cast<int64_t>(S) * B > (int64_t(1) << 20))
        return ULY_ERR_UNSUPPORTED;
    return check_docs(N, cu, num_docs);
}

uly_status check_swap_args(const void *a, const void *b, int64_t B, int64_t N, int32_t H, int32_t d, int32_t P,
                           uly_dtype dt)
{
    if (a == nullptr || b == nullptr)
        return ULY_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || H < 1 || P < 1 || P > H)
        return ULY_ERR_INVALID_ARG;
    if (H % P != 0 || N % P != 0)
        return ULY_ERR_INVALID_ARG;
    if (d != 64 && d != 128)
        return ULY_ERR_UNSUPPORTED;
    const int es = esize_of(dt);
    if (es == 0)
        return ULY_ERR_INVALID_ARG;
    if (H / P > 256 || static_cast<int64_t>(H / P) * d * es > 196608)
        return ULY_ERR_UNSUPPORTED;
    if (N / P > (int64_t(1) << 31) - 1 || static_cast<int64_t>(P) * B > (int64_t(1) << 31) - 1)
        return ULY_ERR_UNSUPPORTED;
    if (!aligned16(a) || !aligned16(b))
        return ULY_ERR_MISALIGNED;
    const size_t bytes = static_cast<size_t>(B) * N * H * d * es;
    if (overlap(a, bytes, b, bytes))
        return ULY_ERR_OVERLAP;
    return ULY_OK;
}

uly_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ULY_OK : ULY_ERR_CUDA; }

}  // namespace

namespace uly {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

unsigned *device_status_ptr()
{
    const int dev = current_device();
    if (dev < 0)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess)
            g_status_ptr[dev] = static_cast<unsigned *>(p);
    }
    return g_status_ptr[dev];
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

int num_sms()
{
    const int dev = current_device();
    if (dev < 0)
        return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 1;
    }
    return g_sms[dev];
}

cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream)
{
    WaitCfg w{device_status_ptr(), limit_ns};
    if (w.status == nullptr)
        return cudaErrorInvalidDevice;
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(w);
    return cudaGetLastError();
}

}  // namespace uly

extern "C" {

uly_status ulysses_seq_to_head(const void *x_seq, void *x_head, int64_t B, int64_t N, int32_t H, int32_t d,
                               int32_t P, uly_dtype dtype, void *stream)
{
    ULY_NVTX_RANGE();
    const uly_status st = check_swap_args(x_seq, x_head, B, N, H, d, P, dtype);
    if (st != ULY_OK)
        return st;
    if (uly::tensor_map_encoder() == nullptr || uly::device_status_ptr() == nullptr)
        return ULY_ERR_CUDA;
    return from_cuda(uly::launch_swap(true, x_seq, x_head, B, N, H, d, P, esize_of(dtype),
                                      static_cast<cudaStream_t>(stream)));
}

uly_status ulysses_head_to_seq(const void *x_head, void *x_seq, int64_t B, int64_t N, int32_t H, int32_t d,
                               int32_t P, uly_dtype dtype, void *stream)
{
    ULY_NVTX_RANGE();
    const uly_status st = check_swap_args(x_head, x_seq, B, N, H, d, P, dtype);
    if (st != ULY_OK)
        return st;
    if (uly::tensor_map_encoder() == nullptr || uly::device_status_ptr() == nullptr)
        return ULY_ERR_CUDA;
    return from_cuda(uly::launch_swap(false, x_head, x_seq, B, N, H, d, P, esize_of(dtype),
                                      static_cast<cudaStream_t>(stream)));
}

uly_status ulysses_swap_batch(const uly_swap_desc *descs_host, int32_t n_descs, int64_t B, int64_t N, int32_t d,
                              int32_t P, uly_dtype dtype, void *stream)
{
    ULY_NVTX_RANGE();
    if (descs_host == nullptr || n_descs < 1 || n_descs > uly::kSwapMaxBatch)
        return ULY_ERR_INVALID_ARG;
    uly::SwapDesc descs[uly::kSwapMaxBatch];
    const int es = esize_of(dtype);
    for (int i = 0; i < n_descs; ++i) {
        const uly_swap_desc &x = descs_host[i];
        if (x.to_head != 0 && x.to_head != 1)
            return ULY_ERR_INVALID_ARG;
        const uly_status st = check_swap_args(x.src, x.dst, B, N, x.H, d, P, dtype);
        if (st != ULY_OK)
            return st;
        descs[i] = uly::SwapDesc{x.src, x.dst, x.H, x.to_head};
    }
    // the entries run concurrently: no entry may write where another reads or writes
    for (int i = 0; i < n_descs; ++i) {
        const size_t bi = static_cast<size_t>(B) * N * descs_host[i].H * d * es;
        for (int j = 0; j < n_descs; ++j) {
            if (i == j)
                continue;
            const size_t bj = static_cast<size_t>(B) * N * descs_host[j].H * d * es;
            if (overlap(descs_host[i].dst, bi, descs_host[j].src, bj) ||
                overlap(descs_host[i].dst, bi, descs_host[j].dst, bj))
                return ULY_ERR_OVERLAP;
        }
    }
    if (uly::tensor_map_encoder() == nullptr || uly::device_status_ptr() == nullptr)
        return ULY_ERR_CUDA;
    return from_cuda(uly::launch_swap_batch(descs, n_descs, B, N, d, P, es, static_cast<cudaStream_t>(stream)));
}

uly_status ulysses_attn_tile_order(int64_t N, int32_t causal, const int32_t *cu_seqlens_host, int32_t num_docs,
                                   int32_t for_bwd, int32_t *out)
{
    if (out == nullptr || N < 1 || N > (int64_t(1) << 30) || (causal != 0 && causal != 1) ||
        (for_bwd != 0 && for_bwd != 1))
        return ULY_ERR_INVALID_ARG;
    const uly_status st = check_docs(N, cu_seqlens_host, num_docs);
    if (st != ULY_OK)
        return st;
    uly::tile_order_host(for_bwd != 0, N, causal, cu_seqlens_host, num_docs, out);
    return ULY_OK;
}

size_t ulysses_attn_workspace_size(int64_t B, int64_t N, int32_t Hq_local, int32_t Hkv_local, int32_t d,
                                   int32_t num_shards, int32_t num_docs, int32_t for_bwd, uly_dtype dtype)
{
    if (B < 1 || N < 1 || Hq_local < 1 || Hkv_local < 1 || num_shards < 1 || num_docs < 0 ||
        Hq_local % Hkv_local != 0 || (d != 64 && d != 128) || esize_of(dtype) == 0 ||
        (dtype == ULY_BF16 && d != 128))
        return 0;
    return ws_layout(B, N, Hq_local, d, num_shards, num_docs, for_bwd != 0, dtype).total;
}

}  // extern "C"

namespace uly {

uly_status attn_fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t N,
                         int32_t Hq_local, int32_t Hkv_local, int32_t d, int32_t num_shards, int32_t causal,
                         const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale, uly_dtype dtype,
                         void *workspace, size_t workspace_bytes, void *stream, uly::RowLayout L)
{
    if (!q || !k || !v || !o || !lse || !workspace)
        return ULY_ERR_INVALID_ARG;
    uly_status st = check_attn_args(B, N, Hq_local, Hkv_local, d, num_shards, causal, cu_seqlens_host, num_docs,
                                    dtype);
    if (st != ULY_OK)
        return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(workspace))
        return ULY_ERR_MISALIGNED;
    const WsLayout W = ws_layout(B, N, Hq_local, d, num_shards, num_docs, false, dtype);
    if (workspace_bytes < W.total)
        return ULY_ERR_WORKSPACE;
    if (uly::tensor_map_encoder() == nullptr || uly::device_status_ptr() == nullptr)
        return ULY_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uly::AttnShape sh;
    sh.SB = static_cast<int64_t>(num_shards) * B;
    sh.N = N;
    sh.Hq = Hq_local;
    sh.Hkv = Hkv_local;
    sh.d = d;
    sh.causal = causal;
    sh.num_docs = cu_seqlens_host ? num_docs : 0;
    sh.cu_dev = nullptr;
    sh.cu_host = cu_seqlens_host;
    sh.order_dev = nullptr;
    sh.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(d));
    sh.L = L;
    sh.q_elems = sh.SB * N * Hq_local * d;
    sh.kv_elems = sh.SB * N * Hkv_local * d;
    sh.lse_elems = sh.SB * N * Hq_local;
    sh.status = uly::device_status_ptr();
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (cu_seqlens_host) {
        // cu_seqlens and the tile walk order, adjacent in the workspace: one
        // copy (from pageable memory, staged before the call returns)
        std::vector<int32_t> host((W.order_off - W.cu_off) / sizeof(int32_t) + (N + 127) / 128);
        std::copy(cu_seqlens_host, cu_seqlens_host + num_docs + 1, host.begin());
        uly::tile_order_host(false, N, causal, cu_seqlens_host, num_docs,
                             host.data() + (W.order_off - W.cu_off) / sizeof(int32_t));
        cudaError_t e = cudaMemcpyAsync(ws + W.cu_off, host.data(), host.size() * sizeof(int32_t),
                                        cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess)
            return ULY_ERR_CUDA;
        sh.cu_dev = reinterpret_cast<int32_t *>(ws + W.cu_off);
        sh.order_dev = reinterpret_cast<int32_t *>(ws + W.order_off);
    }
    if (dtype == ULY_FP32)
        return from_cuda(uly::launch_attn_fwd_f32(sh, static_cast<const float *>(q), static_cast<const float *>(k),
                                                  static_cast<const float *>(v), static_cast<float *>(o), lse, s));
    return from_cuda(uly::launch_attn_fwd_bf16(sh, q, k, v, o, lse, s));
}

uly_status attn_bwd_impl(const void *q, const void *k, const void *v, const void *o, const float *lse,
                         const void *dout, void *dq, void *dk, void *dv, int64_t B, int64_t N, int32_t Hq_local,
                         int32_t Hkv_local, int32_t d, int32_t num_shards, int32_t causal,
                         const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale, uly_dtype dtype,
                         void *workspace, size_t workspace_bytes, void *stream, uly::RowLayout L)
{
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
        return ULY_ERR_INVALID_ARG;
    uly_status st = check_attn_args(B, N, Hq_local, Hkv_local, d, num_shards, causal, cu_seqlens_host, num_docs,
                                    dtype);
    if (st != ULY_OK)
        return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
        return ULY_ERR_MISALIGNED;
    const WsLayout W = ws_layout(B, N, Hq_local, d, num_shards, num_docs, true, dtype);
    if (workspace_bytes < W.total)
        return ULY_ERR_WORKSPACE;
    if (uly::tensor_map_encoder() == nullptr || uly::device_status_ptr() == nullptr)
        return ULY_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uly::AttnShape sh;
    sh.SB = static_cast<int64_t>(num_shards) * B;
    sh.N = N;
    sh.Hq = Hq_local;
    sh.Hkv = Hkv_local;
    sh.d = d;
    sh.causal = causal;
    sh.num_docs = cu_seqlens_host ? num_docs : 0;
    sh.cu_dev = nullptr;
    sh.cu_host = cu_seqlens_host;
    sh.order_dev = nullptr;
    sh.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(d));
    sh.L = L;
    sh.q_elems = sh.SB * N * Hq_local * d;
    sh.kv_elems = sh.SB * N * Hkv_local * d;
    sh.lse_elems = sh.SB * N * Hq_local;
    sh.status = uly::device_status_ptr();
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (cu_seqlens_host) {
        // cu_seqlens and the tile walk order, adjacent in the workspace: one
        // copy (from pageable memory, staged before the call returns)
        std::vector<int32_t> host((W.order_off - W.cu_off) / sizeof(int32_t) + (N + 127) / 128);
        std::copy(cu_seqlens_host, cu_seqlens_host + num_docs + 1, host.begin());
        uly::tile_order_host(true, N, causal, cu_seqlens_host, num_docs,
                             host.data() + (W.order_off - W.cu_off) / sizeof(int32_t));
        cudaError_t e = cudaMemcpyAsync(ws + W.cu_off, host.data(), host.size() * sizeof(int32_t),
                                        cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess)
            return ULY_ERR_CUDA;
        sh.cu_dev = reinterpret_cast<int32_t *>(ws + W.cu_off);
        sh.order_dev = reinterpret_cast<int32_t *>(ws + W.order_off);
    }
    if (dtype == ULY_FP32)
        return from_cuda(uly::launch_attn_bwd_f32(
            sh, static_cast<const float *>(q), static_cast<const float *>(k), static_cast<const float *>(v),
            static_cast<const float *>(o), lse, static_cast<const float *>(dout), static_cast<float *>(dq),
            static_cast<float *>(dk), static_cast<float *>(dv), reinterpret_cast<float *>(ws + W.D_off), s));
    uly::BwdScratch scr;
    scr.lse2 = reinterpret_cast<float *>(ws + W.lse2_off);
    scr.D = reinterpret_cast<float *>(ws + W.D_off);
    scr.dq_acc = reinterpret_cast<float *>(ws + W.acc_off);
    scr.Npad = W.Npad;
    return from_cuda(uly::launch_attn_bwd_bf16(sh, q, k, v, o, lse, dout, dq, dk, dv, scr, s));
}

uly::RowLayout head_rows(int64_t B, int64_t N, int32_t S) { return uly::RowLayout{0, static_cast<int>(B), N, S}; }

}  // namespace uly

namespace {

// Arguments of the sequence-layout calls, mapped onto per-shard sizes.
uly_status check_seq_args(int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d, int32_t P, uly_dtype dtype)
{
    if (B < 1 || N < 1 || P < 1 || Hq < 1 || Hkv < 1)
        return ULY_ERR_INVALID_ARG;
    if (N % P != 0 || Hq % P != 0 || Hkv % P != 0 || P > Hkv)
        return ULY_ERR_INVALID_ARG;
    // a 128-token tile must not straddle two sequence shards
    if (dtype == ULY_BF16 && (N / P) % 128 != 0)
        return ULY_ERR_UNSUPPORTED;
    (void)d;
    return ULY_OK;
}

}  // namespace

extern "C" {

uly_status ulysses_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t N,
                            int32_t Hq_local, int32_t Hkv_local, int32_t d, int32_t num_shards, int32_t causal,
                            const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale, uly_dtype dtype,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    ULY_NVTX_RANGE();
    return uly::attn_fwd_impl(q, k, v, o, lse, B, N, Hq_local, Hkv_local, d, num_shards, causal, cu_seqlens_host,
                         num_docs, softmax_scale, dtype, workspace, workspace_bytes, stream,
                         uly::head_rows(B, N, num_shards));
}

uly_status ulysses_attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                            const void *dout, void *dq, void *dk, void *dv, int64_t B, int64_t N, int32_t Hq_local,
                            int32_t Hkv_local, int32_t d, int32_t num_shards, int32_t causal,
                            const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale, uly_dtype dtype,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    ULY_NVTX_RANGE();
    return uly::attn_bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, N, Hq_local, Hkv_local, d, num_shards, causal,
                         cu_seqlens_host, num_docs, softmax_scale, dtype, workspace, workspace_bytes, stream,
                         uly::head_rows(B, N, num_shards));
}

uly_status ulysses_attn_fwd_seq(const void *q_seq, const void *k_seq, const void *v_seq, void *o_seq, float *lse,
                                int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int32_t causal,
                                const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale,
                                uly_dtype dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    ULY_NVTX_RANGE();
    const uly_status st = check_seq_args(B, N, Hq, Hkv, d, P, dtype);
    if (st != ULY_OK)
        return st;
    return uly::attn_fwd_impl(q_seq, k_seq, v_seq, o_seq, lse, B, N, Hq / P, Hkv / P, d, P, causal, cu_seqlens_host,
                         num_docs, softmax_scale, dtype, workspace, workspace_bytes, stream,
                         uly::RowLayout{1, static_cast<int>(B), N / P, P});
}

uly_status ulysses_attn_bwd_seq(const void *q_seq, const void *k_seq, const void *v_seq, const void *o_seq,
                                const float *lse, const void *dout_seq, void *dq_seq, void *dk_seq, void *dv_seq,
                                int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int32_t causal,
                                const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale,
                                uly_dtype dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    ULY_NVTX_RANGE();
    const uly_status st = check_seq_args(B, N, Hq, Hkv, d, P, dtype);
    if (st != ULY_OK)
        return st;
    return uly::attn_bwd_impl(q_seq, k_seq, v_seq, o_seq, lse, dout_seq, dq_seq, dk_seq, dv_seq, B, N, Hq / P, Hkv / P,
                         d, P, causal, cu_seqlens_host, num_docs, softmax_scale, dtype, workspace, workspace_bytes,
                         stream, uly::RowLayout{1, static_cast<int>(B), N / P, P});
}

size_t ulysses_ring_attn_workspace_size(int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d, int32_t P,
                                        int32_t for_bwd, uly_dtype dtype)
{
    if (B < 1 || N < 1 || P < 1 || N % P != 0)
        return 0;
    return uly::ring_workspace_size(B, N, Hq, Hkv, d, P, for_bwd != 0, dtype);
}

namespace {
uly_status check_ring(const void *const *ptrs, int nptr, int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d,
                      int32_t P, int32_t causal, uly_dtype dtype, void *workspace, size_t ws_bytes, bool bwd)
{
    for (int i = 0; i < nptr; ++i)
        if (ptrs[i] == nullptr)
            return ULY_ERR_INVALID_ARG;
    if (P < 1 || N < 1 || N % P != 0)
        return ULY_ERR_INVALID_ARG;
    const uly_status st = check_attn_args(B, N / P, Hq, Hkv, d, P, causal, nullptr, 0, dtype);
    if (st != ULY_OK)
        return st;
    for (int i = 0; i < nptr; ++i)
        if (!aligned16(ptrs[i]))
            return ULY_ERR_MISALIGNED;
    if (workspace == nullptr || !aligned16(workspace))
        return workspace == nullptr ? ULY_ERR_INVALID_ARG : ULY_ERR_MISALIGNED;
    if (ws_bytes < uly::ring_workspace_size(B, N, Hq, Hkv, d, P, bwd, dtype))
        return ULY_ERR_WORKSPACE;
    if (uly::tensor_map_encoder() == nullptr || uly::device_status_ptr() == nullptr)
        return ULY_ERR_CUDA;
    return ULY_OK;
}
}  // namespace

uly_status ulysses_ring_attn_fwd(const void *q_seq, const void *k_seq, const void *v_seq, void *o_seq, float *lse,
                                 int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int32_t causal,
                                 float softmax_scale, uly_dtype dtype, void *workspace, size_t workspace_bytes,
                                 void *stream)
{
    ULY_NVTX_RANGE();
    const void *ptrs[5] = {q_seq, k_seq, v_seq, o_seq, lse};
    const uly_status st = check_ring(ptrs, 5, B, N, Hq, Hkv, d, P, causal, dtype, workspace, workspace_bytes, false);
    if (st != ULY_OK)
        return st;
    return uly::ring_fwd(q_seq, k_seq, v_seq, o_seq, lse, B, N, Hq, Hkv, d, P, causal, softmax_scale, dtype,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

uly_status ulysses_ring_attn_bwd(const void *q_seq, const void *k_seq, const void *v_seq, const void *o_seq,
                                 const float *lse, const void *dout_seq, void *dq_seq, void *dk_seq, void *dv_seq,
                                 int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int32_t causal,
                                 float softmax_scale, uly_dtype dtype, void *workspace, size_t workspace_bytes,
                                 void *stream)
{
    ULY_NVTX_RANGE();
    const void *ptrs[9] = {q_seq, k_seq, v_seq, o_seq, lse, dout_seq, dq_seq, dk_seq, dv_seq};
    const uly_status st = check_ring(ptrs, 9, B, N, Hq, Hkv, d, P, causal, dtype, workspace, workspace_bytes, true);
    if (st != ULY_OK)
        return st;
    return uly::ring_bwd(q_seq, k_seq, v_seq, o_seq, lse, dout_seq, dq_seq, dk_seq, dv_seq, B, N, Hq, Hkv, d, P,
                         causal, softmax_scale, dtype, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t ulysses_sharded_ce_workspace_size(int64_t B, int64_t N, int32_t P)
{
    if (B < 1 || N < 1 || P < 1 || N % P != 0)
        return 0;
    return uly::sharded_ce_workspace(B, N, P);
}

uly_status ulysses_sharded_ce_loss(const void *logits, const int64_t *labels, void *dlogits, float *shard_loss,
                                   int64_t *shard_good, float *total_loss, int64_t B, int64_t N, int32_t V,
                                   int32_t P, uly_dtype dtype, void *workspace, size_t workspace_bytes,
                                   void *stream)
{
    ULY_NVTX_RANGE();
    if (!logits || !labels || !shard_loss || !shard_good || !total_loss || !workspace)
        return ULY_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || P < 1 || V < 1 || N % P != 0 || esize_of(dtype) == 0)
        return ULY_ERR_INVALID_ARG;
    if (B * N > (int64_t(1) << 31) - 1)
        return ULY_ERR_UNSUPPORTED;
    if (!aligned16(logits) || !aligned16(labels) || !aligned16(shard_loss) || !aligned16(shard_good) ||
        !aligned16(total_loss) || !aligned16(workspace) || (dlogits != nullptr && !aligned16(dlogits)))
        return ULY_ERR_MISALIGNED;
    const size_t bytes = static_cast<size_t>(B) * N * V * esize_of(dtype);
    if (dlogits != nullptr && overlap(logits, bytes, dlogits, bytes))
        return ULY_ERR_OVERLAP;
    if (workspace_bytes < uly::sharded_ce_workspace(B, N, P))
        return ULY_ERR_WORKSPACE;
    if (uly::device_status_ptr() == nullptr)
        return ULY_ERR_CUDA;
    return from_cuda(uly::launch_sharded_ce(logits, labels, dlogits, shard_loss, shard_good, total_loss, B, N, V, P,
                                            esize_of(dtype), workspace, static_cast<cudaStream_t>(stream)));
}

uly_status ulysses_get_device_status(void *stream, uint32_t *site_out)
{
    ULY_NVTX_RANGE();
    unsigned *p = uly::device_status_ptr();
    if (p == nullptr)
        return ULY_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return ULY_ERR_CUDA;
    unsigned host[2] = {0, 0};
    if (cudaMemcpy(host, p, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ULY_ERR_CUDA;
    const unsigned zero[2] = {0, 0};
    if (host[0] != 0 && cudaMemcpy(p, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return ULY_ERR_CUDA;
    if (site_out)
        *site_out = host[1];
    if (host[0] & uly::kDevTimeout)
        return ULY_ERR_TIMEOUT;
    if (host[0] & uly::kDevBounds)
        return ULY_ERR_BOUNDS;
    if (host[0] & uly::kDevBadArg)
        return ULY_ERR_INVALID_ARG;
    return ULY_OK;
}

uly_status ulysses_set_wait_limit_ns(uint64_t limit_ns)
{
    if (limit_ns < 1000)
        return ULY_ERR_INVALID_ARG;
    g_wait_limit_ns.store(limit_ns);
    return ULY_OK;
}

uly_status ulysses_selftest_wait_timeout(uint64_t limit_ns, void *stream)
{
    ULY_NVTX_RANGE();
    if (limit_ns < 1000 || limit_ns > 10000000000ull)
        return ULY_ERR_INVALID_ARG;
    return from_cuda(uly::launch_selftest_timeout(limit_ns, static_cast<cudaStream_t>(stream)));
}

uly_status ulysses_selftest_bounds(void *stream)
{
    ULY_NVTX_RANGE();
#ifdef ULY_DEBUG
    unsigned *status = uly::device_status_ptr();
    if (status == nullptr)
        return ULY_ERR_CUDA;
    selftest_bounds_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    return from_cuda(cudaGetLastError());
#else
    (void)stream;
    return ULY_ERR_UNSUPPORTED;
#endif
}

const char *ulysses_status_string(uly_status status)
{
    switch (status) {
    case ULY_OK:
        return "ok";
    case ULY_ERR_INVALID_ARG:
        return "invalid argument";
    case ULY_ERR_UNSUPPORTED:
        return "unsupported configuration";
    case ULY_ERR_MISALIGNED:
        return "pointer not 16-byte aligned";
    case ULY_ERR_OVERLAP:
        return "input and output overlap";
    case ULY_ERR_CUDA:
        return "CUDA error";
    case ULY_ERR_TIMEOUT:
        return "device-side wait timed out";
    case ULY_ERR_WORKSPACE:
        return "workspace missing or too small";
    case ULY_ERR_SCRATCH_LIMIT:
        return "sizes exceed the fixed scratch of the no-allocation entry point";
    case ULY_ERR_BOUNDS:
        return "a bounds check of the debug build failed";
    }
    return "unknown status";
}

int32_t ulysses_version(void) { return 100; }

}  // extern "C"
