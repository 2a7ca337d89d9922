// seq<->head all-to-all of Ulysses sequence parallelism on one GPU.
//
// Index map (Transformers docs "Ulysses sequence parallelism", the all-to-all
// diagram): rank s of the sequence layout holds tokens [s*N/P, (s+1)*N/P) for
// all H heads; after the swap rank r holds all N tokens for the contiguous
// head block [r*H/P, (r+1)*H/P).
//
//   head[r][b][s*Np + t][h][k] = seq[s][b][t][r*Hp + h][k]     (Np = N/P, Hp = H/P)
//
// For a fixed (s, b, r) and a run of T tokens, the head-side bytes are one
// contiguous block of T*Hp*d elements, while the seq-side bytes are T pieces
// of Hp*d elements spaced H*d apart.  A 5-D TMA tensor map over the seq
// buffer, dims {d, Hp, P, Np, P*B}, moves the strided side in one
// instruction (load for seq->head, store for head->seq); a plain bulk copy
// moves the contiguous side.  One elected thread per CTA keeps a ring of
// shared-memory stages full, so every byte crosses HBM exactly once in each
// direction in 16-byte-aligned bulk transfers.  Two CTAs share each SM (two
// independent rings of 32 KB stages keep more transfers in flight than one
// thread alone issues); rows too large for three stages in half the shared
// memory run one CTA per SM instead.
//
// One launch moves a batch of up to four tensors that share B, N, d, P and
// the dtype (Q, K and V have different head counts; O going back while dO
// comes in are two directions): their work items form one list that every
// CTA strides through, so small tensors do not each pay a launch's fill and
// drain (the all-to-all diagram exchanges Q, K and V together).
#include <cstring>

#include "uly_internal.h"

namespace uly {
namespace {

constexpr int kSwapSmemBytes = 196608;  // largest ring of stages per CTA
constexpr int kSwapPairRing = 98304;     // ring when two CTAs share an SM
constexpr int kSwapMaxStages = 8;

// One tensor of a batch.
struct SwapTensor {
    uint8_t *head;       // head-layout buffer (src for head->seq, dst for seq->head)
    int64_t row_bytes;   // Hp * d * esize: one token of one head block
    int64_t nchunks;     // ceil(Np / T)
    int64_t item0;       // first item of this tensor in the batch's list
    int64_t nitems;      // P (src shard) * B * nchunks * P (dst head block)
    int64_t head_bytes;  // extent of the head-layout buffer (bounds checks of debug builds)
    int T;               // tokens per work item (TMA box height)
    int to_head;         // 1: seq->head, 0: head->seq
};

struct SwapParams {
    CUtensorMap maps[kSwapMaxBatch];  // 5-D maps over each tensor's seq buffer
    SwapTensor t[kSwapMaxBatch];
    int ntensors;
    int64_t B, N, Np;    // batch, tokens, tokens per shard
    int P;               // virtual ranks
    int64_t nitems;      // all tensors
    int stages;
    uint32_t stage_alloc;  // bytes between stages
    WaitCfg w;
};

// global item -> (tensor, s, b, chunk, r); consecutive items of a tensor
// share the seq-side chunk.
struct Item {
    int tn, s, b, r;
    int64_t t0;
    int nt;
};

__device__ __forceinline__ Item decode(const SwapParams &p, int64_t it)
{
    Item x;
    x.tn = 0;
#pragma unroll 1
    while (x.tn + 1 < p.ntensors && it >= p.t[x.tn + 1].item0)
        ++x.tn;
    const SwapTensor &t = p.t[x.tn];
    int64_t rest = it - t.item0;
    x.r = static_cast<int>(rest % p.P);
    rest /= p.P;
    const int64_t c = rest % t.nchunks;
    rest /= t.nchunks;
    x.b = static_cast<int>(rest % p.B);
    x.s = static_cast<int>(rest / p.B);
    x.t0 = c * t.T;
    const int64_t left = p.Np - x.t0;
    x.nt = static_cast<int>(left < t.T ? left : t.T);
    return x;
}

__device__ __forceinline__ uint8_t *head_ptr(const SwapParams &p, const Item &x)
{
    // head[r][b][s*Np + t0] : contiguous nt * row_bytes
    const SwapTensor &t = p.t[x.tn];
    return t.head + ((static_cast<int64_t>(x.r) * p.B + x.b) * p.N + static_cast<int64_t>(x.s) * p.Np + x.t0) *
                        t.row_bytes;
}

__global__ void __launch_bounds__(32, 1) swap_kernel(const __grid_constant__ SwapParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kSwapMaxStages];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    if (threadIdx.x != 0)
        return;
    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    if (first >= p.nitems)
        return;
    const int64_t n_local = (p.nitems - first + stride - 1) / stride;
    for (int i = 0; i < p.stages; ++i)
        mbar_init(&full[i], 1);
    fence_mbar_init();
    for (int i = 0; i < p.ntensors; ++i)
        prefetch_tmap(&p.maps[i]);

    auto issue_load = [&](int64_t k) {
        const int st = static_cast<int>(k % p.stages);
        const Item x = decode(p, first + k * stride);
        const SwapTensor &t = p.t[x.tn];
        uint8_t *buf = smem + static_cast<int64_t>(st) * p.stage_alloc;
        if (t.to_head) {
            // strided seq-side gather: box {d, Hp, 1, T, 1}; rows past Np are zero-filled
            mbar_expect_tx(&full[st], static_cast<uint32_t>(t.T * t.row_bytes));
            tma_load_5d(buf, &p.maps[x.tn], &full[st], 0, 0, x.r, static_cast<int>(x.t0),
                        x.s * static_cast<int>(p.B) + x.b);
        } else {
            const uint32_t bytes = static_cast<uint32_t>(x.nt * t.row_bytes);
            const bool ok = ULY_IN_BOUNDS(p.w.status, head_ptr(p, x) - t.head, bytes, t.head_bytes, 0x31);
            mbar_expect_tx(&full[st], ok ? bytes : 0u);
            if (ok)
                bulk_g2s(buf, head_ptr(p, x), bytes, &full[st]);
        }
    };

    int64_t issued = 0;
    for (; issued < n_local && issued < p.stages; ++issued)
        issue_load(issued);

    int64_t k = 0;
    bool ok = true;
    for (; k < n_local; ++k) {
        const int st = static_cast<int>(k % p.stages);
        const Item x = decode(p, first + k * stride);
        const SwapTensor &t = p.t[x.tn];
        if (!mbar_wait(&full[st], static_cast<uint32_t>((k / p.stages) & 1), p.w, t.to_head ? 0x11 : 0x12)) {
            ok = false;
            break;
        }
        const uint8_t *buf = smem + static_cast<int64_t>(st) * p.stage_alloc;
        if (t.to_head) {
            if (ULY_IN_BOUNDS(p.w.status, head_ptr(p, x) - t.head, x.nt * t.row_bytes, t.head_bytes, 0x32))
                bulk_s2g(head_ptr(p, x), buf, static_cast<uint32_t>(x.nt * t.row_bytes));
        } else {
            // strided seq-side scatter; tokens past Np are clipped by the map
            fence_async_smem();
            tma_store_5d(&p.maps[x.tn], buf, 0, 0, x.r, static_cast<int>(x.t0), x.s * static_cast<int>(p.B) + x.b);
        }
        bulk_commit();
        // refill the stage released by the previous item's store; with a
        // single stage, the one this item's store is still reading
        if (issued < n_local && (k >= 1 || p.stages == 1)) {
            if (p.stages == 1)
                bulk_wait_read<0>();
            else
                bulk_wait_read<1>();
            issue_load(issued);
            ++issued;
        }
    }
    if (!ok) {
        // drain loads still in flight into this CTA's shared memory
        for (int64_t j = k; j < issued; ++j)
            mbar_wait(&full[j % p.stages], static_cast<uint32_t>((j / p.stages) & 1), p.w, 0x13);
    }
    bulk_wait_all<0>();
}

// Tokens per work item for rows of row_bytes: about 32 KB per item.
int tokens_per_item(int64_t row_bytes, int64_t Np)
{
    int T = static_cast<int>(32768 / row_bytes);
    if (T < 1)
        T = 1;
    if (T > 256)
        T = 256;
    if (T > Np)
        T = static_cast<int>(Np);
    return T;
}

}  // namespace

cudaError_t launch_swap_batch(const SwapDesc *descs, int n, int64_t B, int64_t N, int d, int P, int esize,
                              cudaStream_t stream)
{
    if (n < 1 || n > kSwapMaxBatch)
        return cudaErrorInvalidValue;
    const int64_t Np = N / P;
    SwapParams p;
    memset(&p, 0, sizeof(p));
    p.ntensors = n;
    p.B = B;
    p.N = N;
    p.Np = Np;
    p.P = P;
    p.w = wait_cfg();
    uint32_t stage_alloc = 0;
    int64_t items = 0;
    for (int i = 0; i < n; ++i) {
        const int H = descs[i].H;
        const int Hp = H / P;
        const int64_t row_bytes = static_cast<int64_t>(Hp) * d * esize;
        if (row_bytes > kSwapSmemBytes || Hp > 256 || d > 256)
            return cudaErrorInvalidValue;
        const int T = tokens_per_item(row_bytes, Np);
        const uint32_t stage_bytes = static_cast<uint32_t>(T * row_bytes);
        const uint32_t a = (stage_bytes + 1023) & ~1023u;
        stage_alloc = a > stage_alloc ? a : stage_alloc;

        // 5-D map over the seq buffer: {d, Hp, P, Np, P*B}, box {d, Hp, 1, T, 1}
        const bool to_head = descs[i].to_head != 0;
        const uint8_t *seq = static_cast<const uint8_t *>(to_head ? descs[i].src : descs[i].dst);
        const CUtensorMapDataType dt = esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32;
        cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hp), static_cast<cuuint64_t>(P),
                              static_cast<cuuint64_t>(Np), static_cast<cuuint64_t>(P) * static_cast<cuuint64_t>(B)};
        cuuint64_t strides[4] = {static_cast<cuuint64_t>(d) * esize, static_cast<cuuint64_t>(row_bytes),
                                 static_cast<cuuint64_t>(H) * d * esize,
                                 static_cast<cuuint64_t>(Np) * H * d * esize};
        cuuint32_t box[5] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(Hp), 1, static_cast<cuuint32_t>(T),
                             1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        CUresult cr = tensor_map_encoder()(&p.maps[i], dt, 5, const_cast<uint8_t *>(seq), dims, strides, box, estr,
                                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS)
            return cudaErrorInvalidValue;

        SwapTensor &t = p.t[i];
        t.head = static_cast<uint8_t *>(to_head ? descs[i].dst : const_cast<void *>(descs[i].src));
        t.row_bytes = row_bytes;
        t.T = T;
        t.nchunks = (Np + T - 1) / T;
        t.item0 = items;
        t.nitems = static_cast<int64_t>(P) * B * t.nchunks * P;
        t.head_bytes = B * N * static_cast<int64_t>(H) * d * esize;
        t.to_head = to_head ? 1 : 0;
        items += t.nitems;
    }
    p.nitems = items;
    // two CTAs per SM with half the ring each, unless that leaves fewer than three stages
    const bool pair = kSwapPairRing / stage_alloc >= 3;
    int stages = static_cast<int>((pair ? kSwapPairRing : kSwapSmemBytes) / stage_alloc);
    if (stages > kSwapMaxStages)
        stages = kSwapMaxStages;
    p.stages = stages;
    p.stage_alloc = stage_alloc;

    const size_t smem = static_cast<size_t>(stages) * stage_alloc + 1024;
    int64_t grid = (pair ? 2 : 1) * static_cast<int64_t>(num_sms());
    if (grid > p.nitems)
        grid = p.nitems;
    cudaError_t e = cudaFuncSetAttribute(swap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    swap_kernel<<<static_cast<unsigned>(grid), 32, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_swap(bool to_head, const void *src, void *dst, int64_t B, int64_t N, int H, int d, int P,
                        int esize, cudaStream_t stream)
{
    SwapDesc one{src, dst, H, to_head ? 1 : 0};
    return launch_swap_batch(&one, 1, B, N, d, P, esize, stream);
}

}  // namespace uly
