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
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int kSwapSmemBytes = 196608;  // largest ring of stages per CTA
constexpr int kSwapPairRing = 98304;     // ring when two CTAs share an SM
constexpr int kSwapMaxStages = 8;

__device__ __forceinline__ void tma_store_5d(const CUtensorMap *map, const void *smem_src, int c0, int c1, int c2,
                                             int c3, int c4)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group"
        " [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(map),
        "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

struct SwapParams {
    uint8_t *head;       // head-layout buffer (src for head->seq, dst for seq->head)
    int64_t B, N, Np;    // batch, tokens, tokens per shard
    int P;               // virtual ranks
    int64_t row_bytes;   // Hp * d * esize: one token of one head block
    int T;               // tokens per work item (TMA box height)
    int64_t nchunks;     // ceil(Np / T)
    int64_t nitems;      // P (src shard) * B * nchunks * P (dst head block)
    int stages;
    uint32_t stage_bytes;  // T * row_bytes
    WaitCfg w;
};

// item -> (s, b, chunk, r); consecutive items share the seq-side chunk.
struct Item {
    int s, b, r;
    int64_t t0;
    int nt;
};

__device__ __forceinline__ Item decode(const SwapParams &p, int64_t it)
{
    Item x;
    x.r = static_cast<int>(it % p.P);
    int64_t rest = it / p.P;
    const int64_t c = rest % p.nchunks;
    rest /= p.nchunks;
    x.b = static_cast<int>(rest % p.B);
    x.s = static_cast<int>(rest / p.B);
    x.t0 = c * p.T;
    const int64_t left = p.Np - x.t0;
    x.nt = static_cast<int>(left < p.T ? left : p.T);
    return x;
}

__device__ __forceinline__ uint8_t *head_ptr(const SwapParams &p, const Item &x)
{
    // head[r][b][s*Np + t0] : contiguous nt * row_bytes
    return p.head + ((static_cast<int64_t>(x.r) * p.B + x.b) * p.N + static_cast<int64_t>(x.s) * p.Np + x.t0) *
                        p.row_bytes;
}

template <bool kToHead>
__global__ void __launch_bounds__(32, 1) swap_kernel(const __grid_constant__ CUtensorMap seq_map, SwapParams p)
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
    prefetch_tmap(&seq_map);

    auto issue_load = [&](int64_t k) {
        const int st = static_cast<int>(k % p.stages);
        const Item x = decode(p, first + k * stride);
        uint8_t *buf = smem + static_cast<int64_t>(st) * p.stage_bytes;
        if (kToHead) {
            // strided seq-side gather: box {d, Hp, 1, T, 1}; rows past Np are zero-filled
            mbar_expect_tx(&full[st], p.stage_bytes);
            tma_load_5d(buf, &seq_map, &full[st], 0, 0, x.r, static_cast<int>(x.t0), x.s * static_cast<int>(p.B) + x.b);
        } else {
            const uint32_t bytes = static_cast<uint32_t>(x.nt * p.row_bytes);
            mbar_expect_tx(&full[st], bytes);
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
        if (!mbar_wait(&full[st], static_cast<uint32_t>((k / p.stages) & 1), p.w, kToHead ? 0x11 : 0x12)) {
            ok = false;
            break;
        }
        const Item x = decode(p, first + k * stride);
        const uint8_t *buf = smem + static_cast<int64_t>(st) * p.stage_bytes;
        if (kToHead) {
            bulk_s2g(head_ptr(p, x), buf, static_cast<uint32_t>(x.nt * p.row_bytes));
        } else {
            // strided seq-side scatter; tokens past Np are clipped by the map
            fence_async_smem();
            tma_store_5d(&seq_map, buf, 0, 0, x.r, static_cast<int>(x.t0), x.s * static_cast<int>(p.B) + x.b);
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

}  // namespace

cudaError_t launch_swap(bool to_head, const void *src, void *dst, int64_t B, int64_t N, int H, int d, int P,
                        int esize, cudaStream_t stream)
{
    const int Hp = H / P;
    const int64_t Np = N / P;
    const int64_t row_bytes = static_cast<int64_t>(Hp) * d * esize;
    if (row_bytes > kSwapSmemBytes || Hp > 256 || d > 256)
        return cudaErrorInvalidValue;
    int T = static_cast<int>(32768 / row_bytes);
    if (T < 1)
        T = 1;
    if (T > 256)
        T = 256;
    if (T > Np)
        T = static_cast<int>(Np);
    const uint32_t stage_bytes = static_cast<uint32_t>(T * row_bytes);
    const uint32_t stage_alloc = (stage_bytes + 1023) & ~1023u;
    // two CTAs per SM with half the ring each, unless that leaves fewer than three stages
    const bool pair = kSwapPairRing / stage_alloc >= 3;
    int stages = static_cast<int>((pair ? kSwapPairRing : kSwapSmemBytes) / stage_alloc);
    if (stages > kSwapMaxStages)
        stages = kSwapMaxStages;

    // 5-D map over the seq buffer: {d, Hp, P, Np, P*B}
    const uint8_t *seq = static_cast<const uint8_t *>(to_head ? src : dst);
    CUtensorMap map;
    const CUtensorMapDataType dt = esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32;
    cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hp), static_cast<cuuint64_t>(P),
                          static_cast<cuuint64_t>(Np), static_cast<cuuint64_t>(P) * static_cast<cuuint64_t>(B)};
    cuuint64_t strides[4] = {static_cast<cuuint64_t>(d) * esize, static_cast<cuuint64_t>(row_bytes),
                             static_cast<cuuint64_t>(H) * d * esize,
                             static_cast<cuuint64_t>(Np) * H * d * esize};
    cuuint32_t box[5] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(Hp), 1, static_cast<cuuint32_t>(T), 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult cr = tensor_map_encoder()(&map, dt, 5, const_cast<uint8_t *>(seq), dims, strides, box, estr,
                                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    SwapParams p;
    p.head = static_cast<uint8_t *>(to_head ? dst : const_cast<void *>(src));
    p.B = B;
    p.N = N;
    p.Np = Np;
    p.P = P;
    p.row_bytes = row_bytes;
    p.T = T;
    p.nchunks = (Np + T - 1) / T;
    p.nitems = static_cast<int64_t>(P) * B * p.nchunks * P;
    p.stages = stages;
    p.stage_bytes = stage_bytes;
    p.w = wait_cfg();

    const size_t smem = static_cast<size_t>(stages) * ((stage_bytes + 1023) & ~1023u) + 1024;
    int64_t grid = (pair ? 2 : 1) * static_cast<int64_t>(num_sms());
    if (grid > p.nitems)
        grid = p.nitems;
    cudaError_t e;
    if (to_head) {
        e = cudaFuncSetAttribute(swap_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        swap_kernel<true><<<static_cast<unsigned>(grid), 32, smem, stream>>>(map, p);
    } else {
        e = cudaFuncSetAttribute(swap_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        swap_kernel<false><<<static_cast<unsigned>(grid), 32, smem, stream>>>(map, p);
    }
    return cudaGetLastError();
}

}  // namespace uly
