// Attention backward for the bf16 path on tcgen05 tensor cores, head_dim 128.
//
// Gradient of the forward in attn_fwd_bf16.cu (training needs it; the blog
// summary's Trainer discussion requires correct gradients).  With
// P_ij = exp(s_ij - lse_i) recomputed from the stored log-sum-exp and
// D_i = <dO_i, O_i>:
//   dV_j = sum_i P_ij dO_i,   dS_ij = P_ij (<dO_i, v_j> - D_i),
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,
// dK, dV summed over the G query heads that share KV head j.
//
// Kernels:
//   bwd_pre    : D_i and lse_i*log2(e) into fp32 scratch (padded rows get
//                D = 0, lse = +inf so their probabilities are exactly 0).
//   bwd_main   : one CTA per (shard*batch, KV head, 128-key tile).  K and V
//                stay in shared memory; the CTA walks every 128-row query
//                tile that may attend to its keys, and for each of them the
//                G query heads of the group back to back (their Q/dO rows
//                are neighbours in memory).  dK and dV accumulate in TMEM across the whole
//                group (no atomics); each dQ partial is added into an fp32
//                accumulator with coalesced vector reductions.
//   dq_convert : fp32 accumulator * scale -> bf16 dQ in the head layout.
//
// bwd_main warp roles (576 threads):
//   warps 0-15: 4 column quarters x 4 TMEM lane quarters.  Thread = key row j
//               (TMEM lane) for 32 of the 128 query columns: S^T -> P^T (bf16,
//               into TMEM for the dV product), dP^T -> dS^T (bf16, into shared
//               memory for the dK and dQ products).  The same warps read their
//               32 d-columns of each dQ partial (TMEM lane = query row) and
//               reduce them into global memory, and write dK/dV at the end.
//   warp  16  : TMA producer (K, V once; Q, dO, lse, D per iteration, 2 stages)
//   warp  17  : tcgen05.mma issuer and TMEM owner.
// TMEM (512 columns): S^T/P^T | dP^T, later dQ | dV | dK.
// Per (key tile, query tile) the MMAs are S^T = K Q^T, dP^T = V dO^T,
// dV += P^T dO, dK += dS^T Q, dQ = dS K.
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kD = 128;
constexpr int kTile = kBM * kD * 2;  // 32 KB
constexpr int kChunk = 128 * 64 * 2; // 16 KB
constexpr int kCompWarps = 16;                  // 4 column quarters x 4 TMEM lane quarters
constexpr int kProdWarp = kCompWarps, kMmaWarp = kCompWarps + 1;
constexpr int kThreads = (kCompWarps + 2) * 32;  // 576

struct BwdSmem {
    static constexpr int kK = 0;
    static constexpr int kV = kTile;
    static constexpr int kQ = 2 * kTile;       // [2]
    static constexpr int kdO = 4 * kTile;      // [2]
    static constexpr int kdS = 6 * kTile;
    static constexpr int kLse = 7 * kTile;     // [2][128] fp32
    static constexpr int kDv = kLse + 1024;    // [2][128] fp32
    static constexpr int kBars = kDv + 1024;
    static constexpr int kTotal = kBars + 128;
};

struct BwdParams {
    int64_t SB, N, Npad;
    int Hq, Hkv, G, n_ktiles;
    int group;  // problems interleaved in the grid
    const int32_t *order;  // with documents: key tiles, longest walk first
    int causal;
    const int32_t *cu;
    int num_docs;
    float scale_log2;
    float scale;
    const float *lse2;  // [SB][Hq][Npad]
    const float *Dv;    // [SB][Hq][Npad]
    float *dq_acc;      // [SB][Hq][Npad/128][32][128][4]
    uint16_t *dk, *dv;  // rows like k, v
    int64_t kv_elems;   // extent of dk, dv (bounds checks of debug builds)
    WaitCfg w;
    RowLayout L;
};

__device__ __forceinline__ void doc_range(const BwdParams &p, int64_t i, int64_t &lo, int64_t &hi)
{
    lo = 0;
    hi = p.N;
    if (p.cu == nullptr)
        return;
    int a = 0, b = p.num_docs;
    while (b - a > 1) {
        const int m = (a + b) >> 1;
        if (static_cast<int64_t>(p.cu[m]) <= i)
            a = m;
        else
            b = m;
    }
    lo = p.cu[a];
    hi = p.cu[a + 1];
}

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ------------------------------------------------------------------ pre
// One warp per (shard*batch, token): the token's Hq rows of O and dO are
// adjacent in both layouts (Hq x 256 contiguous bytes each), so the warp reads
// them in 512-byte runs, two heads per pass (lanes 0-15 and 16-31, 16 bytes
// a lane), and reduces each head's dot product within its half-warp.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t *__restrict__ o,
                                                      const uint16_t *__restrict__ dout,
                                                      const float *__restrict__ lse, float *__restrict__ lse2,
                                                      float *__restrict__ Dv, int64_t SB, int64_t N, int64_t Npad,
                                                      int Hq, RowLayout L, int64_t q_elems, unsigned *status)
{
    const int64_t row_elems = SB * Hq * Npad;  // lse2, D
    (void)q_elems;
    (void)status;
    (void)row_elems;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = lane_id();
    if (gw >= SB * Npad)
        return;
    const int64_t i = gw % Npad;
    const int64_t sb = gw / Npad;
    if (i >= N) {
        // padded rows: probabilities exactly 0 in the main kernel
        for (int h = lane; h < Hq; h += 32) {
            if (!ULY_IN_BOUNDS(status, (sb * Hq + h) * Npad + i, 1, row_elems, 0x21))
                break;
            Dv[(sb * Hq + h) * Npad + i] = 0.f;
            lse2[(sb * Hq + h) * Npad + i] = INFINITY;
        }
        return;
    }
    const int64_t off = L.off(N, sb, i, Hq, 0, kD);
    // the token's Hq rows are adjacent: one check covers every read below
    if (!ULY_IN_BOUNDS(status, off, static_cast<int64_t>(Hq) * kD, q_elems, 0x22))
        return;
    const uint4 *o4 = reinterpret_cast<const uint4 *>(o + off);
    const uint4 *d4 = reinterpret_cast<const uint4 *>(dout + off);
    const int n16 = Hq * (kD / 8);  // 16-byte pieces of the token's rows
    for (int u0 = 0; u0 < n16; u0 += 32) {
        const int u = u0 + lane;
        float acc = 0.f;
        if (u < n16) {
            const uint4 a = o4[u], b = d4[u];
            acc = bf16lo(a.x) * bf16lo(b.x);
            acc = fmaf(bf16hi(a.x), bf16hi(b.x), acc);
            acc = fmaf(bf16lo(a.y), bf16lo(b.y), acc);
            acc = fmaf(bf16hi(a.y), bf16hi(b.y), acc);
            acc = fmaf(bf16lo(a.z), bf16lo(b.z), acc);
            acc = fmaf(bf16hi(a.z), bf16hi(b.z), acc);
            acc = fmaf(bf16lo(a.w), bf16lo(b.w), acc);
            acc = fmaf(bf16hi(a.w), bf16hi(b.w), acc);
        }
#pragma unroll
        for (int sft = 8; sft > 0; sft >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, sft);
        if (u < n16 && (lane & 15) == 0) {
            const int h = u / (kD / 8);
            const int64_t row = (sb * Hq + h) * Npad + i;
            if (ULY_IN_BOUNDS(status, row, 1, row_elems, 0x23) &&
                ULY_IN_BOUNDS(status, (sb * Hq + h) * N + i, 1, SB * Hq * N, 0x24)) {
                Dv[row] = acc;
                lse2[row] = lse[(sb * Hq + h) * N + i] * 1.4426950408889634f;
            }
        }
    }
}

// ---------------------------------------------------------- dq convert
// One block per 32-row slab of one (sb, h, 128-row tile).  In the accumulator
// each of the slab's 32 column groups is 32 rows x 16 B = 512 contiguous bytes;
// the slab is staged through shared memory and written as whole bf16 rows, so
// both the reads and the writes are contiguous runs.
constexpr int kCvtRows = 32;
constexpr int kCvtPitch = kD + 4;  // floats per staged row; +4 spreads the group stores over all banks

__global__ void __launch_bounds__(256) dq_convert_kernel(const float *__restrict__ acc, uint16_t *__restrict__ dq,
                                                         int64_t SB, int64_t N, int64_t Npad, int Hq, float scale,
                                                         RowLayout L, int64_t q_elems, unsigned *status)
{
    const int64_t acc_elems = SB * Hq * Npad * kD;
    (void)q_elems;
    (void)status;
    (void)acc_elems;
    __shared__ __align__(16) float tile[kCvtRows * kCvtPitch];
    const int64_t ntiles = Npad / kBM;
    int64_t rest = blockIdx.x;
    const int slab = static_cast<int>(rest % (kBM / kCvtRows));
    rest /= kBM / kCvtRows;
    const int64_t mt = rest % ntiles;
    rest /= ntiles;
    const int h = static_cast<int>(rest % Hq);
    const int64_t sb = rest / Hq;
    const int64_t src_off = ((sb * Hq + h) * ntiles + mt) * (32 * kBM * 4);
    // the tile's whole accumulator block: covers every read below
    if (!ULY_IN_BOUNDS(status, src_off, 32 * kBM * 4, acc_elems, 0x25))
        return;
    const float *src = acc + src_off;
    const int r0 = slab * kCvtRows;
    // consecutive threads take consecutive rows of one column group
    for (int k = threadIdx.x; k < 32 * kCvtRows; k += 256) {
        const int g = k / kCvtRows, r = k % kCvtRows;
        *reinterpret_cast<float4 *>(tile + r * kCvtPitch + g * 4) =
            *reinterpret_cast<const float4 *>(src + (g * kBM + r0 + r) * 4);
    }
    __syncthreads();
    // a warp writes whole rows: lane l holds columns 4l .. 4l+3
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = w; r < kCvtRows; r += 8) {
        const int64_t i = mt * kBM + r0 + r;
        if (i >= N)
            break;
        const float4 v = *reinterpret_cast<const float4 *>(tile + r * kCvtPitch + lane * 4);
        uint2 out;
        out.x = pack_bf16x2(v.x * scale, v.y * scale);
        out.y = pack_bf16x2(v.z * scale, v.w * scale);
        const int64_t doff = L.off(N, sb, i, Hq, h, kD) + lane * 4;
        if (ULY_IN_BOUNDS(status, doff, 4, q_elems, 0x26))
            *reinterpret_cast<uint2 *>(dq + doff) = out;
    }
}

// ----------------------------------------------------------------- main
// kDecode: 0 = problem-major, key tiles in index order; 1 = groups of
// problems interleaved; 2 = the same with the host's key-tile order.
template <int kDecode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         BwdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    // the shared-memory budget leaves no room to align by hand: the dynamic
    // window starts 1024-aligned when the kernel declares no static shared
    // memory; refuse to run otherwise
    if ((smem_u32(smem_raw) & 1023u) != 0) {
        if (threadIdx.x == 0)
            atomicOr(p.w.status, kDevBadArg);
        return;
    }
    uint8_t *smem = smem_raw;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BwdSmem::kBars);
    uint64_t *kv_full = bars + 0;
    uint64_t *q_full = bars + 1;   // [2]
    uint64_t *q_empty = bars + 3;  // [2]
    uint64_t *s_full = bars + 5;
    uint64_t *dp_full = bars + 6;
    uint64_t *ds_full = bars + 7;
    uint64_t *p_full = bars + 13;
    uint64_t *ds_empty = bars + 8;
    uint64_t *dq_full = bars + 9;
    uint64_t *dq_empty = bars + 10;
    uint64_t *dkv_done = bars + 11;
    uint64_t *drain = bars + 12;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 14);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id();
    const int lane = lane_id();

    // ---- work unit: problem-major (all resident CTAs share one (shard*batch,
    // KV head) problem, so its Q/dO tiles and dQ accumulator stay in L2), key
    // tiles with the most query tiles first within a problem.  Where one key
    // tile's walk is long next to a problem's share of the GPU (short
    // sequences, documents), the last problem's longest walks would run on
    // alone at the end; there groups of problems interleave their key tiles
    // instead (the launcher picks the group size).  With documents a key
    // tile's walk follows its place in its document, and the host's order
    // puts the longest walks first ----
    int n_blk, prob;
    if constexpr (kDecode == 0) {
        n_blk = static_cast<int>(blockIdx.x % p.n_ktiles);
        prob = static_cast<int>(blockIdx.x / p.n_ktiles);
    } else {
        // groups of p.group problems, key tiles interleaved across the group
        const int64_t nprob = p.SB * p.Hkv;
        const int64_t grp = blockIdx.x / (static_cast<int64_t>(p.group) * p.n_ktiles);
        const int64_t rem = blockIdx.x % (static_cast<int64_t>(p.group) * p.n_ktiles);
        const int64_t gsize = (nprob - grp * p.group < p.group) ? nprob - grp * p.group : p.group;
        const int rank = static_cast<int>(rem / gsize);
        n_blk = kDecode == 2 ? p.order[rank] : rank;
        prob = static_cast<int>(grp * p.group + rem % gsize);
    }
    const int kvh = prob % p.Hkv;
    const int sb = prob / p.Hkv;
    const int64_t kv0 = static_cast<int64_t>(n_blk) * kBN;
    const int64_t key_last = (kv0 + kBN - 1 < p.N - 1) ? kv0 + kBN - 1 : p.N - 1;
    int64_t row_lo, row_hi, tmp;
    doc_range(p, kv0, row_lo, tmp);
    doc_range(p, key_last, tmp, row_hi);
    if (p.causal)
        row_lo = kv0;
    const int m_lo = static_cast<int>(row_lo / kBM);
    const int n_m = static_cast<int>((row_hi - 1) / kBM) - m_lo + 1;
    const int n_it = p.G * n_m;

    if (warp == kProdWarp && lane == 0) {
        for (int i = 0; i < 14; ++i)
            mbar_init(&bars[i], 1);
        mbar_init(ds_full, kCompWarps);  // one elected arrival per compute warp
        mbar_init(p_full, kCompWarps);
        mbar_init(dq_empty, kCompWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tS = tbase, tdP = tbase + 128, tdV = tbase + 256, tdK = tbase + 384;

    if (warp == kProdWarp) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_expect_tx(kv_full, 2 * kTile);
            int c1, c2, c3, c4;
            p.L.tile(sb, kv0, p.Hkv, kvh, c1, c2, c3, c4);
            tma_load_5d(smem + BwdSmem::kK, &tm_k, kv_full, 0, c1, c2, c3, c4);
            tma_load_5d(smem + BwdSmem::kK + kChunk, &tm_k, kv_full, 64, c1, c2, c3, c4);
            tma_load_5d(smem + BwdSmem::kV, &tm_v, kv_full, 0, c1, c2, c3, c4);
            tma_load_5d(smem + BwdSmem::kV + kChunk, &tm_v, kv_full, 64, c1, c2, c3, c4);
            int issued = 0;
            for (int it = 0; it < n_it && !*abort_flag; ++it) {
                const int slot = it & 1;
                const int h = kvh * p.G + it % p.G;
                const int m = m_lo + it / p.G;
                if (!mbar_wait(&q_empty[slot], ((it >> 1) & 1) ^ 1, p.w, 0x51)) {
                    *abort_flag = 1;
                    break;
                }
                const int64_t roff = (static_cast<int64_t>(sb) * p.Hq + h) * p.Npad + static_cast<int64_t>(m) * kBM;
                const bool rows_ok = ULY_IN_BOUNDS(p.w.status, roff, kBM, p.SB * p.Hq * p.Npad, 0x27);
                mbar_expect_tx(&q_full[slot], 2 * kTile + (rows_ok ? 2 * 512 : 0));
                uint8_t *sq = smem + BwdSmem::kQ + slot * kTile;
                uint8_t *sdo = smem + BwdSmem::kdO + slot * kTile;
                p.L.tile(sb, static_cast<int64_t>(m) * kBM, p.Hq, h, c1, c2, c3, c4);
                tma_load_5d(sq, &tm_q, &q_full[slot], 0, c1, c2, c3, c4);
                tma_load_5d(sq + kChunk, &tm_q, &q_full[slot], 64, c1, c2, c3, c4);
                tma_load_5d(sdo, &tm_do, &q_full[slot], 0, c1, c2, c3, c4);
                tma_load_5d(sdo + kChunk, &tm_do, &q_full[slot], 64, c1, c2, c3, c4);
                if (rows_ok) {
                    bulk_g2s(smem + BwdSmem::kLse + slot * 512, p.lse2 + roff, 512, &q_full[slot]);
                    bulk_g2s(smem + BwdSmem::kDv + slot * 512, p.Dv + roff, 512, &q_full[slot]);
                }
                ++issued;
            }
            if (*abort_flag) {
                mbar_wait(kv_full, 0, p.w, 0x5f);
                for (int it = (issued > 2 ? issued - 2 : 0); it < issued; ++it)
                    mbar_wait(&q_full[it & 1], (it >> 1) & 1, p.w, 0x5f);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        // Issue order per iteration it:  dP(it) | dV(it) | S(it+1) | dK(it), dQ(it)
        // so the P part of it+1 and the dS part of it run on the compute
        // warpgroups while the tensor pipe works on the neighbours.
        if (lane == 0) {
            const uint32_t id_kk = idesc_bf16(128, 128, false, false);  // both K-major
            const uint32_t id_kmn = idesc_bf16(128, 128, false, true);  // B MN-major
            const uint32_t id_mnmn = idesc_bf16(128, 128, true, true);  // A and B MN-major
            const uint32_t sK = smem_u32(smem + BwdSmem::kK), sV = smem_u32(smem + BwdSmem::kV);
            const uint32_t sdS = smem_u32(smem + BwdSmem::kdS);
            auto issue_s = [&](int it) {  // S^T = K Q^T
                const uint32_t sQ = smem_u32(smem + BwdSmem::kQ + (it & 1) * kTile);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                    mma_ss(tS, desc_sw128(sK + off, 16, 1024), desc_sw128(sQ + off, 16, 1024), id_kk, kk > 0);
                }
                mma_commit(s_full);
            };
            bool ok = mbar_wait(kv_full, 0, p.w, 0x61) && (n_it == 0 || mbar_wait(&q_full[0], 0, p.w, 0x62));
            if (ok && n_it > 0) {
                tc_fence_after();
                issue_s(0);
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const int slot = it & 1;
                const uint32_t sQ = smem_u32(smem + BwdSmem::kQ + slot * kTile);
                const uint32_t sdO = smem_u32(smem + BwdSmem::kdO + slot * kTile);
                // dP^T = V dO^T into the dP/dQ columns, once dQ(it-1) has been read out
                if (it > 0 && !mbar_wait(dq_empty, (it - 1) & 1, p.w, 0x63)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                    mma_ss(tdP, desc_sw128(sV + off, 16, 1024), desc_sw128(sdO + off, 16, 1024), id_kk, kk > 0);
                }
                mma_commit(dp_full);
                // dV += P^T dO   (A = P^T in TMEM: query columns 32c..32c+31 packed
                // at S cols 32c..32c+15; B = dO, d contiguous)
                if (!mbar_wait(p_full, it & 1, p.w, 0x64)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBM / 16; ++kk)
                    mma_ts(tdV, tS + (kk >> 1) * 32 + (kk & 1) * 8, desc_sw128(sdO + kk * 2048, kChunk, 1024), id_kmn,
                           (it > 0 || kk > 0) ? 1u : 0u);
                // next S^T (overwrites P^T(it), which dV(it) above has already consumed in order)
                if (it + 1 < n_it) {
                    if (!mbar_wait(&q_full[(it + 1) & 1], ((it + 1) >> 1) & 1, p.w, 0x65)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(it + 1);
                }
                if (!mbar_wait(ds_full, it & 1, p.w, 0x66)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dK += dS^T Q   (A = dS^T K-major, B = Q, d contiguous)
#pragma unroll
                for (int kk = 0; kk < kBM / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                    mma_ss(tdK, desc_sw128(sdS + off, 16, 1024), desc_sw128(sQ + kk * 2048, kChunk, 1024), id_kmn,
                           (it > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&q_empty[slot]);  // dK was the last reader of Q, lse, D and dO of this slot
                // dQ = dS K      (A = dS, query index contiguous; B = K, d contiguous)
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ss(tdP, desc_sw128(sdS + kk * 2048, kChunk, 1024), desc_sw128(sK + kk * 2048, kChunk, 1024),
                           id_mnmn, kk > 0);
                mma_commit(dq_full);
                mma_commit(ds_empty);
            }
            if (!ok)
                *abort_flag = 1;
            mma_commit(dkv_done);
            mma_commit(drain);
            mbar_wait(drain, 0, p.w, 0x6f);
        }
    } else {
        // ------------------------------------------------ compute warps
        // Warp w owns query columns 32*cq .. 32*cq+31 (cq = w / 4) of the key
        // rows in TMEM lane quarter w % 4 (TMEM lane = key row).  It also reads
        // its 32 d-columns of each dQ partial (TMEM lane = query row) and
        // reduces them into the accumulator, and writes dK/dV at the end.
        const int cq = warp >> 2;                  // column quarter
        const int q4 = warp & 3;                   // TMEM lane quarter
        const int j = q4 * 32 + lane;              // key row / dQ query row in the tile
        const int64_t key = kv0 + j;
        int64_t lo = 0, hi = 0;                    // rows that may attend to this key: [lo, hi)
        if (key < p.N) {
            doc_range(p, key, lo, hi);
            if (p.causal)
                lo = key;
        }
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
        const int c0 = cq * 32;                    // first query column / d column of this warp
        // dS^T row j, columns c0..c0+31: four 16-byte units of one 64-column chunk
        uint8_t *ds_row = smem + BwdSmem::kdS + (cq >> 1) * kChunk + j * 128;
        bool ok = true;
        // dQ partial: read out of TMEM (frees the dP/dQ columns), then its 8
        // vector reductions (one per group of 4 columns) are spread over the
        // following work: groups 0-2 while the dP product runs, 3-5 after the
        // dS^T hand-off, 6 at the top of the next iteration and 7 in the middle
        // of its P^T computation.  Pushing 64 KB per iteration through the SM's
        // global-reduction path in bursts stalls the warps that are due on the
        // S -> P -> dV and dP -> dS^T chains; this spacing measured fastest.
        uint32_t xq[32];
        float *dq_base = nullptr;
        auto read_dq = [&](int it) {
            const int h = kvh * p.G + it % p.G;
            const int m = m_lo + it / p.G;
            tmem_ld32p(tdP + lane_off + c0, xq);
            tmem_ld_wait();
            tmem_ld_fence32p(xq);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(dq_empty);
            const int64_t qoff =
                (((static_cast<int64_t>(sb) * p.Hq + h) * (p.Npad / kBM) + m) * 32 + c0 / 4) * (kBM * 4) + j * 4;
            // the eight 4-column groups of this row lie in [qoff, qoff + 7 * 128 * 4 + 4)
            dq_base = (static_cast<int64_t>(m) * kBM + j < p.N &&
                       ULY_IN_BOUNDS(p.w.status, qoff, 7 * kBM * 4 + 4, p.SB * p.Hq * p.Npad * kD, 0x28))
                          ? p.dq_acc + qoff
                          : nullptr;
        };
        auto reduce_groups = [&](int g0, int g1) {  // groups g0 .. g1-1 of 8
            if (dq_base != nullptr) {
#pragma unroll
                for (int g = g0; g < g1; ++g)
                    red_add_v4(dq_base + g * (kBM * 4), __uint_as_float(xq[4 * g]), __uint_as_float(xq[4 * g + 1]),
                               __uint_as_float(xq[4 * g + 2]), __uint_as_float(xq[4 * g + 3]));
            }
        };
        for (int it = 0; it < n_it; ++it) {
            const int slot = it & 1;
            const int64_t q0 = static_cast<int64_t>(m_lo + it / p.G) * kBM;
            const float *lse_s = reinterpret_cast<const float *>(smem + BwdSmem::kLse + slot * 512) + c0;
            const float *D_s = reinterpret_cast<const float *>(smem + BwdSmem::kDv + slot * 512) + c0;
            reduce_groups(6, 7);  // of the partial read in the previous iteration
            if (!mbar_wait_warp(s_full, it & 1, p.w, 0x71) ||
                !mbar_wait_warp(&q_full[slot], (it >> 1) & 1, p.w, 0x72)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t u[32];
            tmem_ld32p(tS + lane_off + c0, u);
            tmem_ld_wait();
            tmem_ld_fence32p(u);
            // P^T = 2^(S^T * scale * log2(e) - lse * log2(e)), 0 where masked
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 l4 = *reinterpret_cast<const float4 *>(lse_s + c);
                const float2 x01 = ffma2(make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sl2,
                                         make_float2(-l4.x, -l4.y));
                const float2 x23 = ffma2(make_float2(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), sl2,
                                         make_float2(-l4.z, -l4.w));
                pk[c / 2] = pack_bf16x2(ex2_approx(x01.x), ex2_approx(x01.y));
                pk[c / 2 + 1] = pack_bf16x2(ex2_approx(x23.x), ex2_approx(x23.y));
                if (c == 12)
                    reduce_groups(7, 8);
            }
            if (!((q0 + c0 >= lo) && (q0 + c0 + 32 <= hi))) {
                // boundary tile for this key: zero the probabilities of rows
                // outside [lo, hi)
                const int lo_c = static_cast<int>(max(min(lo - (q0 + c0), int64_t(32)), int64_t(0)));
                const int hi_c = static_cast<int>(max(min(hi - (q0 + c0), int64_t(32)), int64_t(0)));
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const uint32_t keep_lo = (c >= lo_c && c < hi_c) ? 0x0000ffffu : 0u;
                    const uint32_t keep_hi = (c + 1 >= lo_c && c + 1 < hi_c) ? 0xffff0000u : 0u;
                    pk[c / 2] &= (keep_lo | keep_hi);
                }
            }
            // P^T of these 32 query columns, packed, into S columns c0 .. c0+15
            tmem_st16p(tS + lane_off + c0, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(p_full);
            // the previous iteration's dQ partial (frees the dP/dQ columns)
            if (it > 0) {
                if (!mbar_wait_warp(dq_full, (it - 1) & 1, p.w, 0x73)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                read_dq(it - 1);
                reduce_groups(0, 3);
            } else {
                dq_base = nullptr;
            }
            // dS^T needs the shared buffer the previous dK/dQ products read
            if ((it > 0 && !mbar_wait_warp(ds_empty, (it - 1) & 1, p.w, 0x74)) ||
                !mbar_wait_warp(dp_full, it & 1, p.w, 0x75)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t dp[32];
            tmem_ld32p(tdP + lane_off + c0, dp);
            tmem_ld_wait();
            tmem_ld_fence32p(dp);
            // dS^T = P^T (dP^T - D), packed bf16, into the swizzled row
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                uint32_t dsp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = qd * 8 + 2 * e;
                    const float2 d2 = *reinterpret_cast<const float2 *>(D_s + c);
                    const float2 t = fadd2(make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])),
                                           make_float2(-d2.x, -d2.y));
                    const float2 ds = fmul2(make_float2(bf16lo(pk[c / 2]), bf16hi(pk[c / 2])), t);
                    dsp[e] = pack_bf16x2(ds.x, ds.y);
                }
                const int unit = (cq & 1) * 4 + qd;  // 16-byte unit within the 64-column chunk
                *reinterpret_cast<uint4 *>(ds_row + ((unit ^ (j & 7)) * 16)) =
                    make_uint4(dsp[0], dsp[1], dsp[2], dsp[3]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(ds_full);
            reduce_groups(3, 6);
        }
        if (ok && n_it > 0) {
            if (mbar_wait_warp(dq_full, (n_it - 1) & 1, p.w, 0x76)) {
                tc_fence_after();
                reduce_groups(6, 8);  // the rest of the partial before the last
                read_dq(n_it - 1);
                reduce_groups(0, 8);
            } else {
                ok = false;
            }
        }
        if (!ok)
            *abort_flag = 1;
        // ---- dK, dV epilogue: key row j, d columns c0 .. c0+31 ----
        if (mbar_wait_warp(dkv_done, 0, p.w, 0x78) && ok) {
            tc_fence_after();
            const int64_t rowoff = p.L.off(p.N, sb, key < p.N ? key : 0, p.Hkv, kvh, kD) + c0;
            const bool store = key < p.N && ULY_IN_BOUNDS(p.w.status, rowoff, 32, p.kv_elems, 0x29);
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t src = (which ? tdK : tdV) + lane_off + c0;
                const float f = which ? p.scale : 1.f;
                uint16_t *dst = (which ? p.dk : p.dv) + rowoff;
                uint32_t x[32];
                tmem_ld32p(src, x);  // warp-collective: all lanes
                tmem_ld_wait();
                tmem_ld_fence32p(x);
                uint32_t o16[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    o16[c] = (n_it > 0) ? pack_bf16x2(__uint_as_float(x[2 * c]) * f, __uint_as_float(x[2 * c + 1]) * f)
                                        : 0u;
                if (store) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        reinterpret_cast<uint4 *>(dst)[c] =
                            make_uint4(o16[4 * c], o16[4 * c + 1], o16[4 * c + 2], o16[4 * c + 3]);
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        tmem_dealloc(tbase, 512);
}

}  // namespace

cudaError_t launch_attn_bwd_bf16(const AttnShape &s, const void *q, const void *k, const void *v, const void *o,
                                 const float *lse, const void *dout, void *dq, void *dk, void *dv,
                                 const BwdScratch &scr, cudaStream_t stream)
{
    if (s.d != kD)
        return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv, tdo;
    if (make_rows_map_bf16(&tq, q, s, s.Hq) != CUDA_SUCCESS || make_rows_map_bf16(&tk, k, s, s.Hkv) != CUDA_SUCCESS ||
        make_rows_map_bf16(&tv, v, s, s.Hkv) != CUDA_SUCCESS || make_rows_map_bf16(&tdo, dout, s, s.Hq) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t Npad = scr.Npad;
    cudaError_t e;
    // 1. D, lse*log2(e); 2. zero the dQ accumulator
    {
        const int64_t warps = s.SB * Npad;
        const int64_t blocks = (warps * 32 + 255) / 256;
        bwd_pre_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const uint16_t *>(o), static_cast<const uint16_t *>(dout), lse, scr.lse2, scr.D, s.SB, s.N,
            Npad, s.Hq, s.L, s.q_elems, s.status);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        e = cudaMemsetAsync(scr.dq_acc, 0, static_cast<size_t>(s.SB) * s.Hq * Npad * kD * sizeof(float), stream);
        if (e != cudaSuccess)
            return e;
    }
    // 3. main kernel
    BwdParams p;
    p.SB = s.SB;
    p.N = s.N;
    p.Npad = Npad;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.n_ktiles = static_cast<int>((s.N + kBN - 1) / kBN);
    p.causal = s.causal;
    p.cu = s.cu_dev;
    p.num_docs = s.num_docs;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.scale = s.scale;
    p.lse2 = scr.lse2;
    p.Dv = scr.D;
    p.dq_acc = scr.dq_acc;
    p.dk = static_cast<uint16_t *>(dk);
    p.dv = static_cast<uint16_t *>(dv);
    p.kv_elems = s.kv_elems;
    p.w = wait_cfg();
    p.L = s.L;
    {
        int64_t work = 0, longest = 0;
        for (int n = 0; n < p.n_ktiles; ++n) {
            const int64_t kv0 = static_cast<int64_t>(n) * kBN;
            const int64_t key_last = (kv0 + kBN - 1 < s.N - 1) ? kv0 + kBN - 1 : s.N - 1;
            int64_t row_lo, row_hi, t0, t1;
            doc_range_host(s.cu_host, s.num_docs, s.N, kv0, row_lo, t0);
            doc_range_host(s.cu_host, s.num_docs, s.N, key_last, t1, row_hi);
            if (s.causal)
                row_lo = kv0;
            const int64_t n_it = static_cast<int64_t>(p.G) * ((row_hi - 1) / kBM - row_lo / kBM + 1);
            work += n_it;
            longest = n_it > longest ? n_it : longest;
        }
        p.group = group_for(work, longest, s.SB * s.Hkv);
    }
    const size_t smem = BwdSmem::kTotal;
    p.order = s.order_dev;
    auto kernel = p.order ? attn_bwd_bf16_kernel<2> : p.group > 1 ? attn_bwd_bf16_kernel<1> : attn_bwd_bf16_kernel<0>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    const int64_t units = s.SB * s.Hkv * p.n_ktiles;
    kernel<<<static_cast<unsigned>(units), kThreads, smem, stream>>>(tq, tk, tv, tdo, p);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    // 4. dQ = scale * accumulator -> bf16
    {
        const int64_t blocks = s.SB * s.Hq * (Npad / kBM) * (kBM / kCvtRows);
        dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            scr.dq_acc, static_cast<uint16_t *>(dq), s.SB, s.N, Npad, s.Hq, s.scale, s.L, s.q_elems, s.status);
    }
    return cudaGetLastError();
}

}  // namespace uly
