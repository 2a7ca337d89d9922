// Causal / packed-document GQA attention forward, bf16 in, fp32 accumulate,
// on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), head_dim 128.
//
// Computes, for every Ulysses head shard (blog summary step 4, "Local
// Attention"): s_ij = scale <q_i, k_j>, lse_i = ln sum_j exp(s_ij),
// o_i = sum_j exp(s_ij - lse_i) v_j over allowed j (j <= i if causal; same
// document if cu_seqlens is given).  The softmax is evaluated online over key
// tiles (FlashAttention's rescaling, which the Transformers docs recommend as
// the attention backend), so nothing quadratic is ever stored.
//
// One CTA = one 128-row query block of TWO query heads of the same GQA group
// (both attend to the same K/V rows with the same mask), so every K/V tile that
// TMA brings in is used by two MMAs.  Warp roles (320 threads):
//   warps 0-3 : softmax for head h0 (thread = row = TMEM lane)
//   warps 4-7 : softmax for head h1
//   warp  8   : TMA producer (Q once, then K_j, V_j into a 4-slot ring)
//   warp  9   : tcgen05.mma issuer (one thread) and TMEM owner
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  P (bf16) is
// written over the first 64 columns of S and fed to the PV product straight
// from TMEM.  O is rescaled in TMEM only when the running row maximum grows by
// more than 2^8 (lazy rescaling), so P stays below 256.  A tile's exponentials
// are first taken against the running maximum without computing the tile's
// own maximum; their sum proves whether the lazy rule keeps that maximum, and
// only when it may not (or on a row's first tile) is the tile redone exactly.
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile
constexpr int kD = 128;           // head dim
constexpr int kSlots = 4;         // K/V ring slots
constexpr int kTileBytes = kBM * kD * 2;  // 32 KB
constexpr int kChunk = kBM * 64 * 2;      // one 64-column swizzled chunk: 16 KB
constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdSmem {
    // data (1024-aligned offsets from the aligned base)
    static constexpr int kQ0 = 0;
    static constexpr int kQ1 = kTileBytes;
    static constexpr int kSlot0 = 2 * kTileBytes;
    static constexpr int kBars = kSlot0 + kSlots * kTileBytes;
    static constexpr int kTotal = kBars + 256;
};

struct FwdParams {
    int64_t SB, N;
    int Hq, Hkv, G, npairs, n_qtiles;
    int causal;
    const int32_t *cu;
    int num_docs;
    float scale_log2;
    float *lse;
    int64_t lse_elems;  // extent for the bounds checks of debug builds
    const int32_t *order;        // with documents: query tiles, longest walk first
    WaitCfg w;
    RowLayout L;
};

__device__ __forceinline__ void doc_range(const FwdParams &p, int64_t i, int64_t &lo, int64_t &hi)
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

template <bool kOrdered>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         FwdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + FwdSmem::kBars);
    uint64_t *q_full = bars + 0;
    uint64_t *kv_full = bars + 1;             // [kSlots]
    uint64_t *kv_empty = bars + 1 + kSlots;   // [kSlots]
    uint64_t *s_full = bars + 1 + 2 * kSlots; // [2]
    uint64_t *p_full = s_full + 2;            // [2]
    uint64_t *o_done = p_full + 2;            // [1]
    uint64_t *drain = o_done + 1;             // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id();
    const int lane = lane_id();

    // ---- work unit: problem-major (resident CTAs share one (shard*batch,
    // KV head) problem and stream the same K/V tiles through L2), longest
    // query blocks first within a problem: the last blocks without documents,
    // the host's order with them ----
    const int64_t u = blockIdx.x;
    const int pair = static_cast<int>(u % p.npairs);
    const int rank = static_cast<int>((u / p.npairs) % p.n_qtiles);
    const int m_blk = kOrdered ? p.order[rank] : p.n_qtiles - 1 - rank;
    const int64_t prob = u / (static_cast<int64_t>(p.npairs) * p.n_qtiles);
    const int kvh = static_cast<int>(prob % p.Hkv);
    const int sb = static_cast<int>(prob / p.Hkv);
    const int h0 = kvh * p.G + 2 * pair;
    const bool has1 = (2 * pair + 1) < p.G;
    const int64_t q0 = static_cast<int64_t>(m_blk) * kBM;
    const int64_t row_last = (q0 + kBM - 1 < p.N - 1) ? q0 + kBM - 1 : p.N - 1;
    int64_t key_lo, key_hi, dlo, dhi;
    doc_range(p, q0, key_lo, dhi);
    doc_range(p, row_last, dlo, key_hi);
    if (p.causal)
        key_hi = row_last + 1;
    const int kt_lo = static_cast<int>(key_lo / kBN);
    const int n_kv = static_cast<int>((key_hi - 1) / kBN) - kt_lo + 1;

    if (warp == 8 && lane == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);  // one elected arrival per softmax warp
        }
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp == 8) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_o);
            mbar_expect_tx(q_full, has1 ? 2 * kTileBytes : kTileBytes);
            int c1, c2, c3, c4;
            p.L.tile(sb, q0, p.Hq, h0, c1, c2, c3, c4);
            tma_load_5d(smem + FwdSmem::kQ0, &tm_q, q_full, 0, c1, c2, c3, c4);
            tma_load_5d(smem + FwdSmem::kQ0 + kChunk, &tm_q, q_full, 64, c1, c2, c3, c4);
            if (has1) {
                p.L.tile(sb, q0, p.Hq, h0 + 1, c1, c2, c3, c4);
                tma_load_5d(smem + FwdSmem::kQ1, &tm_q, q_full, 0, c1, c2, c3, c4);
                tma_load_5d(smem + FwdSmem::kQ1 + kChunk, &tm_q, q_full, 64, c1, c2, c3, c4);
            }
            int issued = 0;
            for (int j = 0; j < n_kv && !*abort_flag; ++j) {
                const int key0 = (kt_lo + j) * kBN;
                bool ok = true;
                for (int which = 0; which < 2; ++which) {
                    const int it = 2 * j + which;
                    const int slot = it % kSlots;
                    if (!mbar_wait(&kv_empty[slot], ((it / kSlots) & 1) ^ 1, p.w, 0x21)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = smem + FwdSmem::kSlot0 + slot * kTileBytes;
                    const CUtensorMap *tm = which ? &tm_v : &tm_k;
                    mbar_expect_tx(&kv_full[slot], kTileBytes);
                    p.L.tile(sb, key0, p.Hkv, kvh, c1, c2, c3, c4);
                    tma_load_5d(dst, tm, &kv_full[slot], 0, c1, c2, c3, c4);
                    tma_load_5d(dst + kChunk, tm, &kv_full[slot], 64, c1, c2, c3, c4);
                    ++issued;
                }
                if (!ok) {
                    *abort_flag = 1;
                    break;
                }
            }
            if (*abort_flag) {
                // wait (bounded) for every load this thread started
                mbar_wait(q_full, 0, p.w, 0x2f);
                for (int it = (issued > kSlots ? issued - kSlots : 0); it < issued; ++it)
                    mbar_wait(&kv_full[it % kSlots], (it / kSlots) & 1, p.w, 0x2f);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16(kBM, kBN, false, false);
            const uint32_t idesc_pv = idesc_bf16(kBM, kD, false, true);
            const uint32_t sQ[2] = {smem_u32(smem + FwdSmem::kQ0), smem_u32(smem + FwdSmem::kQ1)};
            const uint32_t sSlot0 = smem_u32(smem + FwdSmem::kSlot0);
            const int ntile = has1 ? 2 : 1;
            auto issue_qk = [&](int t, int slot) {
                const uint32_t kaddr = sSlot0 + slot * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                    mma_ss(tbase + t * 128, desc_sw128(sQ[t] + off, 16, 1024), desc_sw128(kaddr + off, 16, 1024),
                           idesc_qk, kk > 0);
                }
                mma_commit(&s_full[t]);
            };
            auto issue_pv = [&](int t, int slot, bool acc) {
                const uint32_t vaddr = sSlot0 + slot * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tbase + 256 + t * 128, tbase + t * 128 + kk * 8,
                           desc_sw128(vaddr + kk * 16 * 128, kChunk, 1024), idesc_pv, (acc || kk > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(q_full, 0, p.w, 0x31) && mbar_wait(&kv_full[0], 0, p.w, 0x32);
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < ntile; ++t)
                    issue_qk(t, 0);
                mma_commit(&kv_empty[0]);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int itV = 2 * j + 1, itK = 2 * j + 2;
                const int slotV = itV % kSlots, slotK = itK % kSlots;
                const bool more = j + 1 < n_kv;
                if (!mbar_wait(&kv_full[slotV], (itV / kSlots) & 1, p.w, 0x33) ||
                    !mbar_wait(&p_full[0], j & 1, p.w, 0x34)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(0, slotV, j > 0);
                if (more) {
                    if (!mbar_wait(&kv_full[slotK], (itK / kSlots) & 1, p.w, 0x35)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_qk(0, slotK);
                }
                if (has1) {
                    if (!mbar_wait(&p_full[1], j & 1, p.w, 0x36)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(1, slotV, j > 0);
                }
                mma_commit(&kv_empty[slotV]);
                if (more) {
                    if (has1)
                        issue_qk(1, slotK);
                    mma_commit(&kv_empty[slotK]);
                }
            }
            if (!ok)
                *abort_flag = 1;
            mma_commit(o_done);
            mma_commit(drain);
            mbar_wait(drain, 0, p.w, 0x3f);
        }
    } else {
        // ------------------------------------------------ softmax warpgroups
        const int t = warp >> 2;  // tile 0 or 1
        const int wq = warp & 3;  // TMEM lane quarter
        const int r = wq * 32 + lane;
        const int64_t row = q0 + r;
        if (t == 0 || has1) {
            const int h = h0 + t;
            int64_t lo, hi;
            doc_range(p, row < p.N ? row : p.N - 1, lo, hi);
            if (p.causal && row + 1 < hi)
                hi = row + 1;
            const uint32_t tS = tbase + t * 128 + (static_cast<uint32_t>(wq * 32) << 16);
            const uint32_t tO = tbase + 256 + t * 128 + (static_cast<uint32_t>(wq * 32) << 16);
            float m = -INFINITY, l = 0.f;
            uint32_t u[kBN];  // S row, then P row (fp32 bit patterns)
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                if (!mbar_wait_warp(&s_full[t], j & 1, p.w, 0x41 + t)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < kBN; cb += 32)
                    tmem_ld32p(tS + cb, u + cb);
                tmem_ld_wait();
#pragma unroll
                for (int cb = 0; cb < kBN; cb += 32)
                    tmem_ld_fence32p(u + cb);
                const int64_t key0 = static_cast<int64_t>(kt_lo + j) * kBN;
                const bool masked = key0 < lo || key0 + kBN > hi;
                // no key of this tile is allowed for this row (a row of a later
                // document in a query tile that straddles a document boundary)
                const bool row_empty = key0 >= hi || key0 + kBN <= lo;
                if (masked) {
                    // allowed columns of this tile: [lo_c, hi_c)
                    const int lo_c = static_cast<int>(max(lo - key0, int64_t(0)));
                    const int hi_c = static_cast<int>(min(hi - key0, int64_t(kBN)));
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c < lo_c || c >= hi_c)
                            u[c] = __float_as_uint(-INFINITY);
                }
                // Speculate that the running maximum m still holds: the tile's
                // exponentials against m all stay <= 2^8 exactly when the lazy
                // rescale rule would keep m, and their sum <= 2^8 proves it.  On
                // a row's first tile with an allowed key, or when the sum says the
                // maximum may have grown, the tile is redone exactly from S, still
                // in TMEM.  A row that has seen no allowed key yet and has none in
                // this tile either takes the speculative pass against 0: all its
                // scores are -inf, its exponentials exactly 0.
                const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
                float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                const bool first = __any_sync(0xffffffffu, m == -INFINITY && !row_empty);
                if (!first) {
                    // p = 2^(s * scale * log2(e) - m) on the SFU (masked scores are
                    // -inf and give exactly 0); the scale-and-shift and the row sum
                    // run as packed f32x2 pairs, the sum in four independent chains
                    const float m_ref = (m == -INFINITY) ? 0.f : m;
                    const float2 nm2 = make_float2(-m_ref, -m_ref);
#pragma unroll
                    for (int c = 0; c < kBN; c += 2) {
                        const float2 x = ffma2(make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sl2, nm2);
                        const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                        rs2[(c >> 1) & 3] = fadd2(rs2[(c >> 1) & 3], pv);
                        u[c] = __float_as_uint(pv.x);
                        u[c + 1] = __float_as_uint(pv.y);
                    }
                }
                float rsum;
                {
                    const float2 r01 = fadd2(rs2[0], rs2[1]), r23 = fadd2(rs2[2], rs2[3]);
                    const float2 r = fadd2(r01, r23);
                    rsum = r.x + r.y;
                }
                float alpha = 1.f;
                bool rescale = false;
                if (kOrdered && first) {
                    // a row's first tile (with documents these are frequent: rows
                    // of a later document in a tile that straddles a boundary
                    // meet their first allowed key late): S, masked above, is
                    // still in registers; its row maximum, then the exponentials
                    // against it.  Bit-identical to the redo below; compiled into
                    // the documents instance only, where it is 3 % faster (the
                    // instance without documents ran 1 % slower with it)
                    float pm[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pm[e] = -INFINITY;
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        pm[c & 7] = fmaxf(pm[c & 7], __uint_as_float(u[c]));
                    const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                           fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
                    const float m_cand = mx * p.scale_log2;
                    if (m_cand > m + kRescaleThreshold) {
                        alpha = ex2_approx(m - m_cand);
                        rescale = (j > 0) && (m != -INFINITY);
                        m = m_cand;
                    }
                    const float m_use = (m == -INFINITY) ? 0.f : m;
                    const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        rs2[e] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t pk[32];
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            const float2 x = ffma2(make_float2(__uint_as_float(u[half * 64 + c]),
                                                               __uint_as_float(u[half * 64 + c + 1])),
                                                   sl2, nm2);
                            const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            rs2[(c >> 1) & 3] = fadd2(rs2[(c >> 1) & 3], pv);
                            pk[c >> 1] = pack_bf16x2(pv.x, pv.y);
                        }
                        tmem_st32p(tS + half * 32, pk);
                    }
                    const float2 r01 = fadd2(rs2[0], rs2[1]), r23 = fadd2(rs2[2], rs2[3]);
                    const float2 r = fadd2(r01, r23);
                    rsum = r.x + r.y;
                } else if (first || __any_sync(0xffffffffu, !(rsum <= 256.f))) {
                    // exact: row maximum of S, then the exponentials, 64 columns at a time
                    float pm[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pm[e] = -INFINITY;
                    const int lo_c = masked ? static_cast<int>(max(lo - key0, int64_t(0))) : 0;
                    const int hi_c = masked ? static_cast<int>(min(hi - key0, int64_t(kBN))) : kBN;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[64];
                        tmem_ld32p(tS + half * 64, v);
                        tmem_ld32p(tS + half * 64 + 32, v + 32);
                        tmem_ld_wait();
                        tmem_ld_fence32p(v);
                        tmem_ld_fence32p(v + 32);
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const int cg = half * 64 + c;
                            const float sv = (cg < lo_c || cg >= hi_c) ? -INFINITY : __uint_as_float(v[c]);
                            pm[c & 7] = fmaxf(pm[c & 7], sv);
                        }
                    }
                    const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                           fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
                    const float m_cand = mx * p.scale_log2;
                    if (m_cand > m + kRescaleThreshold) {
                        alpha = ex2_approx(m - m_cand);
                        rescale = (j > 0) && (m != -INFINITY);
                        m = m_cand;
                    }
                    const float m_use = (m == -INFINITY) ? 0.f : m;
                    const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        rs2[e] = make_float2(0.f, 0.f);
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[64];
                        tmem_ld32p(tS + half * 64, v);
                        tmem_ld32p(tS + half * 64 + 32, v + 32);
                        tmem_ld_wait();
                        tmem_ld_fence32p(v);
                        tmem_ld_fence32p(v + 32);
                        uint32_t pk[32];
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            const int cg = half * 64 + c;
                            const float s0 = (cg < lo_c || cg >= hi_c) ? -INFINITY : __uint_as_float(v[c]);
                            const float s1 = (cg + 1 < lo_c || cg + 1 >= hi_c) ? -INFINITY : __uint_as_float(v[c + 1]);
                            const float2 x = ffma2(make_float2(s0, s1), sl2, nm2);
                            const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            rs2[(c >> 1) & 3] = fadd2(rs2[(c >> 1) & 3], pv);
                            pk[c >> 1] = pack_bf16x2(pv.x, pv.y);
                        }
                        // P of S columns half*64.. lands on S columns this thread has read
                        tmem_st32p(tS + half * 32, pk);
                    }
                    const float2 r01 = fadd2(rs2[0], rs2[1]), r23 = fadd2(rs2[2], rs2[3]);
                    const float2 r = fadd2(r01, r23);
                    rsum = r.x + r.y;
                } else {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t pk[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            pk[c] = pack_bf16x2(__uint_as_float(u[half * 64 + 2 * c]),
                                                __uint_as_float(u[half * 64 + 2 * c + 1]));
                        tmem_st32p(tS + half * 32, pk);
                    }
                }
                l = l * alpha + rsum;
                if (__any_sync(0xffffffffu, rescale)) {
                    const float a = rescale ? alpha : 1.f;
#pragma unroll
                    for (int cb = 0; cb < kD; cb += 32) {
                        uint32_t o32[32];
                        tmem_ld32p(tO + cb, o32);
                        tmem_ld_wait();
                        tmem_ld_fence32p(o32);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o32[c] = __float_as_uint(__uint_as_float(o32[c]) * a);
                        tmem_st32p(tO + cb, o32);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[t]);
            }
            if (!ok)
                *abort_flag = 1;
            // O epilogue: row r, normalised to bf16, into this head's Q tile
            // (free once o_done has seen every product complete) in the
            // 128-byte swizzled layout of the tensor map, then one thread
            // stores the 128-row tile with two TMA copies (rows past the end
            // are clipped by the map).  One thread per row writing its own
            // 256 bytes would send 32 rows through every warp-wide store.
            const bool have_o = mbar_wait_warp(o_done, 0, p.w, 0x48 + t) && ok;
            uint8_t *stage = smem + (t ? FwdSmem::kQ1 : FwdSmem::kQ0);
            if (have_o) {
                tc_fence_after();
                const float inv = 1.f / l;
#pragma unroll
                for (int cb = 0; cb < kD; cb += 32) {
                    uint32_t o32[32];
                    tmem_ld32p(tO + cb, o32);
                    tmem_ld_wait();
                    tmem_ld_fence32p(o32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int unit = cb / 8 + q;  // 16-byte unit of the row, 0..15
                        const uint4 val = make_uint4(
                            pack_bf16x2(__uint_as_float(o32[8 * q]) * inv, __uint_as_float(o32[8 * q + 1]) * inv),
                            pack_bf16x2(__uint_as_float(o32[8 * q + 2]) * inv, __uint_as_float(o32[8 * q + 3]) * inv),
                            pack_bf16x2(__uint_as_float(o32[8 * q + 4]) * inv, __uint_as_float(o32[8 * q + 5]) * inv),
                            pack_bf16x2(__uint_as_float(o32[8 * q + 6]) * inv, __uint_as_float(o32[8 * q + 7]) * inv));
                        *reinterpret_cast<uint4 *>(stage + (unit >> 3) * kChunk + r * 128 +
                                                   (((unit & 7) ^ (r & 7)) << 4)) = val;
                    }
                }
                fence_async_smem();
                if (row < p.N) {
                    const int64_t li = (static_cast<int64_t>(sb) * p.Hq + h) * p.N + row;
                    if (ULY_IN_BOUNDS(p.w.status, li, 1, p.lse_elems, 0x12))
                        p.lse[li] = (m + __log2f(l)) * 0.69314718055994530942f;
                }
            }
            named_bar_sync(1 + t, 128);  // the head's four warps have staged their rows
            if (r == 0 && have_o) {
                int c1, c2, c3, c4;
                p.L.tile(sb, q0, p.Hq, h, c1, c2, c3, c4);
                tma_store_5d(&tm_o, stage, 0, c1, c2, c3, c4);
                tma_store_5d(&tm_o, stage + kChunk, 64, c1, c2, c3, c4);
                bulk_commit();
                bulk_wait_read<0>();  // the tile is read before the CTA's shared memory goes
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9)
        tmem_dealloc(tbase, 512);
}

}  // namespace

CUresult make_rows_map_bf16(CUtensorMap *map, const void *base, const AttnShape &s, int H)
{
    // head layout: [S][B][N][H][d]; seq layout: [P][B][N/P][P*H][d]
    const int64_t B = s.L.B;
    const int64_t outer = s.L.seq ? s.L.P : s.SB / B;
    const int64_t T = s.L.seq ? s.L.Np : s.N;
    const int64_t Hd = s.L.seq ? static_cast<int64_t>(H) * s.L.P : H;
    cuuint64_t dims[5] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(Hd), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(B), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[4] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(Hd) * kD * 2,
                             static_cast<cuuint64_t>(T) * Hd * kD * 2, static_cast<cuuint64_t>(B) * T * Hd * kD * 2};
    cuuint32_t box[5] = {64, 1, kBM, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return tensor_map_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

cudaError_t launch_attn_fwd_bf16(const AttnShape &s, const void *q, const void *k, const void *v, void *o,
                                 float *lse, cudaStream_t stream)
{
    if (s.d != kD)
        return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv, to;
    if (make_rows_map_bf16(&tq, q, s, s.Hq) != CUDA_SUCCESS || make_rows_map_bf16(&tk, k, s, s.Hkv) != CUDA_SUCCESS ||
        make_rows_map_bf16(&tv, v, s, s.Hkv) != CUDA_SUCCESS || make_rows_map_bf16(&to, o, s, s.Hq) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    FwdParams p;
    p.SB = s.SB;
    p.N = s.N;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.npairs = (p.G + 1) / 2;
    p.n_qtiles = static_cast<int>((s.N + kBM - 1) / kBM);
    p.causal = s.causal;
    p.cu = s.cu_dev;
    p.num_docs = s.num_docs;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.lse = lse;
    p.lse_elems = s.lse_elems;
    p.w = wait_cfg();
    p.L = s.L;
    p.order = s.order_dev;
    const int64_t units = p.SB * p.Hkv * p.npairs * p.n_qtiles;
    const size_t smem = FwdSmem::kTotal + 1024;
    auto kernel = p.order ? attn_fwd_bf16_kernel<true> : attn_fwd_bf16_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    kernel<<<static_cast<unsigned>(units), kThreads, smem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

}  // namespace uly
