/*
 * ulysses.h -- C ABI of the GB300 (sm_103a) Ulysses sequence-parallel hot path.
 *
 * The path (Transformers docs "Ulysses sequence parallelism", introduction and
 * its all-to-all diagram; Hugging Face Ulysses blog summary, "How Ulysses
 * Sequence Parallelism Works", steps 3-5):
 *   1. seq->head all-to-all: P sequence shards [N/P, H, d] become P head
 *      shards [N, H/P, d];
 *   2. local attention over every head shard, full sequence, causal, with
 *      GQA K/V sharing and optional packed-document masking; and its
 *      backward;
 *   3. head->seq all-to-all back.
 * On one GPU the P ranks are P virtual ranks: P contiguous shards inside one
 * device allocation, so the all-to-all is a device-local permutation.
 *
 * Conventions for every call:
 *  - Pointers named x_*, q, k, v, o, lse, dout, dq, dk, dv and workspace are
 *    DEVICE pointers owned by the caller; the library never allocates, frees
 *    or keeps them.  Host pointers are marked _host.
 *  - Every pointer must be 16-byte aligned (ULY_ERR_MISALIGNED otherwise).
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *    stream) and never synchronise, except ulysses_get_device_status.
 *  - Arguments are validated on the host before anything is launched; on
 *    failure nothing is launched and the status says why.
 *  - dtype: ULY_BF16 (bf16 storage, fp32 accumulation) or ULY_FP32 (fp32
 *    throughout, the correctness path).
 *  - Layouts are row-major, outermost first:
 *      seq layout  : [P][B][N/P][H][d]   (P contiguous sequence shards)
 *      head layout : [P][B][N][H/P][d]   (P contiguous head shards)
 *      lse         : [S][B][Hq][N] fp32, natural logarithm of the row's sum
 *                    of exp(scaled scores)
 *    where S is the number of head shards an attention call covers.
 *  - Thread safety: calls on different streams with different buffers and
 *    workspaces may run concurrently.  The device status word is shared by
 *    all calls on a device.
 */
#ifndef ULYSSES_H
#define ULYSSES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ULY_OK = 0,
    ULY_ERR_INVALID_ARG = 1, /* a size, count or flag is out of range */
    ULY_ERR_UNSUPPORTED = 2, /* valid for the method, not handled by this library */
    ULY_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
    ULY_ERR_OVERLAP = 4,     /* input and output buffers overlap */
    ULY_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
    ULY_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out */
    ULY_ERR_WORKSPACE = 7,   /* workspace missing or smaller than required */
    ULY_ERR_SCRATCH_LIMIT = 8, /* sizes need more scratch than ulysses_attn_bwd_noalloc has */
    ULY_ERR_BOUNDS = 9        /* a bounds check of the debug build failed (see below) */
} uly_status;

typedef enum { ULY_BF16 = 0, ULY_FP32 = 1 } uly_dtype;

/* ---------------------------------------------------------------- swaps */

/*
 * seq->head all-to-all, emulated over P virtual ranks in one allocation.
 * Source: Transformers docs "Ulysses sequence parallelism", the all-to-all
 * diagram (rank r keeps every token and receives the contiguous head block
 * r); blog summary "How Ulysses Sequence Parallelism Works", step 3.
 *
 *   x_head[r][b][n][h][k] = x_seq[n / (N/P)][b][n % (N/P)][r*H/P + h][k]
 *
 * x_seq  : device, [P][B][N/P][H][d], read only.
 * x_head : device, [P][B][N][H/P][d], fully written.
 * B >= 1, N >= 1 with N % P == 0 (sequences are padded to a multiple of the
 * SP size), H % P == 0 (the number of heads must be divisible by the SP size),
 * 1 <= P <= H, d in {64, 128}.  The two buffers must not overlap.
 * The copy is exact (bit for bit) for either dtype.
 */
uly_status ulysses_seq_to_head(const void *x_seq, void *x_head, int64_t B, int64_t N, int32_t H,
                               int32_t d, int32_t P, uly_dtype dtype, void *stream);

/*
 * head->seq all-to-all: the exact inverse of ulysses_seq_to_head (the second
 * all-to-all of the same diagram; blog summary step 5).  It is also the
 * backward of seq->head, and seq->head is the backward of head->seq.
 *
 *   x_seq[s][b][t][r*H/P + h][k] = x_head[r][b][s*(N/P) + t][h][k]
 *
 * Same argument rules as ulysses_seq_to_head.
 */
uly_status ulysses_head_to_seq(const void *x_head, void *x_seq, int64_t B, int64_t N, int32_t H,
                               int32_t d, int32_t P, uly_dtype dtype, void *stream);

/*
 * A batch of up to four swaps in one launch, e.g. Q, K and V on their way to
 * the head layout (the all-to-all diagram moves them together), dQ, dK and dV
 * on their way back, or O going back while dO comes in.  Every tensor of the
 * batch shares B, N, d, P and dtype; each has its own head count H and its
 * own direction.  The results are those of the single calls, bit for bit.
 *
 * descs_host : host array of n_descs entries (1 <= n_descs <= 4), read before
 *              the call returns:
 *   src, dst : device buffers as in ulysses_seq_to_head (to_head = 1) or
 *              ulysses_head_to_seq (to_head = 0);
 *   H        : the tensor's head count, H % P == 0.
 * Same argument rules as ulysses_seq_to_head for every entry.  In addition no
 * entry's dst may overlap another entry's src or dst (ULY_ERR_OVERLAP): the
 * entries are copied concurrently.
 */
typedef struct {
    const void *src;
    void *dst;
    int32_t H;
    int32_t to_head;
} uly_swap_desc;

uly_status ulysses_swap_batch(const uly_swap_desc *descs_host, int32_t n_descs, int64_t B, int64_t N,
                              int32_t d, int32_t P, uly_dtype dtype, void *stream);

/* ------------------------------------------------------------ attention */

/*
 * Bytes of device workspace ulysses_attn_fwd (for_bwd = 0) or
 * ulysses_attn_bwd (for_bwd = 1) needs for these sizes.  Returns 0 for sizes
 * the call would reject.  num_docs = 0 means one document (no packing).
 */
size_t ulysses_attn_workspace_size(int64_t B, int64_t N, int32_t Hq_local, int32_t Hkv_local,
                                   int32_t d, int32_t num_shards, int32_t num_docs,
                                   int32_t for_bwd, uly_dtype dtype);

/*
 * The order in which the bf16 attention kernels walk the 128-row tiles of
 * a sequence (host only; no device work).  out[0 .. ceil(N/128)) receives
 * every tile index once, longest walk first.  Forward (for_bwd = 0): query
 * tiles, a tile's walk being the key tiles its rows may attend to (their
 * documents' keys, up to the row itself when causal); ties keep the later
 * tile first.  Backward (for_bwd = 1): key tiles, the walk being the query
 * tiles that may attend to the keys; ties keep the earlier tile first.
 * With packed documents a tile's walk follows its place in its document, so
 * the attention calls sort the tiles like this themselves (the order goes
 * into the workspace next to cu_seqlens); without documents the walk only
 * depends on the index and this is the kernels' index order.  Exposed for
 * inspection and tests.
 * out : host, ceil(N/128) int32.
 * Errors: ULY_ERR_INVALID_ARG for out == NULL, N < 1, causal or for_bwd not
 * 0/1, or cu_seqlens the attention calls would reject.
 */
uly_status ulysses_attn_tile_order(int64_t N, int32_t causal, const int32_t *cu_seqlens_host,
                                   int32_t num_docs, int32_t for_bwd, int32_t *out);

/*
 * Attention forward over `num_shards` consecutive head shards (blog summary,
 * step 4 "Local Attention": every rank attends over all N tokens for its
 * heads).  For shard s, batch b, local query head h (local KV head h / G,
 * G = Hq_local / Hkv_local), row i:
 *   s_ij  = softmax_scale * <q_i, k_j>            for allowed j
 *   lse_i = ln sum_j exp(s_ij)
 *   o_i   = sum_j exp(s_ij - lse_i) v_j
 * allowed: j <= i if causal; and doc(i) == doc(j) if cu_seqlens_host is not
 * NULL (packed documents, the block-diagonal mask of FlashAttention-style
 * varlen attention that the Transformers docs recommend for packing).
 *
 * q, o       : device, [num_shards][B][N][Hq_local][d]
 * k, v       : device, [num_shards][B][N][Hkv_local][d]
 * lse        : device fp32, [num_shards][B][Hq_local][N]
 * cu_seqlens_host : host int32 [num_docs + 1], 0 = cu[0] <= cu[1] <= ... <=
 *              cu[num_docs] = N, or NULL (one document).  Copied before return.
 * softmax_scale <= 0 selects 1/sqrt(d).
 * workspace  : device, >= ulysses_attn_workspace_size(..., for_bwd=0) bytes.
 * Requires Hq_local % Hkv_local == 0, d in {64, 128} (bf16: d == 128).
 */
uly_status ulysses_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                            int64_t B, int64_t N, int32_t Hq_local, int32_t Hkv_local, int32_t d,
                            int32_t num_shards, int32_t causal, const int32_t *cu_seqlens_host,
                            int32_t num_docs, float softmax_scale, uly_dtype dtype, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Attention backward (the gradient of ulysses_attn_fwd, which training needs;
 * the Trainer discussion in the blog summary requires the gradients to be
 * correct).  With P_ij = exp(s_ij - lse_i) and D_i = <dO_i, O_i>:
 *   dV_j = sum_i P_ij dO_i
 *   dS_ij = P_ij (<dO_i, v_j> - D_i)
 *   dQ_i = softmax_scale sum_j dS_ij k_j
 *   dK_j = softmax_scale sum_i dS_ij q_i
 * dK and dV are summed over the G query heads sharing a KV head.
 *
 * q, k, v, o, lse : as returned/used by ulysses_attn_fwd (o and lse from it).
 * dout, dq        : device, like q.   dk, dv : device, like k.  All written.
 * workspace       : device, >= ulysses_attn_workspace_size(..., for_bwd=1);
 *                   holds fp32 scratch (D, scaled lse, the dQ accumulator).
 * Other arguments as in ulysses_attn_fwd.
 */
uly_status ulysses_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dout, void *dq, void *dk, void *dv,
                            int64_t B, int64_t N, int32_t Hq_local, int32_t Hkv_local, int32_t d,
                            int32_t num_shards, int32_t causal, const int32_t *cu_seqlens_host,
                            int32_t num_docs, float softmax_scale, uly_dtype dtype, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * The swap -> attention -> swap pipeline without the swaps: attention over all
 * P head shards read straight from the sequence-sharded buffers, outputs
 * written straight back to them.  Same results as
 *   ulysses_seq_to_head(q/k/v) ; ulysses_attn_fwd(num_shards = P) ;
 *   ulysses_head_to_seq(o)
 * because on one device head shard r is just a strided view of the seq
 * buffer (the all-to-all moves data between GPUs; on one GPU it only
 * relabels rows).  Source: as ulysses_seq_to_head and ulysses_attn_fwd.
 *
 * q_seq, o_seq : device, [P][B][N/P][Hq][d]     k_seq, v_seq : [P][B][N/P][Hkv][d]
 * lse          : device fp32, [P][B][Hq/P][N]   (head shard r, local head h)
 * Hq, Hkv are the GLOBAL head counts; H % P == 0 for both (ULY_ERR_INVALID_ARG).
 * bf16 also needs (N/P) % 128 == 0 so that no 128-token tile straddles two
 * sequence shards (ULY_ERR_UNSUPPORTED otherwise).  workspace: as
 * ulysses_attn_workspace_size(B, N, Hq/P, Hkv/P, d, P, num_docs, 0, dtype).
 * Other arguments, validation and errors as ulysses_attn_fwd.
 */
uly_status ulysses_attn_fwd_seq(const void *q_seq, const void *k_seq, const void *v_seq, void *o_seq,
                                float *lse, int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d,
                                int32_t P, int32_t causal, const int32_t *cu_seqlens_host,
                                int32_t num_docs, float softmax_scale, uly_dtype dtype, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Backward of ulysses_attn_fwd_seq: dout_seq in, dq_seq / dk_seq / dv_seq out,
 * all in the sequence-sharded layout (the backward of the swaps is the
 * inverse swap, so no swap is needed here either).  workspace: as
 * ulysses_attn_workspace_size(B, N, Hq/P, Hkv/P, d, P, num_docs, 1, dtype).
 */
uly_status ulysses_attn_bwd_seq(const void *q_seq, const void *k_seq, const void *v_seq,
                                const void *o_seq, const float *lse, const void *dout_seq,
                                void *dq_seq, void *dk_seq, void *dv_seq, int64_t B, int64_t N,
                                int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int32_t causal,
                                const int32_t *cu_seqlens_host, int32_t num_docs, float softmax_scale,
                                uly_dtype dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * ulysses_attn_bwd without a workspace, for callers that cannot allocate
 * device memory: code running inside an allocator's own hooks, a process
 * whose device memory pool is fixed up front, a plugin that is handed only
 * the tensors it works on, or a latency-critical path that must not take the
 * allocator's locks.  The pages have no counterpart: the method itself does
 * not care where scratch lives.
 *
 * Same arguments and results as ulysses_attn_bwd, minus workspace.  The fp32
 * scratch (lse*log2(e), D, the dQ accumulator, the cu_seqlens copy) lives in
 * one fixed 64 MiB device array inside the library; every GPU that loads
 * this part of the library holds those 64 MiB until the process exits.
 * Sizes whose scratch (ulysses_attn_workspace_size(..., for_bwd=1, ...))
 * exceeds 64 MiB return ULY_ERR_SCRATCH_LIMIT and launch nothing; for bf16
 * that is about 129,000 (shard x batch x query-head x padded-row) rows, e.g.
 * N = 8192 with 8 local query heads and 1 shard fits.
 * The call itself makes no cudaMalloc and calls no allocating library
 * routine.  The array is part of the library's device code, which the CUDA
 * runtime loads onto a device lazily: the first call on each device looks up
 * the array's device address, and that lookup loads the module, so the
 * driver reserves the 64 MiB (and the module's code) inside that first call.
 * A caller whose restricted context cannot afford that reservation (a fixed
 * pool with its memory already committed, an allocator hook) must make the
 * first call on each device outside that context, at start-up, and also
 * before any stream capture; later calls reserve nothing.
 * stream and every pointer must belong to the CURRENT device (the scratch
 * address is the current device's).  After cudaDeviceReset the cached
 * address is stale: do not call this entry point again in that process.
 * All calls share the array: calls that overlap on the GPU (other streams,
 * other threads) race and must not be issued; sequential calls are safe
 * because each one rewrites or clears every scratch byte it reads.
 */
uly_status ulysses_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                    const float *lse, const void *dout, void *dq, void *dk, void *dv,
                                    int64_t B, int64_t N, int32_t Hq_local, int32_t Hkv_local,
                                    int32_t d, int32_t num_shards, int32_t causal,
                                    const int32_t *cu_seqlens_host, int32_t num_docs,
                                    float softmax_scale, uly_dtype dtype, void *stream);

/* --------------------------------------------------------- ring attention */

/*
 * Ring attention over P virtual ranks, the pages' alternative to Ulysses
 * ("Sequence Parallelism for Long-Context AI Training", "Advanced Scaling:
 * Ring Attention and Ulysses"; blog summary, "Comparing Ulysses and Ring
 * Attention"): rank r keeps its chunk of Q for ALL heads and the K/V chunks
 * travel round the ring; in P steps every query chunk meets every key chunk
 * (step k: query chunk r with key chunk (r - k) mod P; causal keeps only
 * r >= k after step 0), and the partial results are merged through their
 * log-sum-exp.  The result equals causal attention over all N tokens, i.e.
 * the same as the Ulysses path, without any head sharding.
 *
 * q_seq, o_seq, dout_seq, dq_seq : device, [P][B][N/P][Hq][d]
 * k_seq, v_seq, dk_seq, dv_seq   : device, [P][B][N/P][Hkv][d]
 * lse : device fp32, [P][B][Hq][N/P] (chunk, batch, head, position in chunk)
 * Hq, Hkv are the total head counts (ring attention does not shard heads).
 * N % P == 0; otherwise the rules of ulysses_attn_fwd on each chunk
 * (N/P tokens), without packed documents.
 * workspace : device, >= ulysses_ring_attn_workspace_size(..., for_bwd).
 * The backward uses the final o and lse of the forward.
 */
size_t ulysses_ring_attn_workspace_size(int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d,
                                        int32_t P, int32_t for_bwd, uly_dtype dtype);
uly_status ulysses_ring_attn_fwd(const void *q_seq, const void *k_seq, const void *v_seq, void *o_seq,
                                 float *lse, int64_t B, int64_t N, int32_t Hq, int32_t Hkv, int32_t d,
                                 int32_t P, int32_t causal, float softmax_scale, uly_dtype dtype,
                                 void *workspace, size_t workspace_bytes, void *stream);
uly_status ulysses_ring_attn_bwd(const void *q_seq, const void *k_seq, const void *v_seq,
                                 const void *o_seq, const float *lse, const void *dout_seq,
                                 void *dq_seq, void *dk_seq, void *dv_seq, int64_t B, int64_t N,
                                 int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int32_t causal,
                                 float softmax_scale, uly_dtype dtype, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* -------------------------------------------------------- sharded loss */

/* Bytes of device workspace ulysses_sharded_ce_loss needs (0 if invalid). */
size_t ulysses_sharded_ce_workspace_size(int64_t B, int64_t N, int32_t P);

/*
 * Next-token cross entropy of a sequence-parallel batch and its
 * good-token-weighted aggregation across the P ranks (Accelerate PR
 * "Deepspeed Ulysses/ALST integration", user API step 2: shift_labels, the
 * per-rank loss, all_gather of losses and good-token counts, then
 * sum_r loss_r * good_r / max(sum_r good_r, 1); the Transformers docs list
 * label shifting and loss aggregation among what the Trainer does for SP).
 *
 * Labels are shifted over the WHOLE sequence before sharding: the target of
 * the last token of rank r's chunk is the first label of rank r+1's chunk;
 * the last token of each sequence gets -100 (ignored).
 *
 * logits     : device, [P][B][N/P][V] (each rank's LM-head output), read.
 * labels     : device int64, [P][B][N/P], unshifted; -100 = ignored.  Values
 *              outside [0, V) other than -100 are ignored and reported as
 *              ULY_ERR_INVALID_ARG by ulysses_get_device_status.
 * dlogits    : device, like logits, or NULL.  If given, receives
 *              d total_loss / d logits = (softmax - onehot(target)) / max(T, 1)
 *              on good rows and 0 on ignored rows (T = all good tokens).
 * shard_loss : device fp32 [P]: rank r's mean CE over its good tokens (0 if none).
 * shard_good : device int64 [P]: rank r's good-token count.
 * total_loss : device fp32 [1]: the aggregated loss.
 * workspace  : device, >= ulysses_sharded_ce_workspace_size(B, N, P).
 * N % P == 0 (sequences padded to a multiple of the SP size).
 */
uly_status ulysses_sharded_ce_loss(const void *logits, const int64_t *labels, void *dlogits,
                                   float *shard_loss, int64_t *shard_good, float *total_loss,
                                   int64_t B, int64_t N, int32_t V, int32_t P, uly_dtype dtype,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------ diagnostics */

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  ULY_OK if no kernel reported a problem since the last read;
 * ULY_ERR_TIMEOUT if a bounded device-side wait ran out (the kernel then
 * stopped early and its outputs are invalid); ULY_ERR_BOUNDS if a kernel of
 * the debug build found an access outside its buffer (it skipped the access;
 * outputs are invalid); ULY_ERR_INVALID_ARG if a kernel rejected its launch
 * configuration; ULY_ERR_CUDA on a CUDA error.  If site_out is not NULL it
 * receives the id of the first site that reported (a wait, or 0x8000 plus
 * the id of an access).
 */
uly_status ulysses_get_device_status(void *stream, uint32_t *site_out);

/*
 * Sets the per-wait limit (nanoseconds, >= 1000) of every bounded device
 * wait launched afterwards by this process.  Default: 2 s.
 */
uly_status ulysses_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Launches one tiny kernel whose mbarrier wait can never complete (nothing
 * arrives on it), with a limit of limit_ns.  The wait gives up, records
 * ULY_ERR_TIMEOUT in the device status word and the kernel returns.  Used by
 * tests of the timeout path; it faults nothing and hangs nothing.
 */
uly_status ulysses_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/*
 * Debug build only (the library compiled with -DULY_DEBUG, which checks every
 * raw-pointer global access of the swap and attention kernels against its
 * buffer and reports ULY_ERR_BOUNDS instead of making it): launches one tiny
 * kernel whose check is given an offset past its extent, touching no memory,
 * so that the reporting path can be tested.  The release build returns
 * ULY_ERR_UNSUPPORTED and launches nothing.
 */
uly_status ulysses_selftest_bounds(void *stream);

/* Human-readable name of a status code (static string). */
const char *ulysses_status_string(uly_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t ulysses_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ULYSSES_H */
