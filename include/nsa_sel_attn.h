/*
 * nsa_sel_attn.h -- C ABI of the GB300 (sm_103a) selected-attention library.
 *
 * Native Sparse Attention's selected-attention (token-selection) branch: every
 * query token of a GQA group attends, causally, only to the T KV blocks of B_K
 * keys that the selection tensor names for it, with one softmax over the union
 * of those keys ("FSA: An Alternative Efficient Implementation of Native Sparse
 * Attention Kernel", key designs 1-4; Flash-Sparse-Attention README, "Method").
 *
 * Conventions for every entry point
 *   - Pointers named q, k, v, out, lse, dout, dq, dk, dv, sel_idx, cu_seqlens and
 *     workspace are DEVICE pointers unless the name says host_.  The caller owns
 *     every buffer and the stream; the library allocates no device memory.
 *   - Calls are asynchronous on `stream` and never synchronise it, except
 *     nsa_sel_attn_get_status, nsa_sel_attn_profile_collect and the host-buffer
 *     entry nsa_sel_attn_step_host, which say so.
 *   - Arguments are validated before anything is enqueued; a failing check
 *     returns an error and writes nothing.  A CUDA launch error is returned as
 *     NSA_ERR_CUDA.  Nothing aborts or exits.
 *   - Layouts (all contiguous, row-major; packed variable-length batch of S
 *     sequences concatenated along tokens, N = cu_seqlens[S]):
 *       q, out, dout, dq   [N, h_q, head_dim]   (dtype)
 *       k, v, dk, dv       [N, h_k, head_dim]   (dtype)
 *       sel_idx            int32 [h_k, N, topk] block indices local to the token's sequence
 *       cu_seqlens         int32 [S + 1], cu_seqlens[0] = 0, non-decreasing
 *       lse                float32 [h_q, N], natural log, softmax scale included
 *     Query head hq uses KV head hq / (h_q / h_k).  q/k/v/out/dout/dq/dk/dv must be
 *     16-byte aligned; the workspace 256-byte aligned.
 *   - Selection semantics: for token t at position tau of its sequence, slot value b
 *     counts when 0 <= b <= tau / B_K (causal) and b < ceil(len / B_K); -1 marks an
 *     empty slot; duplicates count once; keys b*B_K + i > tau are masked.  Values
 *     below -1 or past the sequence's last block are skipped and also raise the
 *     NSA_DEVERR_BAD_INDEX bit of the device status word.  A token with no valid
 *     block gets out = 0 and lse = -inf.
 *   - Supported envelope: dtype bf16 or fp16; head_dim in {64, 128, 256}
 *     (backward: 128); block_size in {32, 64, 128}; 1 <= topk <= 32;
 *     h_q a multiple of h_k; h_k * N * topk < 2^31.  Anything else returns
 *     NSA_ERR_UNSUPPORTED.
 */
#ifndef NSA_SEL_ATTN_H
#define NSA_SEL_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NSA_API __attribute__((visibility("default")))
#else
#define NSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nsa_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
    NSA_OK = 0,
    NSA_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, misaligned buffer */
    NSA_ERR_UNSUPPORTED = 2,   /* outside the supported envelope above */
    NSA_ERR_WORKSPACE = 3,     /* workspace smaller than nsa_sel_attn_workspace_size */
    NSA_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    NSA_ERR_BAD_INDEX = 5,     /* nsa_sel_attn_get_status: device saw invalid sel_idx/cu_seqlens */
    NSA_ERR_TIMEOUT = 6        /* nsa_sel_attn_get_status: a bounded device wait gave up */
} nsa_status;

typedef enum { NSA_BF16 = 0, NSA_FP16 = 1 } nsa_dtype;

/* Bits of the device status word (read by nsa_sel_attn_get_status). */
enum {
    NSA_DEVERR_BAD_INDEX = 1,     /* sel_idx value < -1 or past the sequence's last block */
    NSA_DEVERR_BAD_SEQLENS = 2,   /* cu_seqlens not starting at 0 / decreasing / not ending at N */
    NSA_DEVERR_TIMEOUT = 4        /* an mbarrier wait hit its iteration limit */
};

typedef struct {
    int32_t num_seqs;      /* S >= 1 */
    int32_t total_tokens;  /* N = cu_seqlens[S] (checked on the device) */
    int32_t h_q;           /* query heads */
    int32_t h_k;           /* KV heads; g = h_q / h_k query heads share one KV head */
    int32_t head_dim;      /* d, same for q, k and v */
    int32_t block_size;    /* B_K, keys per KV block */
    int32_t topk;          /* T, slots per (KV head, token) in sel_idx */
    int32_t dtype;         /* nsa_dtype of q, k, v, out, dout, dq, dk, dv */
} nsa_sel_attn_dims;

/* Workspace bytes for nsa_sel_attn_fwd and nsa_sel_attn_bwd (host only, no CUDA
 * call).  Both start with the same index region, so one buffer of
 * max(fwd_bytes, bwd_bytes) serves a forward followed by a backward that reuses
 * the forward's index (index_ready = 1).  Either output pointer may be NULL. */
NSA_API nsa_status nsa_sel_attn_workspace_size(const nsa_sel_attn_dims *dims, size_t *fwd_bytes,
                                       size_t *bwd_bytes);

/* Index tensors of key design 2 (histogram, exclusive scan, scatter), built into
 * the workspace's index region: counts[h*NB + gb] tokens selected global block gb
 * (gb = local block + blocks of earlier sequences, NB = sum_s ceil(len_s / B_K));
 * offsets = exclusive scan (KV-head major), offsets[h_k*NB] = number of pairs;
 * q_list[offsets[i] + r] = the r-th token, ascending, that selected block i (I_i);
 * slot_map[h, t, k] = position of that (token, slot) pair, -1 when not kept (O_i).
 * nsa_sel_attn_fwd calls this itself; it is exported for tests and for a backward
 * without a forward. */
NSA_API nsa_status nsa_sel_attn_index(const nsa_sel_attn_dims *dims, const int32_t *sel_idx,
                              const int32_t *cu_seqlens, void *workspace, size_t workspace_bytes,
                              nsa_stream_t stream);

/* Device pointers into the workspace's index region (host only, no CUDA call).
 * num_blocks receives the host upper bound NB_max used for the layout; the true
 * NB is written on the device at *nb_device.  Any output pointer may be NULL. */
NSA_API nsa_status nsa_sel_attn_index_view(const nsa_sel_attn_dims *dims, const void *workspace,
                                   const int32_t **counts, const int32_t **offsets,
                                   const int32_t **q_list, const int32_t **slot_map,
                                   const int32_t **nb_device, int32_t *num_blocks);

/* Forward: out (dtype) and lse (float32) from q, k, v and the selection.
 * Builds the index, then runs the per-KV-block main kernel (gathered query rows x
 * one KV block on tcgen05 tensor cores, partial outputs with their own softmax
 * max and sum written to a compact buffer) and the merge kernel that combines the
 * partials of every (token, query head) with log-sum-exp weights (the statistics
 * and reduction stages of key designs 3-4). */
NSA_API nsa_status nsa_sel_attn_fwd(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                            const void *v, const int32_t *sel_idx, const int32_t *cu_seqlens,
                            float scale, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, nsa_stream_t stream);

/* Backward: dq, dk, dv (dtype) from q, k, v, the forward's out and lse, and dout.
 * index_ready = 1 reuses the index that nsa_sel_attn_fwd (or _index) left in this
 * workspace (the backward reuses the forward's I_i / O_i, key design 2);
 * index_ready = 0 rebuilds it.  dk and dv are fully overwritten. */
NSA_API nsa_status nsa_sel_attn_bwd(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                            const void *v, const int32_t *sel_idx, const int32_t *cu_seqlens,
                            float scale, const void *out, const float *lse, const void *dout,
                            void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                            int index_ready, nsa_stream_t stream);

/* Device staging bytes for nsa_sel_attn_step_host (host only). */
NSA_API nsa_status nsa_sel_attn_staging_size(const nsa_sel_attn_dims *dims, size_t *bytes);

/* One training step of the branch from HOST buffers: copies q, k, v, dout,
 * sel_idx and cu_seqlens to the caller's device staging buffer, runs forward and
 * backward (reusing the index), copies out, lse, dq, dk and dv back to the host
 * buffers, and synchronises the stream.  A side stream, created once per device by
 * the library, carries k and v up beside q, then dout while the forward runs, out and
 * lse down while the backward runs, and dk and dv down beside dq; the call returns
 * only after every copy of both streams is complete.  Host buffers should be pinned for the copies
 * to be asynchronous.  host_lse may be NULL to skip that copy. */
NSA_API nsa_status nsa_sel_attn_step_host(const nsa_sel_attn_dims *dims, const void *host_q,
                                  const void *host_k, const void *host_v,
                                  const int32_t *host_sel_idx, const int32_t *host_cu_seqlens,
                                  const void *host_dout, float scale, void *host_out,
                                  float *host_lse, void *host_dq, void *host_dk, void *host_dv,
                                  void *staging, size_t staging_bytes, void *workspace,
                                  size_t workspace_bytes, nsa_stream_t stream);

/* Size of the fixed scratch array used by nsa_sel_attn_fwd_noalloc (16 MiB). */
#define NSA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Forward without any device allocation, for callers that cannot allocate:
 * plugins whose host framework owns all device memory, loops that cannot afford
 * an allocation's synchronisation.  Same inputs,
 * outputs and results as nsa_sel_attn_fwd, but the scratch is a fixed array of
 * NSA_NOALLOC_SCRATCH_BYTES inside the library (held by every GPU that loads the
 * library until exit).  The paper has no counterpart to this entry point.
 *   - Problems whose forward workspace (nsa_sel_attn_workspace_size) exceeds
 *     NSA_NOALLOC_SCRATCH_BYTES are rejected with NSA_ERR_WORKSPACE; nothing runs.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and keeps it; the lookup is repeated when the device's
 *     current context has changed (after cudaDeviceReset, for instance).
 *   - All calls share the one array and it keeps the last call's contents: calls
 *     that may overlap on the GPU (different streams without ordering, several
 *     host threads) race; serialise them.  The call clears the status word itself
 *     and writes every scratch entry it reads, so no clearing is needed between
 *     calls.  Device-side error bits of a call are read with
 *     nsa_sel_attn_fwd_noalloc_status. */
NSA_API nsa_status nsa_sel_attn_fwd_noalloc(const nsa_sel_attn_dims *dims, const void *q,
                                            const void *k, const void *v, const int32_t *sel_idx,
                                            const int32_t *cu_seqlens, float scale, void *out,
                                            float *lse, nsa_stream_t stream);

/* Device status word of the fixed scratch used by nsa_sel_attn_fwd_noalloc: the
 * same contract as nsa_sel_attn_get_status (synchronises `stream`, reads and
 * clears the word, returns NSA_OK, NSA_ERR_BAD_INDEX or NSA_ERR_TIMEOUT and the raw
 * bits).  dims must be those of the call being checked; the same size limit
 * applies.  Like the entry point itself, it allocates nothing.  The paper has no
 * counterpart to this function. */
NSA_API nsa_status nsa_sel_attn_fwd_noalloc_status(const nsa_sel_attn_dims *dims,
                                                   nsa_stream_t stream, int32_t *bits);

/* One-step decode: the one-step decoding preview of the Flash-Sparse-Attention
 * README ("News"), the decoding stage that the papernotes page leaves open
 * (局限与展望).  Every sequence b has one new query token, the last token of its KV
 * cache (local position len_b - 1).  It attends to the keys of the blocks its
 * selection names, with the forward's arithmetic for that token:
 *   - the causal mask (every cached key of a kept block, up to the token itself);
 *   - the same validity, de-duplication and error rules for sel_idx;
 *   - one softmax over the union of the kept blocks.
 *   dims:      num_seqs = B sequences; total_tokens = N cached tokens in all;
 *              h_q, h_k, head_dim, block_size, topk, dtype as for the forward.
 *              Supported: head_dim 64 or 128, g = h_q / h_k <= 16.
 *   q:         [B, h_q, d] (dtype), the new token of each sequence.
 *   k_cache, v_cache: [N, h_k, d] (dtype), packed by cu_seqlens.
 *   sel_idx:   int32 [h_k, B, T], block indices local to each sequence.
 *   cu_seqlens: int32 [B + 1], cache offsets (cu[0] = 0, cu[B] = N).
 *   out:       [B, h_q, d] (dtype); lse: float32 [h_q, B] (natural log, scale
 *              included; -inf and out = 0 for a sequence with no kept key).
 *   device_status: optional int32 in device memory.  NSA_DEVERR_BAD_INDEX is ORed
 *              into it for a value < -1 or past the sequence's last block; NULL
 *              skips the report.
 * No workspace: one CTA per (sequence, KV head) merges its warps' partial results on
 * chip.  Asynchronous on `stream`; q, caches and out 16-byte aligned.  The pages give
 * no decode algorithm; this entry point is the forward restricted to one token per
 * sequence. */
/* Sliding-window branch (the third of Native Sparse Attention's parallel branches: the
 * papernotes page's 领域现状; window_size = 512 in the Flash-Sparse-Attention README's
 * "Usage").  A token at local position tau attends to the keys of (tau - window,
 * tau] of its sequence, causal, one softmax.  It runs on the selected-attention
 * kernels:
 *   nsa_sel_attn_window_select writes the selection rows of the window: int32
 *     [h_k, N, topk], the blocks holding those keys, newest first (c(t), c(t) - 1,
 *     ...), the other slots -1.  topk must be at least ceil((window - 1) / B_K) + 1,
 *     else NSA_ERR_INVALID_ARG.
 *   nsa_sel_attn_fwd_window and nsa_sel_attn_bwd_window are nsa_sel_attn_fwd and
 *     nsa_sel_attn_bwd with the window's lower key bound added to the causal mask
 *     (window >= 1).  Given a window selection, they compute sliding-window
 *     attention.  Given any other selection, they compute that selection restricted
 *     to the window.  Arguments, workspace and errors are those of fwd and bwd. */
NSA_API nsa_status nsa_sel_attn_window_select(const nsa_sel_attn_dims *dims,
                                              const int32_t *cu_seqlens, int window,
                                              int32_t *sel_idx, nsa_stream_t stream);
NSA_API nsa_status nsa_sel_attn_fwd_window(const nsa_sel_attn_dims *dims, const void *q,
                                           const void *k, const void *v, const int32_t *sel_idx,
                                           const int32_t *cu_seqlens, float scale, int window,
                                           void *out, float *lse, void *workspace,
                                           size_t workspace_bytes, nsa_stream_t stream);
NSA_API nsa_status nsa_sel_attn_bwd_window(const nsa_sel_attn_dims *dims, const void *q,
                                           const void *k, const void *v, const int32_t *sel_idx,
                                           const int32_t *cu_seqlens, float scale, int window,
                                           const void *out, const float *lse, const void *dout,
                                           void *dq, void *dk, void *dv, void *workspace,
                                           size_t workspace_bytes, int index_ready,
                                           nsa_stream_t stream);

/* Gated combination of the branch outputs: out[t, hq] = sum_b gates[t, hq, b] * o_b[t,
 * hq] for n_branch = 1..3 branches o0, o1, o2, each [N, h_q, d] (dtype).
 *   gates: float32 [N, h_q, n_branch], the gate values, e.g. sigmoids of a gate
 *     projection.  The projection itself belongs to the model, not to this library.
 *   Backward: d o_b = gates[., b] * dout, and dgates[., b] = sum_d dout * o_b
 *     (fp32).  A NULL do_b skips that branch's output gradient.
 * dims supplies N, h_q, head_dim and dtype.  The branch pointers must be 4-byte
 * aligned.  The pages name the gated three-branch output but give no formula beyond
 * the weighted sum. */
NSA_API nsa_status nsa_gate_combine_fwd(const nsa_sel_attn_dims *dims, int n_branch,
                                        const void *o0, const void *o1, const void *o2,
                                        const float *gates, void *out, nsa_stream_t stream);
NSA_API nsa_status nsa_gate_combine_bwd(const nsa_sel_attn_dims *dims, int n_branch,
                                        const void *o0, const void *o1, const void *o2,
                                        const float *gates, const void *dout, void *do0,
                                        void *do1, void *do2, float *dgates,
                                        nsa_stream_t stream);

/* The step before selected attention: the compressed branch and the top-T block
 * selection that produce sel_idx (Native Sparse Attention's compression and selection
 * branches, papernotes page, 研究背景与动机 "领域现状" and the 方法详解 flowchart's
 * selection tensor T; kernel_size 32, kernel_stride 16, block_size 64, topk 16,
 * init_blocks 1 and local_blocks 2 in the Flash-Sparse-Attention README's "Usage").
 * The pages give no formula for these steps; the library takes these readings:
 *   compression: compressed token i of a sequence is the mean of the keys (values)
 *     at positions [i*stride, i*stride + kernel_size); it exists when that window
 *     lies inside the sequence;
 *   the query at position tau (within its sequence) sees compressed token i when
 *     i*stride + kernel_size - 1 <= tau;
 *   compressed attention: out = softmax(scale * q . kc) vc over the visible
 *     compressed tokens, lse its log-sum-exp; no visible token: out 0, lse -inf;
 *   importance of block j (keys [j*B_K, j*B_K + B_K)) for a (KV head, token): the
 *     sum, over the group's g query heads and the visible compressed tokens whose
 *     window overlaps those keys, of the compressed-attention probability;
 *   selection: among the causal blocks j <= tau / B_K, first the init blocks
 *     (j < init_blocks) and the local blocks (tau/B_K - local_blocks < j), ascending,
 *     then the others by importance, larger first, ties to the lower block; slots
 *     left over are -1.
 *
 * nsa_compress_kv: k, v [N, h_k, d] (dims->dtype) -> kc, vc [R, h_k, d] with
 *   R = floor(N / kernel_stride) rows allocated by the caller (an upper bound on the
 *   compressed tokens when kernel_size >= kernel_stride); the compressed tokens of
 *   sequence s are rows cu_cmp[s] .. cu_cmp[s+1] - 1, and cu_cmp (int32 [S + 1],
 *   written here) ends at their total.  Means are taken in fp32 and rounded to the
 *   dtype.  Malformed cu_seqlens set NSA_DEVERR_BAD_SEQLENS in *device_status (may
 *   be NULL).
 * nsa_cmp_attn_select: q [N, h_q, d], kc / vc and cu_cmp from nsa_compress_kv ->
 *   out [N, h_q, d] (dtype), lse float32 [h_q, N], sel_idx int32 [h_k, N, topk]
 *   (dims->block_size = B_K, dims->topk = T), ready for nsa_sel_attn_fwd.
 *   max_seqlen bounds every sequence's length: it sizes the importance rows, one
 *   fp32 per causal block of each token; a longer sequence sets
 *   NSA_DEVERR_BAD_SEQLENS and its tokens are left unwritten.  The rows live in
 *   shared memory, or, when they would leave a CTA too few tokens there and a
 *   workspace is given, in that workspace (caller-owned device memory of at least
 *   nsa_cmp_workspace_size bytes, 16-byte aligned; NULL and 0 allowed).  Too small a
 *   workspace is NSA_ERR_WORKSPACE; rows that fit neither way NSA_ERR_UNSUPPORTED.
 *   Importance is summed in fp32, so blocks whose importance differs by rounding may
 *   be chosen in either order.
 * nsa_cmp_workspace_size: the workspace bytes nsa_cmp_attn_select uses for these
 *   dims and max_seqlen (0 when shared memory suffices); host only.
 * Both: d in {64, 128}; kernel_size >= kernel_stride >= 1; g <= 128; q, kc, vc, out,
 * k, v 16-byte aligned; errors are returned before any launch. */
NSA_API nsa_status nsa_compress_kv(const nsa_sel_attn_dims *dims, const int32_t *cu_seqlens,
                                   int kernel_size, int kernel_stride, const void *k,
                                   const void *v, void *kc, void *vc, int32_t *cu_cmp,
                                   int32_t *device_status, nsa_stream_t stream);
NSA_API nsa_status nsa_cmp_attn_select(const nsa_sel_attn_dims *dims, const void *q,
                                       const void *kc, const void *vc,
                                       const int32_t *cu_seqlens, const int32_t *cu_cmp,
                                       int kernel_size, int kernel_stride, int max_seqlen,
                                       float scale, int init_blocks, int local_blocks,
                                       void *out, float *lse, int32_t *sel_idx,
                                       int32_t *device_status, void *workspace,
                                       size_t workspace_bytes, nsa_stream_t stream);
NSA_API nsa_status nsa_cmp_workspace_size(const nsa_sel_attn_dims *dims, int kernel_size,
                                          int kernel_stride, int max_seqlen, size_t *bytes);

NSA_API nsa_status nsa_sel_attn_decode(const nsa_sel_attn_dims *dims, const void *q,
                                       const void *k_cache, const void *v_cache,
                                       const int32_t *sel_idx, const int32_t *cu_seqlens,
                                       float scale, void *out, float *lse,
                                       int32_t *device_status, nsa_stream_t stream);

/* Synchronises `stream`, reads and clears the device status word of this
 * workspace.  Returns NSA_OK, NSA_ERR_BAD_INDEX or NSA_ERR_TIMEOUT (the worst
 * seen) and stores the raw bits in *bits when bits is not NULL. */
NSA_API nsa_status nsa_sel_attn_get_status(const nsa_sel_attn_dims *dims, void *workspace,
                                   nsa_stream_t stream, int32_t *bits);

/* Kernel timing for diagnostics.  While enabled, every kernel the library
 * launches is bracketed by CUDA events on its launch stream (the library creates
 * and owns the events).  collect synchronises on them and adds, per kernel id,
 * the launch count and total milliseconds since the last collect; arrays have
 * nsa_sel_attn_num_kernels() entries. */
NSA_API int32_t nsa_sel_attn_num_kernels(void);
NSA_API const char *nsa_sel_attn_kernel_name(int32_t id);
NSA_API nsa_status nsa_sel_attn_profile_enable(int32_t on);
NSA_API nsa_status nsa_sel_attn_profile_collect(int32_t *launches, float *total_ms);

NSA_API const char *nsa_status_string(nsa_status status);

#ifdef __cplusplus
}
#endif

#endif /* NSA_SEL_ATTN_H */
