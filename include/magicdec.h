/*
 * magicdec.h -- C ABI of the GB300 (sm_103a) hot path for MagicDec-style
 * long-context self-speculative decoding.
 *
 * Method: "MagicDec: Breaking the Latency-Throughput Tradeoff for Long Context
 * Generation with Speculative Decoding" (arXiv 2408.11049v5).  A target model
 * drafts gamma tokens with attention over a sparse subset of its own KV cache
 * (StreamingLLM sinks + recent window, or SnapKV observation-window top-k,
 * section 4.4), then verifies them with attention of the gamma+1 speculated
 * queries over the full KV cache (section 3.1, T_V(B,S,gamma)), and keeps the
 * accepted prefix by speculative sampling (Leviathan et al., cited for Eq. 1)
 * or greedy matching (section 5.1).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates nothing and keeps no state between calls, apart from one
 *    device-side error word (see magicdec_device_error).
 *  - bf16 tensors are passed as uint16_t bit patterns.  Layouts are dense
 *    row-major with the shapes given beside each argument.
 *  - Every pointer that a kernel reads or writes in 16-byte vectors must be
 *    16-byte aligned (checked; MAGICDEC_ERR_ALIGN).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    validate their arguments on the host, enqueue kernels and return without
 *    synchronising.  A status other than MAGICDEC_OK means nothing was
 *    enqueued, except MAGICDEC_ERR_CUDA, which reports a launch error.
 *  - Per-sequence lengths live on the device and cannot be checked on the
 *    host: kernels clamp them to [0, capacity].
 *  - Inputs must be finite.
 *  - Workspaces are caller-owned device buffers of at least the size the
 *    matching *_workspace_size() returns.  They must be zero-filled once
 *    before first use; every call leaves them ready for the next call.  Calls
 *    that share one workspace must not overlap on the GPU.
 */
#ifndef MAGICDEC_H
#define MAGICDEC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MAGICDEC_API __attribute__((visibility("default")))
#else
#define MAGICDEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MAGICDEC_OK = 0,
    MAGICDEC_ERR_NULL = -1,        /* a required pointer is NULL */
    MAGICDEC_ERR_SHAPE = -2,       /* a size is out of range or inconsistent */
    MAGICDEC_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
    MAGICDEC_ERR_WORKSPACE = -4,   /* workspace smaller than *_workspace_size() */
    MAGICDEC_ERR_UNSUPPORTED = -5, /* a valid shape the library has no kernel for */
    MAGICDEC_ERR_CUDA = -6         /* the CUDA runtime reported an error */
} magicdec_status;

/* Attention problem shape.  KV cache K/V: [B, L_cap, H_kv, d].  Query head hq
 * reads KV head hq / (H_q / H_kv) (grouped-query attention).  d is 64 or 128;
 * H_q must be a multiple of H_kv. */
typedef struct {
    int B;
    int H_q;
    int H_kv;
    int d;
    int L_cap;
} magicdec_kv_shape;

/* Human-readable name of a status code (static string). */
MAGICDEC_API const char *magicdec_status_string(int status);

/* Copies the device error word of the current device into *out and clears it
 * (synchronises the device).  Non-zero means a kernel gave up on a bounded
 * wait (value 1) or met an inconsistent internal state (value 2), and its
 * outputs are then undefined; or that magicdec_draft_cache_update skipped a
 * row whose slot was at or past the cache capacity (value 3).  In the
 * range-checking build (libmagicdec_debug.so, compiled with
 * MAGICDEC_DEBUG_CHECKS) value 4 means a kernel read a sequence length
 * outside [0, capacity] or a gather index outside [0, L_cap) other than the
 * -1 padding mark; that build still clamps or skips the value as documented
 * for each call, so its outputs equal the release build's, which records
 * nothing for it.  The first error since the last read is kept.  Returns MAGICDEC_OK or
 * MAGICDEC_ERR_CUDA. */
MAGICDEC_API magicdec_status magicdec_device_error(int32_t *out);

/*
 * StreamingLLM draft-KV selection (paper section 4.4 and section 5.1:
 * attention sinks plus a recent window; budget n_sink + n_recent).
 *   seq_len [B] int32   current sequence lengths (clamped below at 0)
 *   idx     [B, H_kv, n_sink + n_recent] int32 out: for each sequence the
 *           positions [0, min(n_sink, len)) then [max(n_sink, len-n_recent),
 *           len), ascending, identical for every KV head; -1 after n_sel[b].
 *   n_sel   [B] int32 out: number of valid entries per sequence.
 * Errors: NULL pointers, B <= 0, H_kv <= 0, n_sink < 0, n_recent < 0,
 * n_sink + n_recent == 0 or above INT_MAX; MAGICDEC_ERR_UNSUPPORTED when B or H_kv exceeds
 * 65535 (the kernel's grid has one block row per KV head and sequence).
 */
MAGICDEC_API magicdec_status magicdec_streaming_select(const int32_t *seq_len, int B, int H_kv, int n_sink,
                                          int n_recent, int32_t *idx, int32_t *n_sel, void *stream);

/* Workspace bytes magicdec_snapkv_select needs for this shape and window. */
MAGICDEC_API size_t magicdec_snapkv_workspace_size(magicdec_kv_shape shape, int window);

/*
 * SnapKV draft-KV selection, run once after prefill (paper section 4.4: a
 * static method whose compact cache is built once; section 5.2: best budget
 * about 2048).  For each sequence of length L = seq_len[b] (clamped to
 * [0, L_cap]) and KV head h, the last `window` positions form the
 * observation window; window row r (position L-window+r) of query head hq has
 * query q_win[b, r, hq, :] and attends causally over positions 0..L-window+r.
 * The score of a prefix position j < L-window is the sum over window rows and
 * over the H_q/H_kv query heads of the group of the softmax probability at j.
 * Scores are max-pooled (kernel pool_kernel, stride 1, clipped at the ends),
 * the budget-window largest are kept (ties to the smaller position), sorted
 * ascending, and the window positions [L-window, L) are appended.  When
 * L <= budget all positions 0..L-1 are kept.
 *   q_win [B, window, H_q, d] bf16;  k [B, L_cap, H_kv, d] bf16
 *   idx   [B, H_kv, budget] int32 out (-1 after n_sel[b]);  n_sel [B] int32 out
 *   ws    workspace of magicdec_snapkv_workspace_size(shape, window) bytes
 * Errors: NULL pointers, bad shape, window <= 0, budget < window,
 * pool_kernel even or <= 0, alignment, workspace too small;
 * MAGICDEC_ERR_UNSUPPORTED when window * (H_q/H_kv) > 256 or pool_kernel > 9.
 */
MAGICDEC_API magicdec_status magicdec_snapkv_select(magicdec_kv_shape shape, const uint16_t *q_win, const uint16_t *k,
                                       const int32_t *seq_len, int window, int pool_kernel, int budget,
                                       int32_t *idx, int32_t *n_sel, void *ws, size_t ws_bytes, void *stream);

/*
 * SnapKV selection with a budget per sequence (heterogeneous batches; paper
 * section 4.3 discusses draft budgets per sequence length).  As
 * magicdec_snapkv_select, except that sequence b keeps budgets[b] positions
 * (device int32 [B], clamped to [window, max_budget]) and idx rows have
 * max_budget entries ([B, H_kv, max_budget], -1 after n_sel[b]); the gather
 * and the draft attention then take n_idx = cap = max_budget and
 * draft_len = n_sel.
 * Errors: as magicdec_snapkv_select, with max_budget in the role of budget.
 */
MAGICDEC_API magicdec_status magicdec_snapkv_select_budgets(magicdec_kv_shape shape, const uint16_t *q_win,
                                                            const uint16_t *k, const int32_t *seq_len, int window,
                                                            int pool_kernel, const int32_t *budgets, int max_budget,
                                                            int32_t *idx, int32_t *n_sel, void *ws, size_t ws_bytes,
                                                            void *stream);

/*
 * Gather of the selected rows into the compact draft cache (paper section
 * 4.4: the static selections copy their rows into a compact cache once).
 *   k, v   [B, L_cap, H_kv, d] bf16;  idx [B, H_kv, n_idx] int32
 *   kc, vc [B, H_kv, cap, d] bf16 out: row i < n_idx of head h is
 *          k[b, idx[b,h,i], h] (zero row when the index is outside [0, L_cap));
 *          rows n_idx..cap-1 are not touched (room for appended tokens).
 * Errors: NULL pointers, bad shape, n_idx < 0, n_idx > cap, alignment.
 */
MAGICDEC_API magicdec_status magicdec_gather_kv(magicdec_kv_shape shape, const uint16_t *k, const uint16_t *v,
                                   const int32_t *idx, int n_idx, int cap, uint16_t *kc, uint16_t *vc,
                                   void *stream);

/*
 * Draft-cache update: append, post-verification refresh and rollback of the
 * compact draft cache (paper section 4.4: the static drafts select once and
 * afterwards only take in new tokens; section 3.1: verification keeps the
 * accepted prefix, so rows the sparse draft wrote for rejected or
 * re-verified positions are replaced).  Layouts of kc, vc [B, H_kv, cap, d]:
 *   ring > 0 (StreamingLLM, sinks + recent window): position q < origin[b]
 *     at slot q; position q >= origin[b] at slot
 *     origin[b] + (q - origin[b]) mod ring.  The occupied slots hold exactly
 *     positions [0, min(len, origin)) and [max(origin, len - ring), len);
 *     from an empty cache, update(0, 0, L) builds the StreamingLLM selection
 *     for length L.  base is not read (may be NULL).
 *   ring == 0 (SnapKV): slots [0, base[b]) hold the rows kept at selection
 *     (magicdec_gather_kv); position q >= origin[b] (the length at selection)
 *     is appended at slot base[b] + q - origin[b].
 * Lengths (device int32 [B], clamped to [0, L_cap]; len_valid to at most
 * min(len_old, len_new)): rows of positions >= len_valid in the compact cache
 * are stale (drafted, or never written); len_old is the length the cache was
 * last brought to, len_new the new one.  The call copies from k, v
 * [B, L_cap, H_kv, d] every position of the new window at or past len_valid,
 * and (ring layout) restores every slot that a position in [len_new, len_old)
 * overwrote with the window position it displaced.  Typical use, per layer:
 * drafting appends position L+i as update(L+i, L+i, L+i+1); after
 * verification with n_acc accepted, update(L, L+gamma, L+n_acc+1).
 *   draft_len [B] int32 out: occupied slots (the draft attention's length),
 *   clamped to cap.
 * Errors: NULL pointers, bad shape, ring < 0, cap <= 0, base NULL when
 * ring == 0, ring > 0 with ring > cap, alignment.  A copy whose slot is at or
 * past cap is skipped and sets the device error word to 3.
 */
MAGICDEC_API magicdec_status magicdec_draft_cache_update(magicdec_kv_shape shape, const uint16_t *k, const uint16_t *v,
                                                         const int32_t *len_valid, const int32_t *len_old,
                                                         const int32_t *len_new, const int32_t *origin,
                                                         const int32_t *base, int ring, int cap, uint16_t *kc,
                                                         uint16_t *vc, int32_t *draft_len, void *stream);

/*
 * Lengths of one speculative step (paper section 3.1: gamma draft steps, one
 * verification of the gamma+1 block, then the sequence keeps its accepted
 * prefix and the emitted token; section 4.4: the static draft caches take in
 * each new position).  For every sequence b:
 *   len = len_in[b] + (n_acc ? n_acc[b] + 1 : 0), clamped to [0, L_cap];
 *   len_out[b] = len;  table[j * B + b] = min(len + j, L_cap), j = 0..gamma+1.
 * With len the number of cached positions at the start of a step, the step's
 * calls take: draft step g appends position len + g before attending,
 * magicdec_draft_cache_update(table[g], table[g], table[g+1]); verification
 * runs at seq_len = table[gamma+1] (the block's K/V at [len, len+gamma+1));
 * after acceptance a second call with n_acc gives the next length, and
 * magicdec_draft_cache_update(table[0], table[gamma], that length) refreshes
 * the verified rows and drops the rejected ones.
 *   len_in, n_acc (nullable: advance by 0), len_out [B] int32 device;
 *   table [(gamma+2) * B] int32 device.  len_out may alias len_in.
 * Errors: NULL pointers, B <= 0, gamma < 0 or > 1024, L_cap <= 0.
 */
MAGICDEC_API magicdec_status magicdec_step_lengths(int B, int gamma, int L_cap, const int32_t *len_in,
                                                   const int32_t *n_acc, int32_t *len_out, int32_t *table,
                                                   void *stream);

/* Workspace bytes magicdec_draft_attn / magicdec_verify_attn need for this
 * shape and query count (n_q = 1 for draft) on the current device. */
MAGICDEC_API size_t magicdec_attn_workspace_size(magicdec_kv_shape shape, int n_q);

/*
 * Draft attention (paper section 4.1, Eq. 3: decoding cost T_D(B,K) over the
 * K-row draft cache).  One query token per sequence attends to rows
 * 0..draft_len[b]-1 of its KV head in the compact cache (draft_len clamped to
 * [0, cap]; an empty cache gives a zero row).  Softmax scale 1/sqrt(d).
 *   shape.L_cap is the compact capacity `cap`.
 *   q  [B, 1, H_q, d] bf16;  kc, vc [B, H_kv, cap, d] bf16;  draft_len [B] int32
 *   out [B, 1, H_q, d] bf16
 * Errors: NULL pointers, bad shape, alignment, workspace too small.
 */
MAGICDEC_API magicdec_status magicdec_draft_attn(magicdec_kv_shape shape, const uint16_t *q, const uint16_t *kc,
                                    const uint16_t *vc, const int32_t *draft_len, uint16_t *out, void *ws,
                                    size_t ws_bytes, void *stream);

/*
 * Verification attention (paper section 3.1, T_V(B,S,gamma); section 3.2:
 * verification loads the same KV as decoding).  The n_q = gamma+1 speculated
 * tokens already occupy cache positions [len-n_q, len), len = seq_len[b]
 * clamped to [0, L_cap]; query row i sees positions 0..len-n_q+i (causal
 * inside the speculated block; a row that sees nothing gives zeros).
 *   q [B, n_q, H_q, d] bf16;  k, v [B, L_cap, H_kv, d] bf16;  seq_len [B] int32
 *   out [B, n_q, H_q, d] bf16
 * Supported: (H_q/H_kv) * n_q <= 32 (MAGICDEC_ERR_UNSUPPORTED beyond).
 * Errors: NULL pointers, bad shape, alignment, workspace too small.
 */
MAGICDEC_API magicdec_status magicdec_verify_attn(magicdec_kv_shape shape, int n_q, const uint16_t *q, const uint16_t *k,
                                     const uint16_t *v, const int32_t *seq_len, uint16_t *out, void *ws,
                                     size_t ws_bytes, void *stream);

/* Workspace bytes magicdec_topk_draft_attn needs: fp32 scores of every query
 * head over the whole cache, B * H_q * (L_cap rounded up to 4) * 4. */
MAGICDEC_API size_t magicdec_topk_attn_workspace_size(magicdec_kv_shape shape);

/*
 * Top-K attention draft (paper section 1 and Figure 1(c); section 4.4,
 * "Static vs Dynamic": the dynamic per-query selection whose acceptance rate
 * the static methods are compared against, and whose search over the whole
 * cache is its selection cost).  For query head h of sequence b, with
 * len = seq_len[b] clamped to [0, L_cap], the scores s_j = q . k_j / sqrt(d)
 * over j < len are ranked, the top_k largest are kept (equal scores: the
 * smaller position first; every position when len <= top_k), and
 *   out = sum_{j kept} softmax(s over the kept positions)_j v_j
 * (a zero row when len == 0).  Query head h reads KV head h / (H_q/H_kv).
 *   q [B, 1, H_q, d] bf16;  k, v [B, L_cap, H_kv, d] bf16;  seq_len [B] int32
 *   out [B, 1, H_q, d] bf16
 *   idx (nullable) [B, H_q, top_k] int32 out: the kept positions in ascending
 *       order, -1 after min(len, top_k)
 *   ws  workspace of magicdec_topk_attn_workspace_size(shape) bytes; no
 *       initial contents needed
 * Supported: H_q/H_kv <= 8 and top_k <= 8192 (MAGICDEC_ERR_UNSUPPORTED).
 * Errors: NULL pointers, bad shape, top_k <= 0, alignment (q, k, v, out, ws),
 * workspace too small.
 */
MAGICDEC_API magicdec_status magicdec_topk_draft_attn(magicdec_kv_shape shape, const uint16_t *q, const uint16_t *k,
                                                      const uint16_t *v, const int32_t *seq_len, int top_k,
                                                      uint16_t *out, int32_t *idx, void *ws, size_t ws_bytes,
                                                      void *stream);

/*
 * PQCache-style dynamic selection (paper section 4.4 and Figure 5: a dynamic
 * KV selection that searches the cache per query through product-quantised
 * keys, with a search cost that grows with the batch).  Keys of each
 * (sequence, KV head) split into M = d/8 sub-vectors of 8 channels; subspace
 * m has C (1..256) centroids.
 *   codebook [B, H_kv, M, C, 8] fp32;  codes [B, H_kv, L_cap, M] uint8
 * A codebook is built at prefill by Lloyd iterations: encode, then update,
 * repeated, from initial centroids chosen by the caller.
 *
 * Encode: codes[b,h,j,m] = the centroid c of subspace m nearest to the key's
 * sub-vector (squared distance, evaluated as |c|^2 - 2 k.c in fp32; equal
 * values: the smaller c), for every position j < L_cap.
 * Errors: NULL pointers, bad shape, M != d/8, C outside [1, 256], alignment
 * (k, codebook); MAGICDEC_ERR_UNSUPPORTED when the codebook of one
 * (sequence, head) does not fit in shared memory.
 */
MAGICDEC_API magicdec_status magicdec_pq_encode(magicdec_kv_shape shape, const uint16_t *k, int M, int C,
                                                const float *codebook, uint8_t *codes, void *stream);

/*
 * Update (one Lloyd step after an encode): centroid c of subspace m becomes
 * the mean of the sub-vectors of positions j < seq_len[b] coded c (exact sum,
 * correctly rounded mean, rounded to fp32); a centroid without positions
 * keeps its value.  codebook is updated in place.
 * Errors as magicdec_pq_encode.
 */
MAGICDEC_API magicdec_status magicdec_pq_update(magicdec_kv_shape shape, const uint16_t *k, const int32_t *seq_len,
                                                int M, int C, const uint8_t *codes, float *codebook, void *stream);

/* Workspace bytes magicdec_pq_draft_attn needs: fp32 approximate scores,
 * B * H_q * (L_cap rounded up to 4) * 4. */
MAGICDEC_API size_t magicdec_pq_attn_workspace_size(magicdec_kv_shape shape);

/*
 * PQ draft attention.  For query head h of sequence b (KV head h/(H_q/H_kv)),
 * with len = seq_len[b] clamped to [0, L_cap]: LUT[m][c] = q_m . centroid(m,c)
 * / sqrt(d); approximate score a_j = sum_m LUT[m][codes[b,h,j,m]] for j < len;
 * the top_k positions by a_j are kept (equal: the smaller position; all when
 * len <= top_k) and
 *   out = sum_{j kept} softmax(q . k_j / sqrt(d) over the kept j) v_j
 * with the EXACT scores (a zero row when len == 0).
 *   q [B, 1, H_q, d] bf16;  k, v [B, L_cap, H_kv, d] bf16;  out [B, 1, H_q, d] bf16
 *   idx (nullable) [B, H_q, top_k] int32 out: kept positions, ascending, -1 padded
 *   ws  workspace of magicdec_pq_attn_workspace_size(shape) bytes
 * Supported: top_k <= 8192.  Errors: as magicdec_pq_encode, plus top_k <= 0,
 * alignment of q, v, out, ws, workspace too small.
 */
MAGICDEC_API magicdec_status magicdec_pq_draft_attn(magicdec_kv_shape shape, const uint16_t *q, const uint16_t *k,
                                                    const uint16_t *v, const int32_t *seq_len, int M, int C,
                                                    const float *codebook, const uint8_t *codes, int top_k,
                                                    uint16_t *out, int32_t *idx, void *ws, size_t ws_bytes,
                                                    void *stream);

/*
 * Verification attention that allocates nothing (no counterpart in the paper;
 * an addition for callers that cannot allocate device memory, such as a
 * plug-in that receives only its input and output buffers from a host
 * runtime, an engine whose memory plan is fixed before it starts, or a
 * process whose device memory is owned by another allocator).  Same
 * arguments, layouts and results as magicdec_verify_attn, without `ws`: its
 * scratch is a 32 MiB array inside the library, which every GPU that loads
 * the library holds until the process exits.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture.
 *  - Every call first clears the part of the array that must start at zero
 *    (the merge counters and scheduler words, 256 KB) with cudaMemsetAsync
 *    on `stream`, then launches on the same stream; so a call that gave up on
 *    a bounded wait (device error word 1) leaves nothing that a later call
 *    can trip over.
 *  - All calls on a device share the array, which keeps the last call's
 *    contents; calls that overlap on the GPU race, so order them (one
 *    stream).
 *  - Returns MAGICDEC_ERR_UNSUPPORTED, and enqueues nothing, when the
 *    kernel's scratch for the current device would not fit in the array.
 * Errors otherwise as magicdec_verify_attn.
 */
MAGICDEC_API magicdec_status magicdec_verify_attn_noalloc(magicdec_kv_shape shape, int n_q, const uint16_t *q,
                                                          const uint16_t *k, const uint16_t *v,
                                                          const int32_t *seq_len, uint16_t *out, void *stream);

/* Workspace bytes magicdec_spec_accept needs. */
MAGICDEC_API size_t magicdec_spec_accept_workspace_size(int B, int gamma, int V);

/*
 * Speculative-sampling accept / resample for one verification step
 * (Leviathan et al., as used for Eq. 1 in paper section 3.1), or greedy
 * verification (paper section 5.1).
 *   target [B, gamma+1, V] fp32 logits of the target at the gamma+1 positions
 *   draft  [B, gamma, V]   fp32 logits of the draft (may be NULL when greedy)
 *   draft_tok [B, gamma] int32; u_acc [B, gamma], u_res [B] uniforms in [0,1)
 * Sampling (greedy == 0), temperature 1, p = softmax(target_i),
 *   q = softmax(draft_i): draft token x is accepted iff u_acc < p(x)/q(x)
 *   (q(x) == 0 accepts iff p(x) > 0; x outside [0,V) is rejected).  At the
 *   first rejection the emitted token is the smallest t whose running sum of
 *   max(0, p - q) exceeds u_res times its total (of p if that total is 0).
 *   If all gamma drafts are accepted, a bonus token is drawn the same way from
 *   softmax(target_gamma).
 * Greedy (greedy != 0): accept while x equals argmax target_i (ties to the
 *   smaller token); emit that argmax at the first mismatch, else the argmax of
 *   target_gamma.
 * Outputs: n_acc [B] accepted count in [0, gamma]; out_tok [B, gamma+1]: the
 *   accepted tokens, then the emitted one, -1 after; n_ambiguous [B]
 *   (nullable): decisions taken near their boundary -- |u - p/q| < 1e-4, a
 *   top-2 logit gap below 1e-4, or u * total within 1e-7 of the total from a
 *   token edge of the inverse CDF.
 * Precision: per-logit exponentials in fp32; normalisers, p/q ratios and
 *   running sums in fp64 / double-float.
 * Errors: NULL pointers, B <= 0, gamma < 0, V <= 0, workspace too small.
 */
MAGICDEC_API magicdec_status magicdec_spec_accept(int B, int gamma, int V, const float *target_logits,
                                     const float *draft_logits, const int32_t *draft_tok, const float *u_acc,
                                     const float *u_res, int greedy, int32_t *n_acc, int32_t *out_tok,
                                     int32_t *n_ambiguous, void *ws, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MAGICDEC_H */
