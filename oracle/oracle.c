/*
 * oracle.c -- plain fp64 CPU oracle for the MagicDec self-speculative
 * decoding hot path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load this library.  It shares no
 * code, header, table or helper with the CUDA library; the two meet only in
 * the seeded inputs they are both given.
 *
 * Every function restates, in plain loops and in double precision, a
 * definition from "MagicDec: Breaking the Latency-Throughput Tradeoff for Long
 * Context Generation with Speculative Decoding" (arXiv 2408.11049v5):
 *   - verification attention: the gamma+1 speculated queries attend to the
 *     full KV cache, causal inside the speculated block (section 3.1, the
 *     verification cost T_V(B,S,gamma); section 3.2);
 *   - draft attention: one query over the K-row sparse draft cache
 *     (section 4.1, Eq. 3, the decoding cost T_D(B,K));
 *   - StreamingLLM selection: attention sinks plus a recent window
 *     (section 4.4 and section 5.1);
 *   - SnapKV selection: observation-window attention scores, summed over the
 *     window rows and the query heads of a KV group, max-pooled, per-KV-head
 *     top-k, observation window always kept (section 4.4, section 5.2);
 *   - the copy of the selected rows into the compact draft cache
 *     (section 4.4) and the
 *     append / rollback of the compact cache as tokens are accepted or
 *     rejected (sections 3.1, 4.4);
 *   - PQCache-style dynamic selection: product-quantised keys (encode and
 *     Lloyd update of the codebooks), approximate scores from per-query
 *     lookup tables, exact attention over the top_k (section 4.4, Figure 5);
 *   - Top-K attention drafting: each draft query attends to its own top_k
 *     highest-scoring positions of the full cache (section 1, Figure 1(c);
 *     section 4.4);
 *   - speculative sampling (Leviathan et al., cited in section 3.1 for
 *     Eq. 1): accept draft token x when u < p(x)/q(x), otherwise resample
 *     from norm(max(0, p - q)); a bonus token from the last target
 *     distribution when all gamma drafts are accepted.  Greedy verification
 *     (the decoding used in section 5.1) accepts while x equals argmax p.
 *
 * Inputs arrive exactly as the GPU path consumes them: bf16 bit patterns
 * (uint16) for Q/K/V, fp32 logits and uniforms, int32 lengths and tokens.
 * Each bf16 value widens exactly to double.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE-754 binary32; widening is exact. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int clamp_len(int32_t len, int hi)
{
    if (len < 0) return 0;
    if (len > hi) return hi;
    return (int)len;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Softmax attention of one query row over n_vis key/value rows.             */
/*   o = sum_j softmax_j(scale * q . k_j) v_j                                 */
/* k_j sits at k0 + j*kstride, v_j at v0 + j*vstride (elements).  An empty    */
/* visible set yields a zero row.                                             */
/* ------------------------------------------------------------------------ */
static void attend_one(const uint16_t *qrow, int d, double scale,
                       const uint16_t *k0, long kstride,
                       const uint16_t *v0, long vstride,
                       int n_vis, double *out)
{
    int c;
    long j;
    for (c = 0; c < d; ++c) out[c] = 0.0;
    if (n_vis <= 0) return;

    double *s = (double *)malloc(sizeof(double) * (size_t)n_vis);
    double *q = (double *)malloc(sizeof(double) * (size_t)d);
    for (c = 0; c < d; ++c) q[c] = bf16_value(qrow[c]);

    double smax = -INFINITY;
    for (j = 0; j < n_vis; ++j) {
        const uint16_t *kr = k0 + j * kstride;
        double acc = 0.0;
        for (c = 0; c < d; ++c) acc += q[c] * bf16_value(kr[c]);
        s[j] = scale * acc;
        if (s[j] > smax) smax = s[j];
    }
    double den = 0.0;
    for (j = 0; j < n_vis; ++j) {
        double w = exp(s[j] - smax);
        const uint16_t *vr = v0 + j * vstride;
        den += w;
        for (c = 0; c < d; ++c) out[c] += w * bf16_value(vr[c]);
    }
    for (c = 0; c < d; ++c) out[c] /= den;
    free(q);
    free(s);
}

/*
 * Verification attention.  q [B, n_q, H_q, d], k/v [B, L_cap, H_kv, d],
 * out [B, n_q, H_q, d] (double).  The n_q = gamma+1 speculated tokens occupy
 * cache positions [len-n_q, len); query row i sees positions 0..len-n_q+i.
 * Query head hq reads KV head hq / (H_q/H_kv).  len = seq_len[b] clamped to
 * [0, L_cap].
 */
int oracle_verify_attn(int B, int H_q, int H_kv, int d, int L_cap, int n_q,
                       const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *seq_len, double *out)
{
    if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv || d <= 0 || n_q <= 0) return -1;
    const int G = H_q / H_kv;
    const double scale = 1.0 / sqrt((double)d);
    long total = (long)B * n_q * H_q;
    long t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < total; ++t) {
        int hq = (int)(t % H_q);
        int i = (int)((t / H_q) % n_q);
        int b = (int)(t / ((long)H_q * n_q));
        int h = hq / G;
        int len = clamp_len(seq_len[b], L_cap);
        int n_vis = len - n_q + i + 1;
        if (n_vis > len) n_vis = len;
        const uint16_t *qrow = q + (((long)b * n_q + i) * H_q + hq) * d;
        const uint16_t *k0 = k + ((long)b * L_cap * H_kv + h) * d;
        const uint16_t *v0 = v + ((long)b * L_cap * H_kv + h) * d;
        attend_one(qrow, d, scale, k0, (long)H_kv * d, v0, (long)H_kv * d, n_vis,
                   out + (((long)b * n_q + i) * H_q + hq) * d);
    }
    return 0;
}

/*
 * Draft attention over the compact draft cache.  q [B, 1, H_q, d],
 * kc/vc [B, H_kv, cap, d] (head-major), out [B, 1, H_q, d].  The single query
 * sees rows 0..len-1 of its KV head, len = draft_len[b] clamped to [0, cap].
 */
int oracle_draft_attn(int B, int H_q, int H_kv, int d, int cap,
                      const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                      const int32_t *draft_len, double *out)
{
    if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv || d <= 0 || cap < 0) return -1;
    const int G = H_q / H_kv;
    const double scale = 1.0 / sqrt((double)d);
    long total = (long)B * H_q;
    long t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < total; ++t) {
        int hq = (int)(t % H_q);
        int b = (int)(t / H_q);
        int h = hq / G;
        int len = clamp_len(draft_len[b], cap);
        const uint16_t *k0 = kc + ((long)b * H_kv + h) * cap * d;
        const uint16_t *v0 = vc + ((long)b * H_kv + h) * cap * d;
        attend_one(q + ((long)b * H_q + hq) * d, d, scale, k0, d, v0, d, len,
                   out + ((long)b * H_q + hq) * d);
    }
    return 0;
}

/*
 * StreamingLLM selection: the first n_sink positions (attention sinks) and the
 * last n_recent positions of each sequence, ascending, without duplicates.
 * idx [B, H_kv, n_sink+n_recent] (the same set for every KV head), entries
 * past n_sel[b] are -1.
 */
int oracle_streaming_select(const int32_t *seq_len, int B, int H_kv,
                            int n_sink, int n_recent, int32_t *idx, int32_t *n_sel)
{
    if (B < 0 || H_kv <= 0 || n_sink < 0 || n_recent < 0) return -1;
    const int width = n_sink + n_recent;
    int b, h, j;
    for (b = 0; b < B; ++b) {
        int len = seq_len[b] < 0 ? 0 : seq_len[b];
        int32_t *row0 = idx + (long)b * H_kv * width;
        int n = 0;
        int sink_end = len < n_sink ? len : n_sink;
        for (j = 0; j < sink_end; ++j) row0[n++] = j;
        int rec_begin = len - n_recent;
        if (rec_begin < n_sink) rec_begin = n_sink;
        for (j = rec_begin; j < len; ++j) row0[n++] = j;
        for (j = n; j < width; ++j) row0[j] = -1;
        for (h = 1; h < H_kv; ++h) memcpy(row0 + (long)h * width, row0, sizeof(int32_t) * width);
        n_sel[b] = n;
    }
    return 0;
}

/*
 * Gather of selected KV rows into the compact draft cache:
 *   kc[b, h, i] = k[b, idx[b, h, i], h], vc likewise, for i < n_idx.
 * idx [B, H_kv, n_idx].  An index outside [0, L_cap) (the -1 padding of a
 * short selection) writes a zero row.  Rows n_idx..cap-1 are left untouched.
 */
int oracle_gather_kv(int B, int H_kv, int d, int L_cap, const uint16_t *k, const uint16_t *v,
                     const int32_t *idx, int n_idx, int cap, uint16_t *kc, uint16_t *vc)
{
    if (B < 0 || H_kv <= 0 || d <= 0 || n_idx < 0 || n_idx > cap) return -1;
    int b, h, i;
    for (b = 0; b < B; ++b)
        for (h = 0; h < H_kv; ++h)
            for (i = 0; i < n_idx; ++i) {
                int32_t pos = idx[((long)b * H_kv + h) * n_idx + i];
                uint16_t *kd = kc + (((long)b * H_kv + h) * cap + i) * d;
                uint16_t *vd = vc + (((long)b * H_kv + h) * cap + i) * d;
                if (pos < 0 || pos >= L_cap) {
                    memset(kd, 0, sizeof(uint16_t) * d);
                    memset(vd, 0, sizeof(uint16_t) * d);
                } else {
                    memcpy(kd, k + (((long)b * L_cap + pos) * H_kv + h) * d, sizeof(uint16_t) * d);
                    memcpy(vd, v + (((long)b * L_cap + pos) * H_kv + h) * d, sizeof(uint16_t) * d);
                }
            }
    return 0;
}

/*
 * SnapKV observation-window scores.  For each sequence (length L = seq_len[b]
 * clamped to [0, L_cap]) and KV head h, the last w prompt positions are the
 * observation window; window row r sits at position L-w+r and its query for
 * head hq is q_win[b, r, hq, :] (q_win is [B, w, H_q, d]).  Row r attends
 * causally to positions 0..L-w+r with the full softmax.  The score of
 * position j is the sum, over the window rows and the G query heads of the KV
 * group, of that row's softmax probability at j:
 *   score[b, h, j] = sum_{hq in group h} sum_r softmax_r(j).
 * Written for every j < L (window positions included), zero for j >= L;
 * score is [B, H_kv, L_cap].  Sequences with L < w score nothing.
 */
int oracle_snapkv_scores(int B, int H_q, int H_kv, int d, int L_cap, int w,
                         const uint16_t *q_win, const uint16_t *k,
                         const int32_t *seq_len, double *score)
{
    if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv || d <= 0 || w <= 0) return -1;
    const int G = H_q / H_kv;
    const double scale = 1.0 / sqrt((double)d);
    long pairs = (long)B * H_kv;
    long p;
#pragma omp parallel for schedule(dynamic, 1)
    for (p = 0; p < pairs; ++p) {
        int b = (int)(p / H_kv), h = (int)(p % H_kv);
        int L = clamp_len(seq_len[b], L_cap);
        double *sc = score + p * L_cap;
        long j;
        int c, g, r;
        for (j = 0; j < L_cap; ++j) sc[j] = 0.0;
        if (L < w) continue;
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        for (g = 0; g < G; ++g) {
            int hq = h * G + g;
            for (r = 0; r < w; ++r) {
                const uint16_t *qrow = q_win + (((long)b * w + r) * H_q + hq) * d;
                int n_vis = L - w + r + 1;
                for (c = 0; c < d; ++c) q[c] = bf16_value(qrow[c]);
                double smax = -INFINITY;
                for (j = 0; j < n_vis; ++j) {
                    const uint16_t *kr = k + (((long)b * L_cap + j) * H_kv + h) * d;
                    double acc = 0.0;
                    for (c = 0; c < d; ++c) acc += q[c] * bf16_value(kr[c]);
                    s[j] = scale * acc;
                    if (s[j] > smax) smax = s[j];
                }
                double den = 0.0;
                for (j = 0; j < n_vis; ++j) den += exp(s[j] - smax);
                for (j = 0; j < n_vis; ++j) sc[j] += exp(s[j] - smax) / den;
            }
        }
        free(q);
        free(s);
    }
    return 0;
}

/*
 * One-dimensional max pooling with stride 1 and an odd kernel, window clipped
 * at both ends: out[j] = max_{|t-j| <= kernel/2, 0 <= t < n} in[t].
 */
int oracle_maxpool1d(const double *in, int n, int kernel, double *out)
{
    if (n < 0 || kernel <= 0 || (kernel & 1) == 0) return -1;
    const int half = kernel / 2;
    int j, t;
    for (j = 0; j < n; ++j) {
        double m = -INFINITY;
        for (t = j - half; t <= j + half; ++t)
            if (t >= 0 && t < n && in[t] > m) m = in[t];
        out[j] = m;
    }
    return 0;
}

typedef struct { double key; int pos; } ranked_t;

/* Larger pooled score first; equal scores by smaller position. */
static int by_score_desc(const void *a, const void *b)
{
    const ranked_t *x = (const ranked_t *)a, *y = (const ranked_t *)b;
    if (x->key > y->key) return -1;
    if (x->key < y->key) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int by_int_asc(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * SnapKV selection.  Scores (oracle_snapkv_scores) over the prefix
 * [0, L-w) are max-pooled with pool_kernel, the budget-w positions with the
 * largest pooled score are kept (ties to the smaller position), sorted
 * ascending, and the w observation-window positions [L-w, L) are appended.
 * When L <= budget every position 0..L-1 is kept.  idx [B, H_kv, budget],
 * entries past n_sel[b] are -1.  pooled (optional, [B, H_kv, L_cap]) receives
 * the pooled prefix scores (zero elsewhere) for margin analysis.
 */
int oracle_snapkv_select(int B, int H_q, int H_kv, int d, int L_cap,
                         const uint16_t *q_win, const uint16_t *k, const int32_t *seq_len,
                         int w, int pool_kernel, int budget,
                         int32_t *idx, int32_t *n_sel, double *pooled)
{
    if (budget < w || w <= 0 || pool_kernel <= 0 || (pool_kernel & 1) == 0) return -1;
    long pairs = (long)B * H_kv;
    double *score = (double *)malloc(sizeof(double) * (size_t)(pairs * L_cap));
    int rc = oracle_snapkv_scores(B, H_q, H_kv, d, L_cap, w, q_win, k, seq_len, score);
    if (rc) { free(score); return rc; }
    const int k_top = budget - w;
    long p;
    for (p = 0; p < pairs; ++p) {
        int b = (int)(p / H_kv);
        int L = clamp_len(seq_len[b], L_cap);
        int32_t *out = idx + p * budget;
        double *pool_row = pooled ? pooled + p * L_cap : NULL;
        int j, n = 0;
        if (pool_row) for (j = 0; j < L_cap; ++j) pool_row[j] = 0.0;
        if (L <= budget) {
            for (j = 0; j < L; ++j) out[n++] = j;
        } else {
            int m = L - w;
            double *pl = (double *)malloc(sizeof(double) * (size_t)m);
            ranked_t *rk = (ranked_t *)malloc(sizeof(ranked_t) * (size_t)m);
            oracle_maxpool1d(score + p * L_cap, m, pool_kernel, pl);
            for (j = 0; j < m; ++j) { rk[j].key = pl[j]; rk[j].pos = j; }
            qsort(rk, (size_t)m, sizeof(ranked_t), by_score_desc);
            for (j = 0; j < k_top; ++j) out[n++] = rk[j].pos;
            qsort(out, (size_t)k_top, sizeof(int32_t), by_int_asc);
            for (j = m; j < L; ++j) out[n++] = j;
            if (pool_row) for (j = 0; j < m; ++j) pool_row[j] = pl[j];
            free(rk);
            free(pl);
        }
        for (j = n; j < budget; ++j) out[j] = -1;
        if ((p % H_kv) == 0) n_sel[b] = n;
    }
    free(score);
    return 0;
}

/*
 * Lengths of one speculative step (section 3.1: gamma draft tokens are
 * verified together with the pending token, n_acc of the drafts are kept and
 * one token is emitted, so the sequence gains n_acc + 1 cached positions).
 * For each sequence: len = len_in + (n_acc ? n_acc + 1 : 0), clamped to
 * [0, L_cap]; len_out = len; table[j * B + b] = min(len + j, L_cap) for
 * j = 0 .. gamma+1 (the lengths that draft step j appends to and that the
 * verification of the gamma+1 block sees).
 */
int oracle_step_lengths(int B, int gamma, int L_cap, const int32_t *len_in, const int32_t *n_acc, int32_t *len_out,
                        int32_t *table)
{
    int b, j;
    if (B <= 0 || gamma < 0 || L_cap <= 0) return -1;
    for (b = 0; b < B; ++b) {
        long len = len_in[b];
        if (n_acc) len += (long)n_acc[b] + 1;
        if (len < 0) len = 0;
        if (len > L_cap) len = L_cap;
        len_out[b] = (int32_t)len;
        for (j = 0; j <= gamma + 1; ++j) table[(long)j * B + b] = (int32_t)(len + j < L_cap ? len + j : L_cap);
    }
    return 0;
}

/*
 * Draft-cache update: keeps the compact draft cache equal to the static
 * selection as the sequence grows by accepted tokens and shrinks when
 * speculated tokens are rejected (section 4.4: the static drafts select once
 * and then only append; section 3.1: after verification the cache keeps the
 * accepted prefix).  Two layouts of kc/vc [B, H_kv, cap, d]:
 *   ring > 0 (StreamingLLM, section 5.1): position q < origin[b] (a sink)
 *     sits at slot q; position q >= origin[b] at slot
 *     origin[b] + (q - origin[b]) mod ring, so the ring holds the last `ring`
 *     positions; after the update the occupied slots hold exactly positions
 *     [0, min(len, origin)) and [max(origin, len - ring), len).
 *   ring == 0 (SnapKV, section 5.2): slots [0, base[b]) hold the rows chosen
 *     at selection time; position q >= origin[b] (the length at selection)
 *     is appended at slot base[b] + q - origin[b].
 * Rows of positions >= len_valid[b] in the compact cache are stale (drafted
 * by the sparse model, or never written); len_old[b] is the length the
 * cache was last brought to, len_new[b] the new length; all three clamp to
 * [0, L_cap] and len_valid to at most min(len_old, len_new).  The update
 * copies from the full cache k/v [B, L_cap, H_kv, d] every position of the
 * new window at or past len_valid, and (ring layout) restores each slot that
 * a position in [len_new, len_old) overwrote with the window position it had
 * displaced (p - ring).  draft_len[b] receives the occupied slot count,
 * clamped to cap.  Returns the number of row writes skipped because their
 * slot was at or past cap, or -1 on invalid arguments.
 */
int oracle_draft_cache_update(int B, int H_kv, int d, int L_cap, const uint16_t *k, const uint16_t *v,
                              const int32_t *len_valid, const int32_t *len_old, const int32_t *len_new,
                              const int32_t *origin, const int32_t *base, int ring, int cap,
                              uint16_t *kc, uint16_t *vc, int32_t *draft_len)
{
    if (B < 0 || H_kv <= 0 || d <= 0 || L_cap < 0 || ring < 0 || cap <= 0) return -1;
    if (ring == 0 && !base) return -1;
    int skipped = 0, b, h;
    for (b = 0; b < B; ++b) {
        const int lo = clamp_len(len_old[b], L_cap), ln = clamp_len(len_new[b], L_cap);
        int lv = clamp_len(len_valid[b], L_cap);
        if (lv > lo) lv = lo;
        if (lv > ln) lv = ln;
        const int o = origin[b] < 0 ? 0 : origin[b];
        long n_ops = 0, cap_ops = 2L * (ring > 0 ? ring : 0) + (ln > lv ? ln - lv : 0) + 1;
        long *src = (long *)malloc(sizeof(long) * (size_t)cap_ops);
        long *dst = (long *)malloc(sizeof(long) * (size_t)cap_ops);
        int q, p, dl;
        if (ring > 0) {
            for (q = lv; q < ln; ++q) {
                if (q >= o && q < ln - ring) continue;          /* displaced before the end */
                src[n_ops] = q;
                dst[n_ops++] = q < o ? q : o + (q - o) % ring;
            }
            for (p = ln; p < lo && p < ln + ring; ++p) {
                if (p < o) continue;
                q = p - ring;
                if (q < o || q >= lv) continue;
                src[n_ops] = q;
                dst[n_ops++] = o + (p - o) % ring;
            }
            dl = ln <= o ? ln : o + ((ln - o) < ring ? (ln - o) : ring);
        } else {
            const int bs = base[b] < 0 ? 0 : base[b];
            for (q = (lv > o ? lv : o); q < ln; ++q) {
                src[n_ops] = q;
                dst[n_ops++] = bs + (q - o);
            }
            dl = bs + (ln > o ? ln - o : 0);
        }
        long i;
        for (i = 0; i < n_ops; ++i) {
            if (dst[i] >= cap) { ++skipped; continue; }
            for (h = 0; h < H_kv; ++h) {
                const size_t from = (((size_t)b * L_cap + (size_t)src[i]) * H_kv + h) * d;
                const size_t to = (((size_t)b * H_kv + h) * cap + (size_t)dst[i]) * d;
                memcpy(kc + to, k + from, sizeof(uint16_t) * (size_t)d);
                memcpy(vc + to, v + from, sizeof(uint16_t) * (size_t)d);
            }
        }
        draft_len[b] = dl < cap ? dl : cap;
        free(src);
        free(dst);
    }
    return skipped;
}

/*
 * Top-K attention draft (section 1, Figure 1(c) and section 4.4: the
 * dynamic per-query selection that the pages use as the acceptance-rate
 * upper bound).  For query head hq of sequence b, with len = seq_len[b]
 * clamped to [0, L_cap], the scores are s_j = scale * q . k_j over the whole
 * prefix j < len (KV head hq / (H_q/H_kv)).  The top_k positions with the
 * largest s_j are kept (equal scores: the smaller position first); when
 * len <= top_k every position is kept.  The output is softmax attention over
 * the kept positions only:  o = sum_{j in S} softmax_{S}(s)_j v_j.
 * q [B, 1, H_q, d], k/v [B, L_cap, H_kv, d], out [B, 1, H_q, d] (double).
 * idx [B, H_q, top_k] receives the kept positions in ascending order, -1
 * past min(len, top_k).  scores (optional, [B, H_q, L_cap]) receives s_j for
 * j < len and 0 elsewhere, for margin analysis.
 */
int oracle_topk_attn(int B, int H_q, int H_kv, int d, int L_cap,
                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const int32_t *seq_len, int top_k,
                     double *out, int32_t *idx, double *scores)
{
    if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv || d <= 0 || L_cap < 0 || top_k <= 0) return -1;
    const int G = H_q / H_kv;
    const double scale = 1.0 / sqrt((double)d);
    long unit;
#pragma omp parallel for schedule(dynamic)
    for (unit = 0; unit < (long)B * H_q; ++unit) {
        const int b = (int)(unit / H_q), hq = (int)(unit % H_q), hk = hq / G;
        const int len = clamp_len(seq_len[b], L_cap);
        const uint16_t *qrow = q + ((long)b * H_q + hq) * d;
        double *o = out + ((long)b * H_q + hq) * d;
        int32_t *sel = idx + unit * top_k;
        double *srow = scores ? scores + unit * L_cap : NULL;
        int c, j, n;
        for (c = 0; c < d; ++c) o[c] = 0.0;
        if (srow) for (j = 0; j < L_cap; ++j) srow[j] = 0.0;
        for (j = 0; j < top_k; ++j) sel[j] = -1;
        if (len == 0) continue;

        ranked_t *rk = (ranked_t *)malloc(sizeof(ranked_t) * (size_t)len);
        for (j = 0; j < len; ++j) {
            const uint16_t *kr = k + (((long)b * L_cap + j) * H_kv + hk) * d;
            double acc = 0.0;
            for (c = 0; c < d; ++c) acc += bf16_value(qrow[c]) * bf16_value(kr[c]);
            rk[j].key = scale * acc;
            rk[j].pos = j;
            if (srow) srow[j] = rk[j].key;
        }
        n = len <= top_k ? len : top_k;
        if (len > top_k) qsort(rk, (size_t)len, sizeof(ranked_t), by_score_desc);
        for (j = 0; j < n; ++j) sel[j] = rk[j].pos;
        qsort(sel, (size_t)n, sizeof(int32_t), by_int_asc);

        double smax = -INFINITY, den = 0.0;
        for (j = 0; j < n; ++j) if (rk[j].key > smax) smax = rk[j].key;
        for (j = 0; j < n; ++j) {
            const double wgt = exp(rk[j].key - smax);
            const uint16_t *vr = v + (((long)b * L_cap + rk[j].pos) * H_kv + hk) * d;
            den += wgt;
            for (c = 0; c < d; ++c) o[c] += wgt * bf16_value(vr[c]);
        }
        for (c = 0; c < d; ++c) o[c] /= den;
        free(rk);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* PQCache-style dynamic selection (section 4.4, Figure 5: dynamic KV          */
/* selection by product quantisation of the keys).  Keys of each (sequence,   */
/* KV head) split into M sub-vectors of d/M channels; subspace m has C         */
/* centroids.  codebook [B, H_kv, M, C, d/M] fp32, codes [B, H_kv, L_cap, M]   */
/* uint8 (head-major: one (sequence, head)'s codes are contiguous).            */
/* ------------------------------------------------------------------------ */

/*
 * Encode: code[j][m] = the centroid c minimising sum_i (k_j[m*ds+i] - c_i)^2
 * (fp64 from the bf16 key and fp32 centroid; equal distances: the smaller c),
 * for every position j < L_cap.  gap (optional, [B, H_kv, L_cap, M]) receives
 * second-best minus best distance for margin analysis.
 */
int oracle_pq_encode(int B, int H_kv, int d, int L_cap, const uint16_t *k, int M, int C,
                     const float *codebook, uint8_t *codes, double *gap)
{
    if (B < 0 || H_kv <= 0 || d <= 0 || M <= 0 || d % M || C <= 0 || C > 256 || L_cap < 0) return -1;
    const int ds = d / M;
    long unit;
#pragma omp parallel for schedule(static)
    for (unit = 0; unit < (long)B * L_cap * H_kv; ++unit) {
        const int h = (int)(unit % H_kv);
        const long bj = unit / H_kv;
        const int b = (int)(bj / L_cap), j = (int)(bj % L_cap);
        const uint16_t *kr = k + unit * d;
        const size_t out_row = ((size_t)b * H_kv + h) * L_cap + j;
        int m, c, i;
        for (m = 0; m < M; ++m) {
            const float *cb = codebook + (((size_t)b * H_kv + h) * M + m) * (size_t)C * ds;
            double best = INFINITY, second = INFINITY;
            int arg = 0;
            for (c = 0; c < C; ++c) {
                double dist = 0.0;
                for (i = 0; i < ds; ++i) {
                    const double t = bf16_value(kr[m * ds + i]) - (double)cb[(size_t)c * ds + i];
                    dist += t * t;
                }
                if (dist < best) { second = best; best = dist; arg = c; }
                else if (dist < second) second = dist;
            }
            codes[out_row * M + m] = (uint8_t)arg;
            if (gap) gap[out_row * M + m] = second - best;
        }
    }
    return 0;
}

/*
 * Update (one Lloyd step after an encode): centroid c of subspace m becomes
 * the fp64 mean of the sub-vectors of the positions j < seq_len[b] coded c,
 * rounded to fp32; a centroid with no position keeps its value.
 */
int oracle_pq_update(int B, int H_kv, int d, int L_cap, const uint16_t *k, const int32_t *seq_len, int M, int C,
                     const uint8_t *codes, float *codebook)
{
    if (B < 0 || H_kv <= 0 || d <= 0 || M <= 0 || d % M || C <= 0 || C > 256 || L_cap < 0) return -1;
    const int ds = d / M;
    long unit;
#pragma omp parallel for schedule(static)
    for (unit = 0; unit < (long)B * H_kv * M; ++unit) {
        const int m = (int)(unit % M);
        const int h = (int)((unit / M) % H_kv);
        const int b = (int)(unit / ((long)M * H_kv));
        const int len = clamp_len(seq_len[b], L_cap);
        double *sum = (double *)calloc((size_t)C * ds, sizeof(double));
        long *cnt = (long *)calloc((size_t)C, sizeof(long));
        int j, i, c;
        for (j = 0; j < len; ++j) {
            const size_t row = ((size_t)b * L_cap + j) * H_kv + h;
            c = codes[(((size_t)b * H_kv + h) * L_cap + j) * M + m];
            if (c >= C) continue;
            cnt[c]++;
            for (i = 0; i < ds; ++i) sum[(size_t)c * ds + i] += bf16_value(k[row * d + m * ds + i]);
        }
        float *cb = codebook + (size_t)unit * C * ds;
        for (c = 0; c < C; ++c)
            if (cnt[c] > 0)
                for (i = 0; i < ds; ++i) cb[(size_t)c * ds + i] = (float)(sum[(size_t)c * ds + i] / (double)cnt[c]);
        free(sum);
        free(cnt);
    }
    return 0;
}

/*
 * PQ draft attention.  For query head hq (KV head hk = hq / G) of sequence b:
 * LUT[m][c] = scale * sum_i q[m*ds+i] * codebook[b,hk,m,c,i]; approximate
 * score a_j = sum_m LUT[m][codes[b,j,hk,m]] for j < len; the top_k positions
 * by a_j are kept (equal: the smaller position; all when len <= top_k); the
 * output is softmax attention with the EXACT scores scale * q . k_j over the
 * kept positions.  idx [B, H_q, top_k] ascending, -1 padded; approx
 * (optional, [B, H_q, L_cap]) receives a_j (0 past len).
 */
int oracle_pq_attn(int B, int H_q, int H_kv, int d, int L_cap, const uint16_t *q, const uint16_t *k,
                   const uint16_t *v, const int32_t *seq_len, int M, int C, const float *codebook,
                   const uint8_t *codes, int top_k, double *out, int32_t *idx, double *approx)
{
    if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv || d <= 0 || M <= 0 || d % M || C <= 0 || C > 256 ||
        top_k <= 0 || L_cap < 0)
        return -1;
    const int G = H_q / H_kv, ds = d / M;
    const double scale = 1.0 / sqrt((double)d);
    long unit;
#pragma omp parallel for schedule(dynamic)
    for (unit = 0; unit < (long)B * H_q; ++unit) {
        const int b = (int)(unit / H_q), hq = (int)(unit % H_q), hk = hq / G;
        const int len = clamp_len(seq_len[b], L_cap);
        const uint16_t *qr = q + ((long)b * H_q + hq) * d;
        double *o = out + unit * d;
        int32_t *sel = idx + unit * top_k;
        double *arow = approx ? approx + unit * L_cap : NULL;
        int c, i, j, m, n;
        for (i = 0; i < d; ++i) o[i] = 0.0;
        for (j = 0; j < top_k; ++j) sel[j] = -1;
        if (arow) for (j = 0; j < L_cap; ++j) arow[j] = 0.0;
        if (len == 0) continue;
        double *lut = (double *)malloc(sizeof(double) * (size_t)M * C);
        for (m = 0; m < M; ++m)
            for (c = 0; c < C; ++c) {
                const float *cv = codebook + ((((size_t)b * H_kv + hk) * M + m) * C + c) * ds;
                double acc = 0.0;
                for (i = 0; i < ds; ++i) acc += bf16_value(qr[m * ds + i]) * (double)cv[i];
                lut[(size_t)m * C + c] = scale * acc;
            }
        ranked_t *rk = (ranked_t *)malloc(sizeof(ranked_t) * (size_t)len);
        for (j = 0; j < len; ++j) {
            const uint8_t *cr = codes + (((size_t)b * H_kv + hk) * L_cap + j) * M;
            double a = 0.0;
            for (m = 0; m < M; ++m) a += lut[(size_t)m * C + (cr[m] < C ? cr[m] : 0)];
            rk[j].key = a;
            rk[j].pos = j;
            if (arow) arow[j] = a;
        }
        n = len <= top_k ? len : top_k;
        if (len > top_k) qsort(rk, (size_t)len, sizeof(ranked_t), by_score_desc);
        for (j = 0; j < n; ++j) sel[j] = rk[j].pos;
        qsort(sel, (size_t)n, sizeof(int32_t), by_int_asc);
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        double smax = -INFINITY, den = 0.0;
        for (j = 0; j < n; ++j) {
            const uint16_t *kr = k + (((size_t)b * L_cap + sel[j]) * H_kv + hk) * d;
            double acc = 0.0;
            for (i = 0; i < d; ++i) acc += bf16_value(qr[i]) * bf16_value(kr[i]);
            s[j] = scale * acc;
            if (s[j] > smax) smax = s[j];
        }
        for (j = 0; j < n; ++j) {
            const double w = exp(s[j] - smax);
            const uint16_t *vr = v + (((size_t)b * L_cap + sel[j]) * H_kv + hk) * d;
            den += w;
            for (i = 0; i < d; ++i) o[i] += w * bf16_value(vr[i]);
        }
        for (i = 0; i < d; ++i) o[i] /= den;
        free(s);
        free(rk);
        free(lut);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Speculative sampling.                                                     */
/* ------------------------------------------------------------------------ */

/* p = softmax(logits) at temperature 1, in double. */
static void softmax_row(const float *logits, int V, double *p)
{
    double m = -INFINITY, s = 0.0;
    int t;
    for (t = 0; t < V; ++t) if ((double)logits[t] > m) m = logits[t];
    for (t = 0; t < V; ++t) { p[t] = exp((double)logits[t] - m); s += p[t]; }
    for (t = 0; t < V; ++t) p[t] /= s;
}

/*
 * Inverse-CDF draw from unnormalised weights wt: the smallest t whose running
 * sum exceeds u * W, W = sum of the weights.  If rounding leaves no such t,
 * the last token with positive weight.  *amb is raised when u*W lies within
 * 1e-7 * W of the running sum at either edge of the chosen token: a single
 * token of a 128K vocabulary is narrower than 1e-4 of the total, so the edge
 * margin is set by the precision of a single-precision evaluation of the same
 * sums (per-logit errors ~1e-6, normalisers and running sums carried in higher
 * precision), not by the 1e-4 acceptance margin.  *edge (nullable) receives
 * the distance from u*W to the nearer inner edge of the chosen token, divided
 * by W (0 when the fallback was taken).
 */
static int inverse_cdf(const double *wt, int V, double u, int *amb, double *edge)
{
    double W = 0.0, c = 0.0, prev;
    int t, last = V - 1;
    for (t = 0; t < V; ++t) W += wt[t];
    for (t = V - 1; t >= 0; --t) if (wt[t] > 0.0) { last = t; break; }
    const double target = u * W, tol = 1e-7 * W;
    for (t = 0; t < V; ++t) {
        prev = c;
        c += wt[t];
        if (c > target) {
            double e = INFINITY;
            if (t > 0) e = target - prev;
            if (t < V - 1 && c - target < e) e = c - target;
            if (e < tol) ++*amb;
            if (edge) *edge = e / W;
            return t;
        }
    }
    ++*amb;
    if (edge) *edge = 0.0;
    return last;
}

/* Argmax (ties to the smaller token); *gap receives the top-2 logit gap. */
static int argmax_row(const float *logits, int V, int *amb, double *gap)
{
    int t, a = 0;
    for (t = 1; t < V; ++t) if (logits[t] > logits[a]) a = t;
    double second = -INFINITY;
    for (t = 0; t < V; ++t) if (t != a && (double)logits[t] > second) second = logits[t];
    *gap = (double)logits[a] - second;
    if (*gap < 1e-4) ++*amb;
    return a;
}

/*
 * Resample weights of one position: max(0, p - q) with p = softmax(target_row)
 * and q = softmax(draft_row), or p itself when that residual is all zero or
 * draft_row is NULL (the bonus draw).  Unnormalised; the draw takes the
 * smallest token whose running sum exceeds u times their total.
 */
static void resample_weights_into(const float *target_row, const float *draft_row, int V, double *p, double *q,
                                  double *w)
{
    int t;
    double W = 0.0;
    softmax_row(target_row, V, p);
    if (!draft_row) {
        for (t = 0; t < V; ++t) w[t] = p[t];
        return;
    }
    softmax_row(draft_row, V, q);
    for (t = 0; t < V; ++t) { w[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0; W += w[t]; }
    if (!(W > 0.0)) for (t = 0; t < V; ++t) w[t] = p[t];
}

int oracle_resample_weights(const float *target_row, const float *draft_row, int V, double *w)
{
    if (V <= 0) return -1;
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    resample_weights_into(target_row, draft_row, V, p, q, w);
    free(q);
    free(p);
    return 0;
}

/*
 * Accept / resample for one verification step.
 *   target [B, gamma+1, V], draft [B, gamma, V] fp32 logits; draft_tok
 *   [B, gamma]; u_acc [B, gamma] and u_res [B] uniforms in [0, 1).
 * Sampling mode (greedy == 0): for i = 0..gamma-1 with p = softmax(target_i),
 *   q = softmax(draft_i), x = draft_tok_i: accept iff u_acc_i < p(x)/q(x)
 *   (q(x) = 0 accepts iff p(x) > 0; an x outside [0, V) is rejected).  At the
 *   first rejection emit an inverse-CDF draw (u_res) from max(0, p - q),
 *   or from p when that residual is all zero, and stop.  If all gamma are
 *   accepted emit a bonus draw from softmax(target_gamma).
 * Greedy mode: accept while x equals argmax target_i (ties to the smaller
 *   token); at the first mismatch emit that argmax; bonus = argmax target_gamma.
 * Outputs: n_acc [B] in [0, gamma]; out_tok [B, gamma+1] holds the n_acc
 *   accepted tokens then the emitted one, -1 after; n_amb [B] (nullable)
 *   counts decisions taken near their boundary: |u - p(x)/q(x)| < 1e-4, a
 *   top-2 logit gap below 1e-4, or an inverse-CDF edge within 1e-7 of the
 *   total.
 * Optional margin outputs (nullable), one value per decision on the path
 * taken, NaN where no decision was taken: acc_margin [B, gamma+1] holds at
 *   position i the distance of that position's decision from its boundary --
 *   |u_acc - p(x)/q(x)| in sampling mode (+inf when the decision is exact:
 *   x out of range or q(x) = 0), the top-2 logit gap in greedy mode (also
 *   at the bonus position); draw_margin [B] holds the inverse-CDF edge
 *   distance of the sampled token divided by the total weight (sampling
 *   mode only).
 */
int oracle_spec_accept(int B, int gamma, int V, const float *target, const float *draft,
                       const int32_t *draft_tok, const float *u_acc, const float *u_res,
                       int greedy, int32_t *n_acc, int32_t *out_tok, int32_t *n_amb,
                       double *acc_margin, double *draw_margin)
{
    if (B < 0 || gamma < 0 || V <= 0) return -1;
    int b;
#pragma omp parallel for schedule(dynamic, 1)
    for (b = 0; b < B; ++b) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        double *wt = (double *)malloc(sizeof(double) * (size_t)V);
        int32_t *out = out_tok + (long)b * (gamma + 1);
        int amb = 0, i, acc = gamma, emitted = -1;
        double *am = acc_margin ? acc_margin + (long)b * (gamma + 1) : NULL;
        double gap, edge = NAN;
        for (i = 0; i <= gamma; ++i) out[i] = -1;
        if (am) for (i = 0; i <= gamma; ++i) am[i] = NAN;
        for (i = 0; i < gamma; ++i) {
            const float *tl = target + ((long)b * (gamma + 1) + i) * V;
            int x = draft_tok[(long)b * gamma + i];
            int ok;
            if (greedy) {
                int a = argmax_row(tl, V, &amb, &gap);
                if (am) am[i] = gap;
                ok = (x == a);
                if (!ok) emitted = a;
            } else {
                const float *dl = draft + ((long)b * gamma + i) * V;
                softmax_row(tl, V, p);
                softmax_row(dl, V, q);
                if (am) am[i] = INFINITY;
                if (x < 0 || x >= V) {
                    ok = 0;
                } else if (q[x] > 0.0) {
                    double ratio = p[x] / q[x];
                    double u = u_acc[(long)b * gamma + i];
                    ok = (u < ratio);
                    if (fabs(u - ratio) < 1e-4) ++amb;
                    if (am) am[i] = fabs(u - ratio);
                } else {
                    ok = (p[x] > 0.0);
                }
                if (!ok) {
                    resample_weights_into(tl, dl, V, p, q, wt);
                    emitted = inverse_cdf(wt, V, u_res[b], &amb, &edge);
                }
            }
            if (!ok) { acc = i; break; }
            out[i] = x;
        }
        if (acc == gamma) {
            const float *tl = target + ((long)b * (gamma + 1) + gamma) * V;
            if (greedy) {
                emitted = argmax_row(tl, V, &amb, &gap);
                if (am) am[gamma] = gap;
            } else {
                resample_weights_into(tl, NULL, V, p, q, wt);
                emitted = inverse_cdf(wt, V, u_res[b], &amb, &edge);
            }
        }
        if (draw_margin) draw_margin[b] = edge;
        out[acc] = emitted;
        n_acc[b] = acc;
        if (n_amb) n_amb[b] = amb;
        free(wt);
        free(q);
        free(p);
    }
    return 0;
}
