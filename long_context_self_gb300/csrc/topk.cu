// Top-K attention drafting.
//
// MagicDec (arXiv 2408.11049), section 1 with Figure 1(c), and section 4.4
// "Static vs Dynamic": the dynamic KV selection that the pages use as the
// acceptance-rate upper bound.  Each draft query attends only to the top_k
// positions of the whole KV cache with the largest scaled score
// s_j = q . k_j / sqrt(d) (equal scores: the smaller position first), so the
// search reads the full K cache at every draft step -- the selection cost
// T_select that makes it impractical at large batch.
//
// Two kernels on the caller's stream:
//   topk_scores_kernel       persistent over (sequence, KV head, 64-position
//                            tile); a producer thread streams K tiles with TMA
//                            into a shared-memory ring; each of four consumer
//                            warps forms S^T = K_tile Q^T for 16 positions x the
//                            G query heads of the KV group with mma.sync and
//                            stores the fp32 scores [B, H_q, L_sc].
//   topk_select_attn_kernel  one CTA per (sequence, query head): radix select of
//                            the top_k scores on the order-preserving 32-bit key
//                            (12 + 12 + 8 bit digits).  A long row takes a low
//                            enough threshold bin from a 2048-key sample and
//                            reads the row once (prefetched to L2), collecting
//                            the positions at or above that bin, in ascending
//                            order, into a short shared-memory list; the exact
//                            first digit, the last two digits and the ordered
//                            selection run on that list.  A shorter row, or one
//                            where the sample leaves too few candidates or too
//                            many, histograms the whole row first (the whole
//                            row is searched when the list overflows).  Then
//                            the softmax over the kept scores and the weighted
//                            sum of the kept V rows.
#include "common.cuh"

namespace magicdec {

constexpr int kTkTileN = 64;                     // positions per K tile
constexpr int kTkHalfBytes = kTkTileN * 128;     // 64 positions x 64 channels, bf16
constexpr int kTkConsumers = 4;                  // warps, 16 positions each
constexpr int kTkMaxStages = 8;
constexpr size_t kTkInflightBytes = 128 * 1024;   // score-pass stages per SM (both CTAs), by default
constexpr int kTkNT = 512;                       // threads of the select kernel
constexpr int kTkNW = kTkNT / 32;
constexpr int kTkBins = 4096;
constexpr int kTkMaxTopK = 8192;
constexpr int kTkMaxGroup = 8;                   // query heads per KV head (the mma N extent)
constexpr int kTkSampleMinLen = 8192;            // rows at least this long (and >= 8 top_k) sample the first digit
constexpr int kSelScores = 0, kSelExact = 1, kSelOnly = 2;   // modes of the select kernel

struct TopkScoreParams {
    const __nv_bfloat16 *q;   // [B, 1, H_q, D]
    float *score;             // [B, H_q, L_sc]
    const int32_t *len;       // [B]
    int *err;
    int B, H_q, H_kv, G, L_cap, L_sc, stages;
    float scale;
};

struct TopkSelParams {
    const float *score;       // [B, H_q, L_sc] selection scores
    const __nv_bfloat16 *q;   // [B, 1, H_q, D]   (exact-score mode)
    const __nv_bfloat16 *k;   // [B, L_cap, H_kv, D] (exact-score mode)
    const __nv_bfloat16 *v;   // [B, L_cap, H_kv, D]
    const int32_t *len;       // [B]
    __nv_bfloat16 *out;       // [B, 1, H_q, D]
    int32_t *idx;             // [B, H_q, top_k] or null
    int B, H_q, H_kv, G, L_cap, L_sc, top_k;
    int cand_cap;             // shared-memory candidate slots
    float scale;              // 1/sqrt(D) (exact-score mode)
    int len_sub;              // kSelOnly: window length kept after the selected prefix
    int32_t *n_sel;           // kSelOnly: [B] kept count
    const int32_t *budgets;   // kSelOnly: [B] per-sequence budgets (null: top_k for all)
};

__device__ __forceinline__ int tk_clamp_len(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }

// Position in the flat tile order (sequence, KV head, tile).  prefix[b] = tiles
// of sequences < b per KV head.
struct TkCursor {
    int b, h, ti, ntiles;
};

__device__ __forceinline__ TkCursor tk_locate(long long t, const int *prefix, int B, int H_kv) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)H_kv * prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    TkCursor c;
    c.b = lo;
    c.ntiles = prefix[lo + 1] - prefix[lo];
    const long long local = t - (long long)H_kv * prefix[lo];
    c.h = (int)(local / c.ntiles);
    c.ti = (int)(local - (long long)c.h * c.ntiles);
    return c;
}

// Next tile; only called while another tile remains in the grid's range.
__device__ __forceinline__ void tk_advance(TkCursor &c, const int *prefix, int H_kv) {
    if (++c.ti < c.ntiles) return;
    c.ti = 0;
    if (++c.h < H_kv) return;
    c.h = 0;
    do {
        ++c.b;
        c.ntiles = prefix[c.b + 1] - prefix[c.b];
    } while (c.ntiles == 0);
}

template <int D>
__global__ void __launch_bounds__((kTkConsumers + 1) * 32, 2)
    topk_scores_kernel(const __grid_constant__ CUtensorMap tmk, const TopkScoreParams p) {
    constexpr int HALVES = D / 64;
    constexpr int STAGE_BYTES = HALVES * kTkHalfBytes;
    constexpr int KS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *stage_base = smem;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + (size_t)p.stages * STAGE_BYTES);
    uint64_t *empty_bar = full_bar + kTkMaxStages;
    int *prefix = reinterpret_cast<int *>(empty_bar + kTkMaxStages);   // [B + 1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kTkConsumers);
        }
        mbar_fence_init();
        prefetch_tensormap(&tmk);
    }
    pdl_wait();
    for (int b = tid; b < p.B; b += blockDim.x)
        prefix[b] = (tk_clamp_len(checked(ld_dep(p.len + b), 0, p.L_cap, p.err), p.L_cap) + kTkTileN - 1) / kTkTileN;
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            const int nt = b < p.B ? prefix[b] : 0;
            int x = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (b < p.B) prefix[b] = run + x - nt;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) prefix[p.B] = run;
    }
    __syncthreads();

    const long long T = (long long)p.H_kv * prefix[p.B];
    const int C = gridDim.x, c = blockIdx.x;
    const long long t_begin = T * c / C, t_end = T * (c + 1) / C;
    const int n = (int)(t_end - t_begin);
    if (n <= 0) return;

    if (warp == kTkConsumers) {
        // ------------------------------------------------------- producer (1 thread)
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        TkCursor cur = tk_locate(t_begin, prefix, p.B, p.H_kv);
        int i = 0;
        for (; i < n; ++i) {
            if (i) tk_advance(cur, prefix, p.H_kv);
            const int stage = i % p.stages;
            const uint32_t phase = (uint32_t)(i / p.stages) & 1u;
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) break;
            mbar_arrive_expect_tx(&full_bar[stage], STAGE_BYTES);
            uint8_t *dst = stage_base + (size_t)stage * STAGE_BYTES;
#pragma unroll
            for (int hf = 0; hf < HALVES; ++hf)
                tma_load_4d(dst + hf * kTkHalfBytes, &tmk, hf * 64, cur.h, cur.ti * kTkTileN, cur.b, &full_bar[stage],
                            pol);
        }
        // the copies issued last land before the CTA may exit
        for (int k = i > p.stages ? i - p.stages : 0; k < i; ++k)
            mbar_wait(&full_bar[k % p.stages], (uint32_t)(k / p.stages) & 1u, p.err);
        return;
    }

    // ----------------------------------------------------------- consumers
    // A = K tile rows (16 positions x 16 channels per k-step) via ldmatrix;
    // B = Q^T (16 channels x 8 query heads), loaded straight into fragments.
    const int mat = lane >> 3, rr = lane & 7;
    const int a_row = warp * 16 + (mat & 1) * 8 + rr;
    const int a_half = mat >> 1;
    const int g0 = 2 * (lane & 3), key_l = lane >> 2;
    TkCursor cur = tk_locate(t_begin, prefix, p.B, p.H_kv);
    int qb_b = -1, qb_h = -1;
    uint32_t bq[KS][2];
    for (int i = 0; i < n; ++i) {
        if (i) tk_advance(cur, prefix, p.H_kv);
        if (cur.b != qb_b || cur.h != qb_h) {
            qb_b = cur.b;
            qb_h = cur.h;
            const int nrow = lane >> 2;
            const bool valid = nrow < p.G;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                p.q + ((long long)qb_b * p.H_q + qb_h * p.G + (valid ? nrow : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                bq[ks][0] = valid ? ld_dep_u32(qrow + ks * 8 + (lane & 3)) : 0u;
                bq[ks][1] = valid ? ld_dep_u32(qrow + ks * 8 + 4 + (lane & 3)) : 0u;
            }
        }
        const int stage = i % p.stages;
        const uint32_t phase = (uint32_t)(i / p.stages) & 1u;
        if (!mbar_wait(&full_bar[stage], phase, p.err)) break;
        const uint32_t base = smem_u32(stage_base + (size_t)stage * STAGE_BYTES);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int ch = ks * 2 + a_half;     // 8-channel chunk index over D
            uint32_t a[4];
            ldsm_x4(base + (ch >> 3) * kTkHalfBytes + swz128(a_row, ch & 7), a[0], a[1], a[2], a[3]);
            mma_bf16(acc, a, bq[ks][0], bq[ks][1]);
        }
        fence_proxy_async_smem();   // reads done before TMA may refill the buffer
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);

        const int len = tk_clamp_len(ld_dep(p.len + cur.b), p.L_cap);
        const int pos = cur.ti * kTkTileN + warp * 16 + key_l;
        float *srow = p.score + ((long long)cur.b * p.H_q + (long long)cur.h * p.G) * p.L_sc;
        if (g0 < p.G) {
            if (pos < len) srow[(long long)g0 * p.L_sc + pos] = acc[0] * p.scale;
            if (pos + 8 < len) srow[(long long)g0 * p.L_sc + pos + 8] = acc[2] * p.scale;
        }
        if (g0 + 1 < p.G) {
            if (pos < len) srow[(long long)(g0 + 1) * p.L_sc + pos] = acc[1] * p.scale;
            if (pos + 8 < len) srow[(long long)(g0 + 1) * p.L_sc + pos + 8] = acc[3] * p.scale;
        }
    }
}

// All eight KV heads of a sequence per stage (d = 128, H_kv = 8, G <= 8): a
// stage is 16 positions x 8 heads of K, 32 KB contiguous in the
// [B, L_cap, H_kv, d] cache, loaded as two TMA boxes of 64 channels x 16
// positions x 8 heads from a tensor map whose position stride precedes its
// head stride (each head's 16 rows are consecutive swizzled rows in shared
// memory).  Consumer warp h forms S^T = K_h Q_h^T for head h's 16 positions
// and G query heads.  The per-pair kernel above fetches 256-byte rows 2 KB
// apart; this traversal streams the same bytes faster.
constexpr int kTkHdHeads = 8, kTkHdPos = 16;
constexpr int kTkHdHalf = kTkHdPos * kTkHdHeads * 128;   // 16 KB: one 64-channel half of a stage
constexpr int kTkHdStage = 2 * kTkHdHalf;

__global__ void __launch_bounds__((kTkHdHeads + 1) * 32, 2)
    topk_scores_heads_kernel(const __grid_constant__ CUtensorMap tmk, const TopkScoreParams p) {
    constexpr int D = 128, KS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *stage_base = smem;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + (size_t)p.stages * kTkHdStage);
    uint64_t *empty_bar = full_bar + kTkMaxStages;
    int *prefix = reinterpret_cast<int *>(empty_bar + kTkMaxStages);   // [B + 1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kTkHdHeads);
        }
        mbar_fence_init();
        prefetch_tensormap(&tmk);
    }
    pdl_wait();
    for (int b = tid; b < p.B; b += blockDim.x)
        prefix[b] = (tk_clamp_len(checked(ld_dep(p.len + b), 0, p.L_cap, p.err), p.L_cap) + kTkHdPos - 1) / kTkHdPos;
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            const int nt = b < p.B ? prefix[b] : 0;
            int x = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (b < p.B) prefix[b] = run + x - nt;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) prefix[p.B] = run;
    }
    __syncthreads();

    // flat list of 16-position tiles ordered (sequence, tile), split evenly across CTAs
    const long long T = prefix[p.B];
    const int C = gridDim.x, c = blockIdx.x;
    const long long t_begin = T * c / C, t_end = T * (c + 1) / C;
    const int n = (int)(t_end - t_begin);
    if (n <= 0) return;
    auto seq_of = [&](long long t) {
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        return lo;
    };

    if (warp == kTkHdHeads) {
        // ------------------------------------------------------- producer (1 thread)
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        int i = 0;
        int b = seq_of(t_begin);                       // steps on with t (a sequence's tiles are consecutive)
        for (; i < n; ++i) {
            const long long t = t_begin + i;
            while (t >= prefix[b + 1]) ++b;
            const int pos0 = (int)(t - prefix[b]) * kTkHdPos;
            const int stage = i % p.stages;
            const uint32_t phase = (uint32_t)(i / p.stages) & 1u;
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) break;
            mbar_arrive_expect_tx(&full_bar[stage], kTkHdStage);
            uint8_t *dst = stage_base + (size_t)stage * kTkHdStage;
            tma_load_4d(dst, &tmk, 0, pos0, 0, b, &full_bar[stage], pol);
            tma_load_4d(dst + kTkHdHalf, &tmk, 64, pos0, 0, b, &full_bar[stage], pol);
        }
        // the copies issued last land before the CTA may exit
        for (int k = i > p.stages ? i - p.stages : 0; k < i; ++k)
            mbar_wait(&full_bar[k % p.stages], (uint32_t)(k / p.stages) & 1u, p.err);
        return;
    }

    // ----------------------------------------------------------- consumers
    // Warp h: A = K_h rows (16 positions x 16 channels per k-step) via
    // ldmatrix; B = Q^T of head h's G query heads, loaded into fragments.
    const int h = warp;
    const int mat = lane >> 3, rr = lane & 7;
    const int a_row = h * kTkHdPos + (mat & 1) * 8 + rr;
    const int a_half = mat >> 1;
    const int g0 = 2 * (lane & 3), key_l = lane >> 2;
    int qb_b = -1;
    uint32_t bq[KS][2];
    int b = seq_of(t_begin);
    for (int i = 0; i < n; ++i) {
        const long long t = t_begin + i;
        while (t >= prefix[b + 1]) ++b;
        if (b != qb_b) {
            qb_b = b;
            const int nrow = lane >> 2;
            const bool valid = nrow < p.G;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                p.q + ((long long)b * p.H_q + h * p.G + (valid ? nrow : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                bq[ks][0] = valid ? ld_dep_u32(qrow + ks * 8 + (lane & 3)) : 0u;
                bq[ks][1] = valid ? ld_dep_u32(qrow + ks * 8 + 4 + (lane & 3)) : 0u;
            }
        }
        const int stage = i % p.stages;
        const uint32_t phase = (uint32_t)(i / p.stages) & 1u;
        if (!mbar_wait(&full_bar[stage], phase, p.err)) break;
        const uint32_t base = smem_u32(stage_base + (size_t)stage * kTkHdStage);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int ch = ks * 2 + a_half;     // 8-channel chunk index over D
            uint32_t a[4];
            ldsm_x4(base + (ch >> 3) * kTkHdHalf + swz128(a_row, ch & 7), a[0], a[1], a[2], a[3]);
            mma_bf16(acc, a, bq[ks][0], bq[ks][1]);
        }
        fence_proxy_async_smem();   // reads done before TMA may refill the buffer
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);

        const int len = tk_clamp_len(ld_dep(p.len + b), p.L_cap);
        const int pos = (int)(t - prefix[b]) * kTkHdPos + key_l;
        float *srow = p.score + ((long long)b * p.H_q + (long long)h * p.G) * p.L_sc;
        if (g0 < p.G) {
            if (pos < len) srow[(long long)g0 * p.L_sc + pos] = acc[0] * p.scale;
            if (pos + 8 < len) srow[(long long)g0 * p.L_sc + pos + 8] = acc[2] * p.scale;
        }
        if (g0 + 1 < p.G) {
            if (pos < len) srow[(long long)(g0 + 1) * p.L_sc + pos] = acc[1] * p.scale;
            if (pos + 8 < len) srow[(long long)(g0 + 1) * p.L_sc + pos + 8] = acc[3] * p.scale;
        }
    }
}

// ---------------------------------------------------------------- selection
// Order-preserving key of an fp32 value (larger value -> larger key); 0 marks
// "no position".
__device__ __forceinline__ uint32_t tk_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float tk_unkey(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Inclusive block-wide scan in thread order over kTkNW warps; *total = block sum.
__device__ __forceinline__ int tk_block_scan(int v, int *wsum, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int y = lane < kTkNW ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        if (lane < kTkNW) wsum[lane] = y;
    }
    __syncthreads();
    const int excl = warp ? wsum[warp - 1] : 0;
    *total = wsum[kTkNW - 1];
    __syncthreads();
    return x + excl;
}

// The digit (bin) holding the remaining-th largest counted key, scanning the
// 4096 bins from the top; returns it and the rank left inside that bin.
__device__ __forceinline__ void tk_find_digit(const int *hist, int remaining, int *wsum, int *s_digit, int *s_rem,
                                              int &digit, int &rem_out) {
    constexpr int BPT = kTkBins / kTkNT;
    const int tid = threadIdx.x;
    int cnt[BPT], sum = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        cnt[j] = hist[kTkBins - 1 - BPT * tid - j];
        sum += cnt[j];
    }
    int total;
    const int incl = tk_block_scan(sum, wsum, &total);
    int above = incl - sum;
    if (above < remaining && remaining <= incl) {
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
            if (above < remaining && remaining <= above + cnt[j]) {
                *s_digit = kTkBins - 1 - BPT * tid - j;
                *s_rem = remaining - above;
            }
            above += cnt[j];
        }
    }
    __syncthreads();
    digit = *s_digit;
    rem_out = *s_rem;
    __syncthreads();
}

// Keys of 4 consecutive positions j..j+3 (j % 4 == 0) of a score row; positions
// at or past `hi` give key 0.  The row holds at least len rounded up to 4.
__device__ __forceinline__ void tk_load4(const float *srow, int j, int hi, uint32_t (&k)[4]) {
    if (j < hi) {
        const float4 f = ld_dep_f4(reinterpret_cast<const float4 *>(srow + j));
        k[0] = tk_key(f.x);
        k[1] = j + 1 < hi ? tk_key(f.y) : 0u;
        k[2] = j + 2 < hi ? tk_key(f.z) : 0u;
        k[3] = j + 3 < hi ? tk_key(f.w) : 0u;
    } else {
        k[0] = k[1] = k[2] = k[3] = 0u;
    }
}

// Selection when more than `cand_cap` positions share or pass the first digit
// (long runs of equal scores): the last two digits and the ordered
// compaction run over the whole row, re-read from L2.
__device__ void tk_select_full_row(const float *srow, int len, int top_k, int d1, int rem, int *hist, int *sel,
                                   int *wsum, int *s_digit, int *s_rem) {
    const int tid = threadIdx.x;
    int d2, d3;
    for (int i = tid; i < kTkBins; i += kTkNT) hist[i] = 0;
    __syncthreads();
    for (int j = tid; j < len; j += kTkNT) {
        const uint32_t k = tk_key(srow[j]);
        if ((int)(k >> 20) == d1) atomicAdd(&hist[(k >> 8) & 4095u], 1);
    }
    __syncthreads();
    tk_find_digit(hist, rem, wsum, s_digit, s_rem, d2, rem);
    for (int i = tid; i < kTkBins; i += kTkNT) hist[i] = 0;
    __syncthreads();
    const uint32_t pre = ((uint32_t)d1 << 12) | (uint32_t)d2;
    for (int j = tid; j < len; j += kTkNT) {
        const uint32_t k = tk_key(srow[j]);
        if ((k >> 8) == pre) atomicAdd(&hist[k & 255u], 1);
    }
    __syncthreads();
    tk_find_digit(hist, rem, wsum, s_digit, s_rem, d3, rem);
    const uint32_t tau = (pre << 8) | (uint32_t)d3;
    const int need_eq = rem;
    int gt_seen = 0, eq_seen = 0;
    for (int base = 0; base < len; base += 4 * kTkNT) {
        const int j0 = base + 4 * tid;
        uint32_t kk[4];
        tk_load4(srow, j0, len, kk);
        int ngt = 0, neq = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ngt += kk[e] > tau;
            neq += kk[e] == tau;
        }
        const int packed = (ngt << 16) | neq;
        int total;
        const int excl = tk_block_scan(packed, wsum, &total) - packed;
        int gb = gt_seen + (excl >> 16), eb = eq_seen + (excl & 0xffff);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (kk[e] > tau) {
                sel[gb + min(eb, need_eq)] = j0 + e;
                ++gb;
            } else if (kk[e] == tau) {
                if (eb < need_eq) sel[gb + eb] = j0 + e;
                ++eb;
            }
        }
        gt_seen += total >> 16;
        eq_seen += total & 0xffff;
    }
    (void)top_k;
}

// MODE kSelScores: the selection scores are the exact scaled scores (Top-K
// attention) and weight the kept rows directly.  kSelExact: they are
// approximate (PQ lookup sums) and only choose the rows; the kept rows' exact
// scores are recomputed from K before the softmax.  kSelOnly (SnapKV): rows
// are (sequence, KV head) pooled-score rows; the budget - len_sub largest of
// the first len - len_sub positions are kept and the last len_sub positions
// (the observation window) appended; no attention.
template <int D, int MODE>
__global__ void __launch_bounds__(kTkNT, 3) topk_select_attn_kernel(const TopkSelParams p) {
    constexpr bool EXACT = MODE == kSelExact;
    constexpr int NW = kTkNW;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    int *hist = reinterpret_cast<int *>(smem_raw);                    // [4096]; later [NW][D] partial outputs
    int *cand_pos = hist + kTkBins;                                   // [cand_cap]
    uint32_t *cand_key = reinterpret_cast<uint32_t *>(cand_pos + p.cand_cap);   // [cand_cap]
    int *sel = reinterpret_cast<int *>(cand_key + p.cand_cap);        // [top_k]
    // (in kSelOnly mode p.top_k is the budget, an upper bound of the kept count)
    __shared__ int wsum[32], woff[NW], wcnt[NW];
    __shared__ float s_exmax[NW];
    __shared__ int s_digit, s_rem, s_total, s_over;
    __shared__ unsigned s_maxkey;
    __shared__ float zsum[NW];

    const int hq = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();
    const int full = tk_clamp_len(ld_dep(p.len + b), p.L_cap);
    const int kvh = hq / p.G;
    const long long row = (long long)b * p.H_q + hq;
    const float *srow = p.score + row * p.L_sc;
    __nv_bfloat16 *o = MODE == kSelOnly ? nullptr : p.out + row * D;
    int32_t *idx_row = p.idx ? p.idx + row * p.top_k : nullptr;
    int len = full, top_k = p.top_k;
    if (MODE == kSelOnly) {
        // SnapKV: everything when the sequence fits the budget; else the
        // window is always kept and budget - window prefix positions compete
        const int w = p.len_sub;
        const int budget = p.budgets ? min(max(ld_dep(p.budgets + b), w), p.top_k) : p.top_k;
        if (full <= budget || budget == w) {
            const int keep_from = full <= budget ? 0 : full - w;
            const int n_keep = full - keep_from;
            for (int i = tid; i < p.top_k; i += kTkNT) idx_row[i] = i < n_keep ? keep_from + i : -1;
            if (hq == 0 && tid == 0) p.n_sel[b] = n_keep;
            return;
        }
        len = full - w;
        top_k = budget - w;
    }
    const int n = min(len, top_k);
    if (len == 0) {
        for (int c = tid; c < D; c += kTkNT) o[c] = __float2bfloat16(0.f);
        if (idx_row)
            for (int i = tid; i < top_k; i += kTkNT) idx_row[i] = -1;
        return;
    }
    const bool select = len > top_k;
    if (select && tid == 0 && (reinterpret_cast<uintptr_t>(srow) & 15) == 0) {
        // the two passes below read the row with a few loads in flight per lane:
        // start the whole row towards L2 now so that they wait on L2, not DRAM
        const uint32_t bytes = (uint32_t)((len + 3) & ~3) * 4u;
        for (uint32_t o = 0; o < bytes; o += 16384u)
            bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(srow) + o, min(16384u, bytes - o));
    }
    // warp w owns positions [lo, hi): contiguous segments keep the ascending order
    const int seg = (((len + NW - 1) / NW) + 3) & ~3;
    const int lo = min(len, warp * seg), hi = min(len, lo + seg);

    // 1. first-digit histogram and the largest key.  A long row samples it: one
    //    128-key block per warp at evenly spaced positions (2048 keys) gives the
    //    lowest bin d_lo that still holds about 1.25 top_k (+16) of the row's
    //    keys at or above it, and the exact first digit is then taken over the
    //    candidates (every key of the top_k lies at or above d_lo whenever at
    //    least top_k candidates are found).  A row where that leaves fewer than
    //    top_k candidates, or more than a warp's slots, counts the whole row and
    //    runs the whole-row search.  Shorter rows count the whole row directly.
    const bool sampled = select && len >= kTkSampleMinLen && len >= 8 * top_k;
    auto count_row = [&](bool count) {   // whole-row histogram (when `count`) and the largest key
        uint32_t mk = 0u;
        for (int base = lo; base < hi; base += 4 * 128) {
            uint32_t kk[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) tk_load4(srow, base + 128 * u + 4 * lane, hi, kk[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (kk[u][e] == 0u) continue;
                    mk = max(mk, kk[u][e]);
                    if (count) atomicAdd(&hist[kk[u][e] >> 20], 1);
                }
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o2));
        if (lane == 0) atomicMax(&s_maxkey, mk);
        __syncthreads();
    };
    for (int i = tid; i < kTkBins; i += kTkNT) hist[i] = 0;
    if (tid == 0) {
        s_maxkey = 0u;
        s_digit = 0;   // a search for more keys than were counted leaves these
        s_rem = 0;
    }
    __syncthreads();
    int d_lo = 0;
    if (sampled) {
        const int sb = (int)((long long)len * warp / NW) & ~3;   // sb + 128 <= len
        uint32_t kk[4];
        tk_load4(srow, sb + 4 * lane, sb + 128, kk);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (kk[e] != 0u) atomicAdd(&hist[kk[e] >> 20], 1);
        __syncthreads();
        constexpr int S = NW * 128;
        const int r_s = min(S, (int)((5LL * top_k * S) / (4LL * len)) + 16);
        int r_left;
        tk_find_digit(hist, r_s, wsum, &s_digit, &s_rem, d_lo, r_left);
    } else {
        count_row(select);
    }

    if (select) {
        int d1 = 0, rem1 = 0;
        if (!sampled) {
            tk_find_digit(hist, top_k, wsum, &s_digit, &s_rem, d1, rem1);
            d_lo = d1;
        }
        // 2. candidates = positions whose first digit is >= d_lo.  One pass over
        //    the row; warp w appends its segment's candidates, in ascending order,
        //    to its own R slots of the list (a sampled row also takes the largest
        //    key here: it is always a candidate).
        const int R = p.cand_cap / NW;
        int *my_pos = cand_pos + warp * R;
        uint32_t *my_key = cand_key + warp * R;
        int cnt = 0;
        uint32_t mk = 0u;
        for (int base = lo; base < hi; base += 4 * 128) {
            uint32_t kk[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) tk_load4(srow, base + 128 * u + 4 * lane, hi, kk[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                int c = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) c += kk[u][e] != 0u && (int)(kk[u][e] >> 20) >= d_lo;
                int x = c;
#pragma unroll
                for (int o2 = 1; o2 < 32; o2 <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o2);
                    if (lane >= o2) x += y;
                }
                int at = cnt + x - c;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (kk[u][e] != 0u && (int)(kk[u][e] >> 20) >= d_lo) {
                        mk = max(mk, kk[u][e]);
                        if (at < R) {
                            my_pos[at] = base + 128 * u + 4 * lane + e;
                            my_key[at] = kk[u][e];
                        }
                        ++at;
                    }
                cnt += __shfl_sync(0xffffffffu, x, 31);
            }
        }
        if (sampled) {
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o2));
            if (lane == 0) atomicMax(&s_maxkey, mk);
        }
        if (lane == 0) wcnt[warp] = cnt;
        __syncthreads();
        if (warp == 0) {
            const int c = lane < NW ? wcnt[lane] : 0;
            const bool over = __any_sync(0xffffffffu, c > R);
            int x = c;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o2);
                if (lane >= o2) x += y;
            }
            if (lane < NW) woff[lane] = x - c;
            if (lane == 31) {
                s_total = x;
                s_over = over ? 1 : 0;
            }
        }
        __syncthreads();
        if (sampled) {
            for (int i = tid; i < kTkBins; i += kTkNT) hist[i] = 0;
            __syncthreads();
            if (s_over || s_total < top_k) {
                // the sample missed: count the whole row, search the whole row
                count_row(true);
                tk_find_digit(hist, top_k, wsum, &s_digit, &s_rem, d1, rem1);
                if (tid == 0) s_over = 1;
                __syncthreads();
            } else {
                // the exact first digit, over the candidates
                for (int i = tid; i < NW * R; i += kTkNT) {
                    if (i - (i / R) * R >= wcnt[i / R]) continue;
                    atomicAdd(&hist[cand_key[i] >> 20], 1);
                }
                __syncthreads();
                tk_find_digit(hist, top_k, wsum, &s_digit, &s_rem, d1, rem1);
            }
        }
        const int n_cand = s_total;
        if (s_over) {
            tk_select_full_row(srow, len, top_k, d1, rem1, hist, sel, wsum, &s_digit, &s_rem);
        } else {
            // 3. the last two digits, over the candidates of bin d1 only
            int d2, d3, rem;
            for (int i = tid; i < kTkBins; i += kTkNT) hist[i] = 0;
            __syncthreads();
            for (int i = tid; i < NW * R; i += kTkNT) {
                if (i - (i / R) * R >= wcnt[i / R]) continue;
                const uint32_t k = cand_key[i];
                if ((int)(k >> 20) == d1) atomicAdd(&hist[(k >> 8) & 4095u], 1);
            }
            __syncthreads();
            tk_find_digit(hist, rem1, wsum, &s_digit, &s_rem, d2, rem);
            for (int i = tid; i < kTkBins; i += kTkNT) hist[i] = 0;
            __syncthreads();
            const uint32_t pre = ((uint32_t)d1 << 12) | (uint32_t)d2;
            for (int i = tid; i < NW * R; i += kTkNT) {
                if (i - (i / R) * R >= wcnt[i / R]) continue;
                const uint32_t k = cand_key[i];
                if ((k >> 8) == pre) atomicAdd(&hist[k & 255u], 1);
            }
            __syncthreads();
            tk_find_digit(hist, rem, wsum, &s_digit, &s_rem, d3, rem);
            const uint32_t tau = (pre << 8) | (uint32_t)d3;
            const int need_eq = rem;
            // 4. ordered selection over the candidates: list index g lives in
            //    warp w's slots where woff[w] <= g < woff[w] + wcnt[w]; thread t
            //    takes g in [t*E, (t+1)*E)
            const int E = (n_cand + kTkNT - 1) / kTkNT;
            const int c0 = min(n_cand, tid * E), c1 = min(n_cand, c0 + E);
            int w0 = 0;
            while (w0 + 1 < NW && c0 >= woff[w0 + 1]) ++w0;
            int ngt = 0, neq = 0;
            for (int g = c0, w = w0; g < c1; ++g) {
                while (w + 1 < NW && g >= woff[w + 1]) ++w;
                const uint32_t k = cand_key[w * R + g - woff[w]];
                ngt += k > tau;
                neq += k == tau;
            }
            const int packed = (ngt << 16) | neq;
            int total;
            const int excl = tk_block_scan(packed, wsum, &total) - packed;
            int gb = excl >> 16, eb = excl & 0xffff;
            for (int g = c0, w = w0; g < c1; ++g) {
                while (w + 1 < NW && g >= woff[w + 1]) ++w;
                const int slot = w * R + g - woff[w];
                const uint32_t k = cand_key[slot];
                if (k > tau) {
                    sel[gb + min(eb, need_eq)] = cand_pos[slot];
                    ++gb;
                } else if (k == tau) {
                    if (eb < need_eq) sel[gb + eb] = cand_pos[slot];
                    ++eb;
                }
            }
        }
    } else {
        for (int i = tid; i < len; i += kTkNT) sel[i] = i;
    }
    __syncthreads();
    if (MODE == kSelOnly) {
        // kept prefix positions (ascending), then the window [len, full)
        for (int i = tid; i < p.top_k; i += kTkNT) idx_row[i] = i < n ? sel[i] : (i < n + (full - len) ? len + (i - n) : -1);
        if (hq == 0 && tid == 0) p.n_sel[b] = n + (full - len);
        return;
    }

    // 5. softmax over the kept scores (the largest key is always kept) and the
    //    weighted sum of their V rows.  A V row is LPR lanes x 16 bytes, so one
    //    load instruction of a warp covers RPI rows; part r of warp w takes kept
    //    entries w + NW * (RPI * t + r).
    constexpr int LPR = D / 8;
    constexpr int RPI = 32 / LPR;
    const int sub = lane % LPR, part = lane / LPR;
    if (EXACT) {
        // exact scaled scores of the kept rows, and in the same pass the
        // softmax-weighted sum of their V rows: lane `sub` of a row group dots
        // channels sub*8 .. +7 of q and the K row (the group's lanes sum), then
        // folds the row into its running (max, sum, output) with the online
        // rule; the row groups merge with the log-sum-exp rule at the end
        float qv[8];
        {
            const uint4 qq = ld_dep_u4(reinterpret_cast<const uint4 *>(p.q + row * D + sub * 8));
            const uint32_t w4[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[c]));
                qv[2 * c] = f.x;
                qv[2 * c + 1] = f.y;
            }
        }
        const long long base = ((long long)b * p.L_cap * p.H_kv + kvh) * D + sub * 8;
        const __nv_bfloat16 *kb = p.k + base, *vb = p.v + base;
        const long long kvstride = (long long)p.H_kv * D;
        const float sl = p.scale * kLog2e;
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = 0.f;
        float z = 0.f, mr = -INFINITY;                       // running max in log2 units
        for (int t = 0; warp + NW * RPI * t < n; ++t) {
            const int i = warp + NW * (RPI * t + part);
            uint4 kr = make_uint4(0u, 0u, 0u, 0u), vr = kr;
            if (i < n) {
                const long long off = (long long)sel[i] * kvstride;
                kr = ld_dep_u4(reinterpret_cast<const uint4 *>(kb + off));
                vr = ld_dep_u4(reinterpret_cast<const uint4 *>(vb + off));
            }
            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
            float dot = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kw[c]));
                dot = fmaf(qv[2 * c], f.x, dot);
                dot = fmaf(qv[2 * c + 1], f.y, dot);
            }
#pragma unroll
            for (int o2 = LPR / 2; o2 > 0; o2 >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o2);
            if (i < n) {
                const float s2 = dot * sl, mn = fmaxf(mr, s2);
                const float al = fast_exp2(mr - mn), wgt = fast_exp2(s2 - mn);
                z = fmaf(z, al, wgt);
                const uint32_t vw[4] = {vr.x, vr.y, vr.z, vr.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vw[c]));
                    acc[2 * c] = fmaf(wgt, f.x, acc[2 * c] * al);
                    acc[2 * c + 1] = fmaf(wgt, f.y, acc[2 * c + 1] * al);
                }
                mr = mn;
            }
        }
        // merge the row groups of the warp, then the warps
#pragma unroll
        for (int o2 = LPR; o2 < 32; o2 <<= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, mr, o2), zo = __shfl_xor_sync(0xffffffffu, z, o2);
            const float mn = fmaxf(mr, mo), mu = mn == -INFINITY ? 0.f : mn;
            const float fa = fast_exp2(mr - mu), fb = fast_exp2(mo - mu);
            z = z * fa + zo * fb;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float ao = __shfl_xor_sync(0xffffffffu, acc[c], o2);
                acc[c] = acc[c] * fa + ao * fb;
            }
            mr = mn;
        }
        float *red = reinterpret_cast<float *>(hist);   // [NW][D]; the histogram is no longer read
        if (part == 0) {
#pragma unroll
            for (int c = 0; c < 8; ++c) red[warp * D + sub * 8 + c] = acc[c];
        }
        if (lane == 0) {
            zsum[warp] = z;
            s_exmax[warp] = mr;
        }
        __syncthreads();
        if (tid < D) {
            float mm = s_exmax[0];
#pragma unroll
            for (int w = 1; w < NW; ++w) mm = fmaxf(mm, s_exmax[w]);
            float sacc = 0.f, zz = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = fast_exp2(s_exmax[w] - mm);   // a warp without rows: exp2(-inf) = 0
                sacc = fmaf(red[w * D + tid], f, sacc);
                zz = fmaf(zsum[w], f, zz);
            }
            o[tid] = __float2bfloat16(sacc / zz);
        }
        if (idx_row)
            for (int i = tid; i < p.top_k; i += kTkNT) idx_row[i] = i < n ? sel[i] : -1;
        return;
    }
    // Top-K: the selection scores are the exact scaled scores, the largest key's is the maximum
    const float m_log2 = tk_unkey(s_maxkey) * kLog2e;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    float z = 0.f;
    const __nv_bfloat16 *vb = p.v + ((long long)b * p.L_cap * p.H_kv + kvh) * D + sub * 8;
    const long long vstride = (long long)p.H_kv * D;
    constexpr int U = 2;
    for (int t0 = 0; warp + NW * RPI * t0 < n; t0 += U) {
        float sc[U];
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = warp + NW * (RPI * (t0 + u) + part);
            sc[u] = -INFINITY;
            raw[u] = make_uint4(0u, 0u, 0u, 0u);
            if (i < n) {
                const int j = sel[i];
                sc[u] = ld_dep_f(srow + j);
                raw[u] = ld_dep_u4(reinterpret_cast<const uint4 *>(vb + (long long)j * vstride));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float wgt = fast_exp2(sc[u] * kLog2e - m_log2);
            z += wgt;
            const uint32_t w4[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[c]));
                acc[2 * c] = fmaf(wgt, f.x, acc[2 * c]);
                acc[2 * c + 1] = fmaf(wgt, f.y, acc[2 * c + 1]);
            }
        }
    }
#pragma unroll
    for (int o2 = LPR; o2 < 32; o2 <<= 1) {
        z += __shfl_xor_sync(0xffffffffu, z, o2);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], o2);
    }
    float *red = reinterpret_cast<float *>(hist);   // [NW][D]; the histogram is no longer read
    if (part == 0) {
#pragma unroll
        for (int c = 0; c < 8; ++c) red[warp * D + sub * 8 + c] = acc[c];
    }
    if (lane == 0) zsum[warp] = z;
    __syncthreads();
    if (tid < D) {
        float s = 0.f, zz = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            s += red[w * D + tid];
            zz += zsum[w];
        }
        o[tid] = __float2bfloat16(s / zz);
    }
    if (idx_row)
        for (int i = tid; i < p.top_k; i += kTkNT) idx_row[i] = i < n ? sel[i] : -1;
}

// ------------------------------------------------------------------- host side
static inline int tk_row_stride(int L_cap) { return (L_cap + 3) & ~3; }

size_t topk_workspace_bytes(int B, int H_q, int L_cap) {
    return (size_t)B * H_q * tk_row_stride(L_cap) * sizeof(float);
}

// Selection + attention kernel: candidates are the top_k plus room for the
// threshold bin's other members.
template <int D>
static magicdec_status launch_select_attn(TopkSelParams tp, int mode, cudaStream_t st) {
    const int smem_cap = magicdec_host::max_smem_optin();
    tp.cand_cap = tp.top_k + 4096;
    const size_t k4 = (size_t)((tp.top_k + 3) & ~3) * 4;
    const size_t smem2 = (size_t)kTkBins * 4 + (size_t)tp.cand_cap * 8 + k4;
    if (smem2 + 2048 > (size_t)smem_cap) return MAGICDEC_ERR_UNSUPPORTED;
    auto k2 = mode == kSelExact  ? topk_select_attn_kernel<D, kSelExact>
              : mode == kSelOnly ? topk_select_attn_kernel<D, kSelOnly>
                                 : topk_select_attn_kernel<D, kSelScores>;
    if (cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    return magicdec_host::launch_pdl(k2, dim3(tp.H_q, tp.B), dim3(kTkNT), smem2, st, tp);
}

template <int D>
static magicdec_status launch_topk_impl(const TopkScoreParams &sp, const TopkSelParams &tp, const CUtensorMap &tmk,
                                        bool heads, cudaStream_t st) {
    // heads: topk_scores_heads_kernel (32 KB stages of all eight heads); else
    // the per-pair kernel (16 KB stages of one head).  Two CTAs per SM either way.
    const int stage_bytes = heads ? kTkHdStage : (D / 64) * kTkHalfBytes;
    const int smem_cap = magicdec_host::max_smem_optin();
    const size_t fixed = 1024 + 2 * kTkMaxStages * sizeof(uint64_t) + (size_t)(sp.B + 1) * sizeof(int);
    const size_t per_cta = (size_t)smem_cap / 2 - 1024;
    if (per_cta <= fixed + 2 * (size_t)stage_bytes) return MAGICDEC_ERR_UNSUPPORTED;
    // Stages: as many as fit, up to 128 KB of K in flight per SM (two CTAs), unless
    // MAGICDEC_TOPK_STAGES asks otherwise.  At B=128, L=32000 the score pass with
    // more in flight was slower on the same GPU: whole Top-K draft 1.833 ms with
    // three 32 KB all-heads stages per CTA against 1.784-1.792 ms with two, and
    // 1.853-1.857 ms with six 16 KB per-pair stages against 1.829 ms with four.
    int stages = (int)((per_cta - fixed) / stage_bytes);
    const char *want_s = getenv("MAGICDEC_TOPK_STAGES");
    const int want = want_s && *want_s ? atoi(want_s) : 0;
    const int cap = want >= 2 ? want : (int)(kTkInflightBytes / (2 * (size_t)stage_bytes));
    if (cap >= 2 && cap < stages) stages = cap;
    if (stages > kTkMaxStages) stages = kTkMaxStages;
    TopkScoreParams s1 = sp;
    s1.stages = stages;
    const size_t smem1 = fixed + (size_t)stages * stage_bytes;
    magicdec_status s;
    if (heads) {
        auto k1 = topk_scores_heads_kernel;
        if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) != cudaSuccess)
            return MAGICDEC_ERR_CUDA;
        s = magicdec_host::launch_pdl(k1, dim3(magicdec_host::sm_count() * 2), dim3((kTkHdHeads + 1) * 32), smem1, st,
                                      tmk, s1);
    } else {
        auto k1 = topk_scores_kernel<D>;
        if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) != cudaSuccess)
            return MAGICDEC_ERR_CUDA;
        s = magicdec_host::launch_pdl(k1, dim3(magicdec_host::sm_count() * 2), dim3((kTkConsumers + 1) * 32), smem1, st,
                                      tmk, s1);
    }
    if (s != MAGICDEC_OK) return s;

    return launch_select_attn<D>(tp, kSelScores, st);
}

magicdec_status launch_topk_draft_attn(int B, int H_q, int H_kv, int D, int L_cap, const void *q, const void *k,
                                       const void *v, const int32_t *len, int top_k, void *out, int32_t *idx,
                                       void *ws, cudaStream_t st) {
    const int G = H_q / H_kv;
    if (G > kTkMaxGroup || top_k > kTkMaxTopK) return MAGICDEC_ERR_UNSUPPORTED;
    const int L_sc = tk_row_stride(L_cap);
    TopkScoreParams sp{};
    sp.q = static_cast<const __nv_bfloat16 *>(q);
    sp.score = static_cast<float *>(ws);
    sp.len = len;
    sp.err = magicdec_host::device_error_word();
    sp.B = B;
    sp.H_q = H_q;
    sp.H_kv = H_kv;
    sp.G = G;
    sp.L_cap = L_cap;
    sp.L_sc = L_sc;
    sp.scale = 1.0f / sqrtf((float)D);
    TopkSelParams tp{};
    tp.score = sp.score;
    tp.q = static_cast<const __nv_bfloat16 *>(q);
    tp.k = static_cast<const __nv_bfloat16 *>(k);
    tp.v = static_cast<const __nv_bfloat16 *>(v);
    tp.scale = sp.scale;
    tp.len = len;
    tp.out = static_cast<__nv_bfloat16 *>(out);
    tp.idx = idx;
    tp.B = B;
    tp.H_q = H_q;
    tp.H_kv = H_kv;
    tp.G = G;
    tp.L_cap = L_cap;
    tp.L_sc = L_sc;
    tp.top_k = top_k;

    CUtensorMap tmk;
    const uint64_t e = 2;
    const char *env = getenv("MAGICDEC_TOPK_HEADS");
    const bool heads = D == 128 && H_kv == kTkHdHeads && !(env && env[0] == '0');
    if (heads) {
        // K as (d, L_cap, H_kv, B), the position stride before the head stride;
        // one box = 64 channels x 16 positions x 8 heads
        const uint64_t dims[4] = {(uint64_t)D, (uint64_t)L_cap, (uint64_t)H_kv, (uint64_t)B};
        const uint64_t strides[3] = {(uint64_t)H_kv * D * e, (uint64_t)D * e, (uint64_t)L_cap * H_kv * D * e};
        const uint32_t box[4] = {64, (uint32_t)kTkHdPos, (uint32_t)kTkHdHeads, 1};
        if (!magicdec_host::encode_tmap_bf16_4d(&tmk, k, dims, strides, box)) return MAGICDEC_ERR_CUDA;
    } else {
        // K as (d, H_kv, L_cap, B); one box = 64 channels x 1 head x 64 positions
        const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H_kv, (uint64_t)L_cap, (uint64_t)B};
        const uint64_t strides[3] = {(uint64_t)D * e, (uint64_t)H_kv * D * e, (uint64_t)L_cap * H_kv * D * e};
        const uint32_t box[4] = {64, 1, kTkTileN, 1};
        if (!magicdec_host::encode_tmap_bf16_4d(&tmk, k, dims, strides, box)) return MAGICDEC_ERR_CUDA;
    }
    if (D == 128) return launch_topk_impl<128>(sp, tp, tmk, heads, st);
    if (D == 64) return launch_topk_impl<64>(sp, tp, tmk, false, st);
    return MAGICDEC_ERR_UNSUPPORTED;
}

// Selection by precomputed scores [B, H_q, L_cap rounded to 4] and attention
// over the kept rows; exact = true recomputes the kept rows' scores from K.
magicdec_status launch_topk_select_attn(int B, int H_q, int H_kv, int D, int L_cap, const void *q, const void *k,
                                        const void *v, const int32_t *len, int top_k, bool exact, const float *score,
                                        void *out, int32_t *idx, cudaStream_t st) {
    const int G = H_q / H_kv;
    if (top_k > kTkMaxTopK) return MAGICDEC_ERR_UNSUPPORTED;
    TopkSelParams tp{};
    tp.score = score;
    tp.q = static_cast<const __nv_bfloat16 *>(q);
    tp.k = static_cast<const __nv_bfloat16 *>(k);
    tp.v = static_cast<const __nv_bfloat16 *>(v);
    tp.len = len;
    tp.out = static_cast<__nv_bfloat16 *>(out);
    tp.idx = idx;
    tp.B = B;
    tp.H_q = H_q;
    tp.H_kv = H_kv;
    tp.G = G;
    tp.L_cap = L_cap;
    tp.L_sc = tk_row_stride(L_cap);
    tp.top_k = top_k;
    tp.scale = 1.0f / sqrtf((float)D);
    if (D == 128) return launch_select_attn<128>(tp, exact ? kSelExact : kSelScores, st);
    if (D == 64) return launch_select_attn<64>(tp, exact ? kSelExact : kSelScores, st);
    return MAGICDEC_ERR_UNSUPPORTED;
}

// SnapKV selection over pooled prefix scores [B, H_kv, L_cap rounded to 4]:
// rows (sequence, KV head); keeps budget - window prefix positions, appends
// the window; idx [B, H_kv, budget], n_sel [B].  With `budgets`, sequence b
// keeps budgets[b] (clamped to [window, budget]) and `budget` is the stride.
magicdec_status launch_snapkv_pick(int B, int H_kv, int L_cap, const float *pooled, const int32_t *len, int window,
                                   int budget, const int32_t *budgets, int32_t *idx, int32_t *n_sel, cudaStream_t st) {
    TopkSelParams tp{};
    tp.budgets = budgets;
    tp.score = pooled;
    tp.len = len;
    tp.idx = idx;
    tp.n_sel = n_sel;
    tp.B = B;
    tp.H_q = H_kv;        // one row per (sequence, KV head)
    tp.H_kv = H_kv;
    tp.G = 1;
    tp.L_cap = L_cap;
    tp.L_sc = tk_row_stride(L_cap);
    tp.top_k = budget;
    tp.len_sub = window;
    return launch_select_attn<128>(tp, kSelOnly, st);
}

}  // namespace magicdec
