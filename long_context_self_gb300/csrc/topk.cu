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
//                            (12 + 12 + 8 bit digits), ascending compaction, then
//                            softmax over the kept scores and the weighted sum
//                            of the kept V rows.  The keys stay in shared memory
//                            when the row fits, else they are re-derived from
//                            the scores in global memory on every pass.
#include "common.cuh"

namespace magicdec {

constexpr int kTkTileN = 64;                     // positions per K tile
constexpr int kTkHalfBytes = kTkTileN * 128;     // 64 positions x 64 channels, bf16
constexpr int kTkConsumers = 4;                  // warps, 16 positions each
constexpr int kTkMaxStages = 8;
constexpr int kTkSelThreads = 1024;              // the block scans below assume exactly 32 warps
constexpr int kTkBins = 4096;
constexpr int kTkMaxTopK = 8192;
constexpr int kTkMaxGroup = 8;                   // query heads per KV head (the mma N extent)

struct TopkScoreParams {
    const __nv_bfloat16 *q;   // [B, 1, H_q, D]
    float *score;             // [B, H_q, L_sc]
    const int32_t *len;       // [B]
    int *err;
    int B, H_q, H_kv, G, L_cap, L_sc, stages;
    float scale;
};

struct TopkSelParams {
    const float *score;       // [B, H_q, L_sc]
    const __nv_bfloat16 *v;   // [B, L_cap, H_kv, D]
    const int32_t *len;       // [B]
    __nv_bfloat16 *out;       // [B, 1, H_q, D]
    int32_t *idx;             // [B, H_q, top_k] or null
    int B, H_q, H_kv, G, L_cap, L_sc, top_k;
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
        prefix[b] = (tk_clamp_len(__ldg(p.len + b), p.L_cap) + kTkTileN - 1) / kTkTileN;
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
                bq[ks][0] = valid ? __ldg(qrow + ks * 8 + (lane & 3)) : 0u;
                bq[ks][1] = valid ? __ldg(qrow + ks * 8 + 4 + (lane & 3)) : 0u;
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);

        const int len = tk_clamp_len(__ldg(p.len + cur.b), p.L_cap);
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

// Inclusive block-wide scan (32 warps) in thread order; *total = block sum.
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
        int y = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        wsum[lane] = y;
    }
    __syncthreads();
    const int excl = warp ? wsum[warp - 1] : 0;
    *total = wsum[31];
    __syncthreads();
    return x + excl;
}

// The digit (bin) holding the remaining-th largest candidate, scanning the
// 4096 bins from the top; returns it and the rank left inside that bin.
__device__ __forceinline__ void tk_find_digit(const int *hist, int remaining, int *wsum, int *s_digit, int *s_rem,
                                              int &digit, int &rem_out) {
    const int tid = threadIdx.x;
    int cnt[4], sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        cnt[j] = hist[kTkBins - 1 - 4 * tid - j];
        sum += cnt[j];
    }
    int total;
    const int incl = tk_block_scan(sum, wsum, &total);
    int above = incl - sum;
    if (above < remaining && remaining <= incl) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (above < remaining && remaining <= above + cnt[j]) {
                *s_digit = kTkBins - 1 - 4 * tid - j;
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

template <int D, bool SMEM_KEYS>
__global__ void __launch_bounds__(kTkSelThreads, 1) topk_select_attn_kernel(const TopkSelParams p) {
    constexpr int CPL = D / 32;                  // value channels per lane
    extern __shared__ __align__(16) uint8_t smem_raw[];
    int *hist = reinterpret_cast<int *>(smem_raw);                 // [4096]; later [32][D] partial outputs
    int *sel = hist + kTkBins;                                     // [top_k rounded to 4]
    uint32_t *ky = reinterpret_cast<uint32_t *>(sel + ((p.top_k + 3) & ~3));   // [L_sc] (SMEM_KEYS)
    __shared__ int wsum[32];
    __shared__ int s_digit, s_rem;
    __shared__ unsigned s_maxkey;
    __shared__ float zsum[32];

    const int hq = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();
    const int len = tk_clamp_len(__ldg(p.len + b), p.L_cap);
    const int kvh = hq / p.G;
    const long long row = (long long)b * p.H_q + hq;
    const float *srow = p.score + row * p.L_sc;
    __nv_bfloat16 *o = p.out + row * D;
    int32_t *idx_row = p.idx ? p.idx + row * p.top_k : nullptr;
    const int n = min(len, p.top_k);
    if (len == 0) {
        for (int c = tid; c < D; c += blockDim.x) o[c] = __float2bfloat16(0.f);
        if (idx_row)
            for (int i = tid; i < p.top_k; i += blockDim.x) idx_row[i] = -1;
        return;
    }
    const bool select = len > p.top_k;
    auto key_at = [&](int j) -> uint32_t {
        if (SMEM_KEYS) return ky[j];
        return tk_key(srow[j]);
    };

    // Keys, the first-digit histogram and the largest key.  The row starts on
    // a 16-byte boundary (L_sc % 4 == 0) and L_sc >= len rounded up to 4.
    for (int i = tid; i < kTkBins; i += blockDim.x) hist[i] = 0;
    if (tid == 0) s_maxkey = 0u;
    __syncthreads();
    uint32_t mk = 0u;
    const int n4 = (len + 3) >> 2;
    for (int i4 = tid; i4 < n4; i4 += blockDim.x) {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(srow) + i4);
        uint32_t k4[4] = {tk_key(f.x), tk_key(f.y), tk_key(f.z), tk_key(f.w)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (4 * i4 + e >= len) {
                k4[e] = 0u;
            } else {
                mk = max(mk, k4[e]);
                if (select) atomicAdd(&hist[k4[e] >> 20], 1);
            }
        }
        if (SMEM_KEYS) reinterpret_cast<uint4 *>(ky)[i4] = make_uint4(k4[0], k4[1], k4[2], k4[3]);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o2));
    if (lane == 0) atomicMax(&s_maxkey, mk);
    __syncthreads();

    if (select) {
        // radix select of the top_k-th key tau; need_eq = how many keys equal
        // to tau are kept (the ones at the smallest positions)
        int d1, d2, d3, rem;
        tk_find_digit(hist, p.top_k, wsum, &s_digit, &s_rem, d1, rem);
        for (int i = tid; i < kTkBins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < len; j += blockDim.x) {
            const uint32_t k = key_at(j);
            if ((int)(k >> 20) == d1) atomicAdd(&hist[(k >> 8) & 4095u], 1);
        }
        __syncthreads();
        tk_find_digit(hist, rem, wsum, &s_digit, &s_rem, d2, rem);
        for (int i = tid; i < kTkBins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const uint32_t pre = ((uint32_t)d1 << 12) | (uint32_t)d2;
        for (int j = tid; j < len; j += blockDim.x) {
            const uint32_t k = key_at(j);
            if ((k >> 8) == pre) atomicAdd(&hist[k & 255u], 1);
        }
        __syncthreads();
        tk_find_digit(hist, rem, wsum, &s_digit, &s_rem, d3, rem);
        const uint32_t tau = (pre << 8) | (uint32_t)d3;
        const int need_eq = rem;

        // ascending compaction: a kept position's slot is (#greater before it)
        // + min(#equal before it, need_eq)
        int gt_seen = 0, eq_seen = 0;
        for (int base = 0; base < len; base += 4 * kTkSelThreads) {
            const int j0 = base + 4 * tid;
            uint32_t kk[4];
            int ngt = 0, neq = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kk[e] = j0 + e < len ? key_at(j0 + e) : 0u;
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
    } else {
        for (int i = tid; i < len; i += blockDim.x) sel[i] = i;
    }
    __syncthreads();

    // softmax over the kept scores (the largest key is always kept) and the
    // weighted sum of their V rows; warp w takes kept entries w, w+32, ...
    const float m_log2 = tk_unkey(s_maxkey) * kLog2e;
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
    float z = 0.f;
    const __nv_bfloat16 *vb = p.v + ((long long)b * p.L_cap * p.H_kv + kvh) * D + lane * CPL;
    const long long vstride = (long long)p.H_kv * D;
    constexpr int U = 4;
    for (int i0 = warp; i0 < n; i0 += 32 * U) {
        float wgt[U];
        uint32_t raw[U][CPL / 2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * 32;
            wgt[u] = 0.f;
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c) raw[u][c] = 0u;
            if (i < n) {
                const int j = sel[i];
                wgt[u] = fast_exp2(tk_unkey(key_at(j)) * kLog2e - m_log2);
                const uint32_t *src = reinterpret_cast<const uint32_t *>(vb + (long long)j * vstride);
                if (CPL == 4) {
                    const uint2 t = __ldg(reinterpret_cast<const uint2 *>(src));
                    raw[u][0] = t.x;
                    raw[u][CPL / 2 - 1] = t.y;
                } else {
                    raw[u][0] = __ldg(src);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            z += wgt[u];
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw[u][c]));
                acc[2 * c] = fmaf(wgt[u], f.x, acc[2 * c]);
                acc[2 * c + 1] = fmaf(wgt[u], f.y, acc[2 * c + 1]);
            }
        }
    }
    float *red = reinterpret_cast<float *>(hist);   // [32][D]; the histogram is no longer read
#pragma unroll
    for (int c = 0; c < CPL; ++c) red[warp * D + lane * CPL + c] = acc[c];
    if (lane == 0) zsum[warp] = z;
    __syncthreads();
    if (tid < D) {
        float s = 0.f, zz = 0.f;
#pragma unroll 8
        for (int w = 0; w < 32; ++w) {
            s += red[w * D + tid];
            zz += zsum[w];
        }
        o[tid] = __float2bfloat16(s / zz);
    }
    if (idx_row)
        for (int i = tid; i < p.top_k; i += blockDim.x) idx_row[i] = i < n ? sel[i] : -1;
}

// ------------------------------------------------------------------- host side
static inline int tk_row_stride(int L_cap) { return (L_cap + 3) & ~3; }

size_t topk_workspace_bytes(int B, int H_q, int L_cap) {
    return (size_t)B * H_q * tk_row_stride(L_cap) * sizeof(float);
}

template <int D>
static magicdec_status launch_topk_impl(const TopkScoreParams &sp, const TopkSelParams &tp, const CUtensorMap &tmk,
                                        cudaStream_t st) {
    constexpr int STAGE_BYTES = (D / 64) * kTkHalfBytes;
    const int smem_cap = magicdec_host::max_smem_optin();
    const size_t fixed = 1024 + 2 * kTkMaxStages * sizeof(uint64_t) + (size_t)(sp.B + 1) * sizeof(int);
    const size_t per_cta = (size_t)smem_cap / 2 - 1024;          // two CTAs per SM
    if (per_cta <= fixed + 2 * STAGE_BYTES) return MAGICDEC_ERR_UNSUPPORTED;
    int stages = (int)((per_cta - fixed) / STAGE_BYTES);
    if (stages > kTkMaxStages) stages = kTkMaxStages;
    TopkScoreParams s1 = sp;
    s1.stages = stages;
    const size_t smem1 = fixed + (size_t)stages * STAGE_BYTES;
    auto k1 = topk_scores_kernel<D>;
    if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    magicdec_status s = magicdec_host::launch_pdl(k1, dim3(magicdec_host::sm_count() * 2),
                                                  dim3((kTkConsumers + 1) * 32), smem1, st, tmk, s1);
    if (s != MAGICDEC_OK) return s;

    const size_t sel_bytes = (size_t)kTkBins * 4 + (size_t)((tp.top_k + 3) & ~3) * 4;
    const size_t key_bytes = (size_t)tp.L_sc * 4;
    const size_t static_reserve = 2048;
    if (sel_bytes + key_bytes + static_reserve <= (size_t)smem_cap) {
        auto k2 = topk_select_attn_kernel<D, true>;
        const size_t smem2 = sel_bytes + key_bytes;
        if (cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2) != cudaSuccess)
            return MAGICDEC_ERR_CUDA;
        return magicdec_host::launch_pdl(k2, dim3(tp.H_q, tp.B), dim3(kTkSelThreads), smem2, st, tp);
    }
    auto k2 = topk_select_attn_kernel<D, false>;
    if (cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel_bytes) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    return magicdec_host::launch_pdl(k2, dim3(tp.H_q, tp.B), dim3(kTkSelThreads), sel_bytes, st, tp);
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
    tp.v = static_cast<const __nv_bfloat16 *>(v);
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

    // K as (d, H_kv, L_cap, B); one box = 64 channels x 1 head x 64 positions
    CUtensorMap tmk;
    const uint64_t e = 2;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H_kv, (uint64_t)L_cap, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)D * e, (uint64_t)H_kv * D * e, (uint64_t)L_cap * H_kv * D * e};
    const uint32_t box[4] = {64, 1, kTkTileN, 1};
    if (!magicdec_host::encode_tmap_bf16_4d(&tmk, k, dims, strides, box)) return MAGICDEC_ERR_CUDA;
    if (D == 128) return launch_topk_impl<128>(sp, tp, tmk, st);
    if (D == 64) return launch_topk_impl<64>(sp, tp, tmk, st);
    return MAGICDEC_ERR_UNSUPPORTED;
}

}  // namespace magicdec
