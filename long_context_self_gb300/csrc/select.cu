// select.cu -- draft-KV selection and gather for MagicDec self-speculation,
// sm_103a.
//
//  * StreamingLLM selection (paper section 4.4 / section 5.1): attention sinks
//    plus a recent window; pure index arithmetic.
//  * SnapKV selection (paper section 4.4 / section 5.2), once after prefill:
//      pass 1  per (sequence, KV head, 1024-position chunk): the M = w*G
//              observation-window query rows stream the chunk's K rows and
//              keep an online (max, sum) of their causal softmax; partials
//              go to the workspace;
//      pass 2  per chunk of the prefix [0, L-w): merge the partials into each
//              row's log-sum-exp, recompute the logits, and sum the softmax
//              probabilities over the M rows per position -> score;
//      top-k   one CTA per (sequence, KV head): max-pool (kernel k, clipped),
//              an 8-bit-digit MSB-first radix select of the k-th largest
//              pooled score, then an order-preserving block compaction that
//              keeps everything above the threshold and the smallest
//              positions among ties; the window is appended.
//    Passes 1-2 stream K once each (bulk copies into padded shared rows, an
//    mbarrier ring) and contract on bf16 mma.sync with fp32 accumulation.
//  * Gather ("pre-gather a sparse KV cache", section 4.4): 16-byte vector
//    row copies into the head-major compact draft cache.
#include <algorithm>

#include "common.cuh"

namespace magicdec {

__device__ __forceinline__ int clamp_len_s(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }

// ------------------------------------------------------------ StreamingLLM
__global__ void streaming_select_kernel(const int32_t *seq_len, int B, int H_kv, int n_sink, int n_recent,
                                        int32_t *idx, int32_t *n_sel) {
    pdl_trigger();
    pdl_wait();
    const int width = n_sink + n_recent;
    const long long total = (long long)B * H_kv * width;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(t % width);
        const int b = (int)(t / ((long long)H_kv * width));
        const int len = max(__ldg(seq_len + b), 0);
        const int sinks = min(n_sink, len);
        const int rec0 = max(n_sink, len - n_recent);
        const int n = sinks + max(0, len - rec0);
        int v = -1;
        if (j < sinks) v = j;
        else if (j < n) v = rec0 + (j - sinks);
        idx[t] = v;
        if (j == 0 && (t / width) % H_kv == 0) n_sel[b] = n;
    }
}

// ------------------------------------------------------------------ gather
// Unit u = one 16-byte chunk of one destination row of K or V:
//   ch = u % CPR, kv = (u / CPR) % 2, row = u / (2*CPR) = (b*H_kv + h)*n_idx + i.
// Each thread moves UNROLL units per iteration so that many loads are in flight.
template <int CPR>
__global__ void __launch_bounds__(256) gather_kv_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                       const int32_t *__restrict__ idx, int H_kv, int L_cap,
                                                       int n_idx, int cap, unsigned total,
                                                       uint4 *__restrict__ kc, uint4 *__restrict__ vc) {
    constexpr int UNROLL = 4;
    pdl_trigger();
    pdl_wait();
    const unsigned stride = gridDim.x * blockDim.x;
    for (unsigned base = blockIdx.x * blockDim.x + threadIdx.x; base < total; base += stride * UNROLL) {
        uint4 val[UNROLL];
        uint4 *dst[UNROLL];
#pragma unroll
        for (int j = 0; j < UNROLL; ++j) {
            const unsigned u = base + j * stride;
            dst[j] = nullptr;
            val[j] = make_uint4(0, 0, 0, 0);
            if (u < total) {
                const unsigned ch = u % CPR;
                const unsigned kv = (u / CPR) & 1u;
                const unsigned row = u / (2 * CPR);
                const unsigned bh = row / (unsigned)n_idx;
                const unsigned i = row - bh * (unsigned)n_idx;
                const unsigned h = bh % (unsigned)H_kv, b = bh / (unsigned)H_kv;
                const int pos = __ldg(idx + row);
                if (pos >= 0 && pos < L_cap) {
                    const uint4 *src = (kv ? v : k) + (((size_t)b * L_cap + pos) * H_kv + h) * CPR + ch;
                    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(val[j].x), "=r"(val[j].y), "=r"(val[j].z), "=r"(val[j].w)
                                 : "l"(src));
                }
                dst[j] = (kv ? vc : kc) + ((size_t)bh * cap + i) * CPR + ch;
            }
        }
#pragma unroll
        for (int j = 0; j < UNROLL; ++j)
            if (dst[j]) *dst[j] = val[j];
    }
}

// ---------------------------------------------------------- SnapKV scoring
constexpr int kSnapTile = 64;
constexpr int kSnapChunk = 1024;                      // positions per CTA
constexpr int kSnapStages = 4;
constexpr int kSnapMaxMT = 12;                        // up to 192 window rows per KV head

struct SnapParams {
    const __nv_bfloat16 *q;     // [B, w, H_q, D]
    const int32_t *len;
    float *part;                // [B, H_kv, n_chunks, MP, 2]  (max, sum) per row and chunk
    float *score;               // [B, H_kv, L_cap]
    int *err;
    int B, H_q, H_kv, G, w, L_cap, M, MT, n_chunks;
    float scale_log2;
};

constexpr int kSnapHalf = kSnapTile * 128;           // one 64-row x 64-channel swizzled box

template <int D, int PASS>
__global__ void __launch_bounds__((kSnapMaxMT + 1) * 32, 1)
    snapkv_pass_kernel(const __grid_constant__ CUtensorMap tmk, const SnapParams p) {
    constexpr int HALVES = D / 64;
    constexpr int TILE_BYTES = HALVES * kSnapHalf;
    constexpr int KS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int MT = p.MT, MP = MT * 16;
    uint8_t *stage_base = smem;
    float *colsum = reinterpret_cast<float *>(smem + kSnapStages * TILE_BYTES);     // [MT][64]
    float *lse = colsum + kSnapMaxMT * 64;                                           // [MP]
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(lse + kSnapMaxMT * 16);
    uint64_t *empty_bar = full_bar + kSnapStages;

    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    pdl_trigger();
    pdl_wait();
    const int L = clamp_len_s(__ldg(p.len + b), p.L_cap);
    if (L < p.w) return;
    const int end = PASS == 1 ? L : L - p.w;
    const int pos_begin = chunk * kSnapChunk;
    const int pos_end = min(pos_begin + kSnapChunk, end);
    if (pos_begin >= pos_end) return;
    const int ntiles = (pos_end - pos_begin + kSnapTile - 1) / kSnapTile;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float sl = p.scale_log2;
    const float NEG_INF = -INFINITY;

    if (tid == 0) {
        for (int s = 0; s < kSnapStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], MT);
        }
        mbar_fence_init();
    }
    if (PASS == 2) {
        // Merge pass-1 partials into each row's log2-sum-exp2 (scaled units).
        const int nvalid = (L + kSnapChunk - 1) / kSnapChunk;
        const float *pb = p.part + ((long long)b * p.H_kv + h) * p.n_chunks * MP * 2;
        for (int r = tid; r < MP; r += blockDim.x) {
            if (r >= p.M) { lse[r] = INFINITY; continue; }
            float mx = NEG_INF;
            for (int cc = 0; cc < nvalid; ++cc) mx = fmaxf(mx, pb[((long long)cc * MP + r) * 2]);
            float sm = 0.f;
            for (int cc = 0; cc < nvalid; ++cc)
                sm += pb[((long long)cc * MP + r) * 2 + 1] * fast_exp2((pb[((long long)cc * MP + r) * 2] - mx) * sl);
            lse[r] = mx * sl + __log2f(sm);
        }
    }
    __syncthreads();

    if (warp == MT) {
        // producer (one thread): TMA boxes of 64 positions x 64 channels of K
        if (lane != 0) return;
        prefetch_tensormap(&tmk);
        const uint64_t pol = policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        for (int ti = 0; ti < ntiles; ++ti) {
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) break;
            mbar_arrive_expect_tx(&full_bar[stage], TILE_BYTES);
            uint8_t *sk = stage_base + stage * TILE_BYTES;
            const int pos0 = pos_begin + ti * kSnapTile;
#pragma unroll
            for (int hf = 0; hf < HALVES; ++hf)
                tma_load_4d(sk + hf * kSnapHalf, &tmk, hf * 64, h, pos0, b, &full_bar[stage], pol);
            ++issued;
            if (++stage == kSnapStages) { stage = 0; phase ^= 1u; }
        }
        int st = stage;
        uint32_t ph = phase;
        for (int kk = 0; kk < min(issued, kSnapStages); ++kk) {
            if (st == 0) { st = kSnapStages - 1; ph ^= 1u; } else { --st; }
            mbar_wait(&full_bar[st], ph, p.err);
        }
        return;
    }

    // consumers: warp mt owns window rows mt*16 .. mt*16+15 over all 64 columns
    const int mt = warp, g = lane >> 2, t4 = lane & 3;
    const int r0 = mt * 16 + g, r1 = r0 + 8;
    const int lim0 = r0 < p.M ? L - p.w + r0 / p.G : L - 1;
    const int lim1 = r1 < p.M ? L - p.w + r1 / p.G : L - 1;
    const long long qstride = (long long)p.H_q * D;
    const __nv_bfloat16 *qb = p.q + (long long)b * p.w * qstride + (long long)h * p.G * D;
    uint32_t qa[KS][4];
    {
        const __nv_bfloat16 *q0 = r0 < p.M ? qb + (r0 / p.G) * qstride + (r0 % p.G) * D : nullptr;
        const __nv_bfloat16 *q1 = r1 < p.M ? qb + (r1 / p.G) * qstride + (r1 % p.G) * D : nullptr;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int c0 = ks * 16 + 2 * t4;
            qa[ks][0] = q0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + c0)) : 0u;
            qa[ks][1] = q1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + c0)) : 0u;
            qa[ks][2] = q0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + c0 + 8)) : 0u;
            qa[ks][3] = q1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + c0 + 8)) : 0u;
        }
    }
    const float lse0 = PASS == 2 ? lse[r0] : 0.f, lse1 = PASS == 2 ? lse[r1] : 0.f;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    float *score_row = p.score + ((long long)b * p.H_kv + h) * p.L_cap;

    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int ti = 0; ti < ntiles; ++ti) {
        if (ok) ok = mbar_wait(&full_bar[stage], phase, p.err);
        const uint32_t kbase = smem_u32(stage_base + stage * TILE_BYTES);
        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        if (ok) {
            const int mat = lane >> 3, rr = lane & 7;
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                const int row = nb * 16 + (mat >> 1) * 8 + rr;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int ch = ks * 2 + (mat & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + (ch >> 3) * kSnapHalf + swz128(row, ch & 7), b0, b1, b2, b3);
                    mma_bf16(sc[2 * nb], qa[ks], b0, b1);
                    mma_bf16(sc[2 * nb + 1], qa[ks], b2, b3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
        if (++stage == kSnapStages) { stage = 0; phase ^= 1u; }

        const int tile_pos = pos_begin + ti * kSnapTile;
        if (PASS == 1) {
            if (tile_pos + kSnapTile - 1 > L - p.w) {
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int pos = tile_pos + n * 8 + 2 * t4 + e;
                        if (pos > lim0 || pos >= pos_end) sc[n][e] = NEG_INF;
                        if (pos > lim1 || pos >= pos_end) sc[n][2 + e] = NEG_INF;
                    }
            } else if (tile_pos + kSnapTile > pos_end) {
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int pos = tile_pos + n * 8 + 2 * t4 + e;
                        if (pos >= pos_end) { sc[n][e] = NEG_INF; sc[n][2 + e] = NEG_INF; }
                    }
            }
            float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
                mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float mu0 = mn0 == NEG_INF ? 0.f : mn0, mu1 = mn1 == NEG_INF ? 0.f : mn1;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                s0 += fast_exp2((sc[n][0] - mu0) * sl) + fast_exp2((sc[n][1] - mu0) * sl);
                s1 += fast_exp2((sc[n][2] - mu1) * sl) + fast_exp2((sc[n][3] - mu1) * sl);
            }
            l0 = l0 * fast_exp2((m0 - mu0) * sl) + s0;
            l1 = l1 * fast_exp2((m1 - mu1) * sl) + s1;
            m0 = mn0;
            m1 = mn1;
        } else {
            // column sums of softmax probabilities over this warp's 16 rows
            float cs[8][2];
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float v = fast_exp2(fmaf(sc[n][e], sl, -lse0)) + fast_exp2(fmaf(sc[n][2 + e], sl, -lse1));
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    cs[n][e] = v;
                }
            if (g == 0) {
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    colsum[mt * 64 + n * 8 + 2 * t4] = cs[n][0];
                    colsum[mt * 64 + n * 8 + 2 * t4 + 1] = cs[n][1];
                }
            }
            named_bar_sync(1, MT * 32);
            for (int col = tid; col < kSnapTile; col += MT * 32) {
                float acc = 0.f;
                for (int w2 = 0; w2 < MT; ++w2) acc += colsum[w2 * 64 + col];
                const int pos = tile_pos + col;
                if (pos < pos_end) score_row[pos] = acc;
            }
            named_bar_sync(1, MT * 32);
        }
    }
    if (PASS == 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if (t4 == 0) {
            float *pb = p.part + (((long long)b * p.H_kv + h) * p.n_chunks + chunk) * MP * 2;
            pb[r0 * 2] = m0;
            pb[r0 * 2 + 1] = l0;
            pb[r1 * 2] = m1;
            pb[r1 * 2 + 1] = l1;
        }
    }
}

// ----------------------------------------------------------- pool + top-k
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix count of `flag` over 1024 threads; returns the
// thread's offset and writes the block total to *total.  Uses scratch[33].
__device__ __forceinline__ int block_excl_count(bool flag, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) scratch[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int x = lane < nw ? scratch[lane] : 0;
        const int own = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane < nw) scratch[lane] = x - own;
        if (lane == 31) scratch[32] = x;
    }
    __syncthreads();
    const int off = scratch[warp] + in_warp;
    *total = scratch[32];
    __syncthreads();
    return off;
}

__global__ void __launch_bounds__(1024) snapkv_topk_kernel(const float *__restrict__ score, uint32_t *keys,
                                                          const int32_t *__restrict__ seq_len, int H_kv,
                                                          int L_cap, int w, int pool, int budget, int32_t *idx,
                                                          int32_t *n_sel) {
    __shared__ int hist[256];
    __shared__ int scratch[40];
    __shared__ int sel_digit, sel_remaining;
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    const int L = clamp_len_s(__ldg(seq_len + b), L_cap);
    int32_t *out = idx + ((long long)b * H_kv + h) * budget;
    if (L <= budget) {
        for (int j = tid; j < budget; j += blockDim.x) out[j] = j < L ? j : -1;
        if (h == 0 && tid == 0) n_sel[b] = L;
        return;
    }
    const int m = L - w, k_top = budget - w, half = pool / 2;
    if (k_top == 0) {
        for (int r = tid; r < w; r += blockDim.x) out[r] = m + r;
        if (h == 0 && tid == 0) n_sel[b] = budget;
        return;
    }
    const float *sc = score + ((long long)b * H_kv + h) * L_cap;
    uint32_t *ky = keys + ((long long)b * H_kv + h) * L_cap;
    for (int j = tid; j < m; j += blockDim.x) {
        float mx = -INFINITY;
        const int lo = max(0, j - half), hi = min(m - 1, j + half);
        for (int t = lo; t <= hi; ++t) mx = fmaxf(mx, sc[t]);
        ky[j] = order_key(mx);
    }
    __syncthreads();

    uint32_t prefix = 0, pmask = 0;
    int remaining = k_top;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < m; j += blockDim.x) {
            const uint32_t kk = ky[j];
            if ((kk & pmask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l covers digits 255-8l down to 248-8l
            int cnt[8], gsum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { cnt[j] = hist[255 - (tid * 8 + j)]; gsum += cnt[j]; }
            int x = gsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (tid >= o) x += y;
            }
            int above = x - gsum;
            if (above < remaining && remaining <= x) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (above < remaining && remaining <= above + cnt[j]) {
                        sel_digit = 255 - (tid * 8 + j);
                        sel_remaining = remaining - above;
                    }
                    above += cnt[j];
                }
            }
        }
        __syncthreads();
        prefix |= (uint32_t)sel_digit << shift;
        pmask |= 255u << shift;
        remaining = sel_remaining;
        __syncthreads();
    }
    const uint32_t tau = prefix;
    const int need_eq = remaining;

    int sel_count = 0, eq_seen = 0;
    for (int base = 0; base < m; base += blockDim.x) {
        const int j = base + tid;
        const bool valid = j < m;
        const uint32_t kk = valid ? ky[j] : 0u;
        const bool gt = valid && kk > tau, eq = valid && kk == tau;
        int eq_total, take_total;
        const int eq_rank = eq_seen + block_excl_count(eq, scratch, &eq_total);
        const bool take = gt || (eq && eq_rank < need_eq);
        const int pos = sel_count + block_excl_count(take, scratch, &take_total);
        if (take && pos < k_top) out[pos] = j;
        sel_count += take_total;
        eq_seen += eq_total;
    }
    for (int r = tid; r < w; r += blockDim.x) out[k_top + r] = m + r;
    if (h == 0 && tid == 0) n_sel[b] = budget;
}

// ------------------------------------------------------------------- host side
magicdec_status launch_streaming_select(const int32_t *seq_len, int B, int H_kv, int n_sink, int n_recent,
                                        int32_t *idx, int32_t *n_sel, cudaStream_t st) {
    const long long total = (long long)B * H_kv * (n_sink + n_recent);
    const int threads = 256;
    const int blocks = (int)std::min<long long>((total + threads - 1) / threads, 65535);
    return magicdec_host::launch_pdl(streaming_select_kernel, dim3(blocks), dim3(threads), 0, st, seq_len, B, H_kv,
                                     n_sink, n_recent, idx, n_sel);
}

magicdec_status launch_gather_kv(int B, int H_kv, int D, int L_cap, const void *k, const void *v,
                                 const int32_t *idx, int n_idx, int cap, void *kc, void *vc, cudaStream_t st) {
    if (n_idx == 0 || B == 0) return MAGICDEC_OK;
    const long long total = (long long)B * H_kv * n_idx * 2 * (D / 8);
    if (total >= (1ll << 32)) return MAGICDEC_ERR_UNSUPPORTED;
    const int threads = 256;
    const long long want = (total + threads * 4 - 1) / (threads * 4);
    const int blocks = (int)std::max<long long>(1, std::min<long long>(want, (long long)magicdec_host::sm_count() * 8));
    const uint4 *k4 = static_cast<const uint4 *>(k), *v4 = static_cast<const uint4 *>(v);
    uint4 *kc4 = static_cast<uint4 *>(kc), *vc4 = static_cast<uint4 *>(vc);
    if (D == 128)
        return magicdec_host::launch_pdl(gather_kv_kernel<16>, dim3(blocks), dim3(threads), 0, st, k4, v4, idx, H_kv,
                                         L_cap, n_idx, cap, (unsigned)total, kc4, vc4);
    return magicdec_host::launch_pdl(gather_kv_kernel<8>, dim3(blocks), dim3(threads), 0, st, k4, v4, idx, H_kv,
                                     L_cap, n_idx, cap, (unsigned)total, kc4, vc4);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t snapkv_workspace_bytes(int B, int H_q, int H_kv, int D, int L_cap, int w) {
    (void)D;
    const int G = H_q / H_kv;
    const int M = w * G;
    const int MP = ((M + 15) / 16) * 16;
    const int n_chunks = (L_cap + kSnapChunk - 1) / kSnapChunk;
    const size_t part = align256((size_t)B * H_kv * n_chunks * MP * 2 * 4);
    const size_t score = align256((size_t)B * H_kv * L_cap * 4);
    const size_t keys = align256((size_t)B * H_kv * L_cap * 4);
    return part + score + keys;
}

template <int D, int PASS>
static magicdec_status launch_snap_pass(const CUtensorMap &tmk, const SnapParams &prm, cudaStream_t st) {
    const size_t smem = 1024 + (size_t)kSnapStages * (D / 64) * kSnapHalf + kSnapMaxMT * 64 * 4 +
                        kSnapMaxMT * 16 * 4 + 2 * kSnapStages * 8;
    auto kern = snapkv_pass_kernel<D, PASS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    return magicdec_host::launch_pdl(kern, dim3(prm.n_chunks, prm.H_kv, prm.B), dim3((prm.MT + 1) * 32), smem, st,
                                     tmk, prm);
}

magicdec_status launch_snapkv_select(int B, int H_q, int H_kv, int D, int L_cap, const void *q_win, const void *k,
                                     const int32_t *seq_len, int w, int pool, int budget, int32_t *idx,
                                     int32_t *n_sel, void *ws, cudaStream_t st) {
    SnapParams prm{};
    prm.q = static_cast<const __nv_bfloat16 *>(q_win);
    prm.len = seq_len;
    prm.B = B;
    prm.H_q = H_q;
    prm.H_kv = H_kv;
    prm.G = H_q / H_kv;
    prm.w = w;
    prm.L_cap = L_cap;
    prm.M = w * prm.G;
    prm.MT = (prm.M + 15) / 16;
    if (prm.MT > kSnapMaxMT) return MAGICDEC_ERR_UNSUPPORTED;
    prm.n_chunks = (L_cap + kSnapChunk - 1) / kSnapChunk;
    prm.scale_log2 = kLog2e / sqrtf((float)D);
    prm.err = magicdec_host::device_error_word();
    const int MP = prm.MT * 16;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    prm.part = reinterpret_cast<float *>(wsb);
    wsb += align256((size_t)B * H_kv * prm.n_chunks * MP * 2 * 4);
    prm.score = reinterpret_cast<float *>(wsb);
    wsb += align256((size_t)B * H_kv * L_cap * 4);
    uint32_t *keys = reinterpret_cast<uint32_t *>(wsb);

    // K as a 4-D view (d, H_kv, L_cap, B); boxes of 64 channels x 64 positions.
    CUtensorMap tmk;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H_kv, (uint64_t)L_cap, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)H_kv * D * 2, (uint64_t)L_cap * H_kv * D * 2};
    const uint32_t box[4] = {64, 1, (uint32_t)kSnapTile, 1};
    if (!magicdec_host::encode_tmap_bf16_4d(&tmk, k, dims, strides, box)) return MAGICDEC_ERR_CUDA;

    magicdec_status s;
    if (D == 128) {
        if ((s = launch_snap_pass<128, 1>(tmk, prm, st)) != MAGICDEC_OK) return s;
        if ((s = launch_snap_pass<128, 2>(tmk, prm, st)) != MAGICDEC_OK) return s;
    } else if (D == 64) {
        if ((s = launch_snap_pass<64, 1>(tmk, prm, st)) != MAGICDEC_OK) return s;
        if ((s = launch_snap_pass<64, 2>(tmk, prm, st)) != MAGICDEC_OK) return s;
    } else {
        return MAGICDEC_ERR_UNSUPPORTED;
    }
    return magicdec_host::launch_pdl(snapkv_topk_kernel, dim3(H_kv, B), dim3(1024), 0, st,
                                     static_cast<const float *>(prm.score), keys, seq_len, H_kv, L_cap, w, pool,
                                     budget, idx, n_sel);
}

}  // namespace magicdec
