// PQCache-style dynamic KV selection.
//
// MagicDec (arXiv 2408.11049) section 4.4 with Figure 5: a dynamic selection
// that searches the KV cache per query through product-quantised keys; its
// search cost grows with the batch.  Keys of each (sequence, KV head) are
// split into M = d/8 sub-vectors of 8 channels; subspace m has C <= 256 fp32
// centroids (codebook [B, H_kv, M, C, 8]); a key's code is the index of the
// nearest centroid per subspace (codes [B, H_kv, L_cap, M] uint8).
//   pq_encode_kernel  nearest centroid (argmin of |c|^2 - 2 k.c in fp32;
//                     ties to the smaller index), the codebook of one
//                     (sequence, head) in shared memory, two keys per thread.
//   pq_update_kernel  one Lloyd update: centroid = mean of its keys.  The keys
//                     are bf16, so the sums are exact and order-independent
//                     as 2^-32 fixed point in shared-memory int64 atomics
//                     (every bf16 value of magnitude >= 2^-25 is a whole
//                     number of units; sums stay below 2^63 for |k| < 2^14
//                     over up to 2^17 positions); the
//                     mean is a correctly rounded fp64 division, rounded to
//                     fp32.  A centroid without keys keeps its value.
//   pq_scores_kernel  per draft step: persistent over 1024-position tiles of
//                     (sequence, KV head); each (sequence, head) builds the
//                     lookup table LUT[m][c][g] = scale * q_g,m . c_m,c for
//                     its G query heads once, then a position's approximate
//                     score for head g is sum_m LUT[m][code_m][g].  With G = 4
//                     the table is laid out so that the lookups of a warp
//                     meet no shared-memory bank conflicts whatever the codes.
// Selection and exact attention over the kept positions run in the Top-K
// select kernel (topk.cu) in its exact-score mode.
#include "common.cuh"

namespace magicdec {

constexpr int kPqDs = 8;              // channels per subspace
constexpr int kPqEncThreads = 256;
constexpr int kPqEncChunk = 2048;     // positions per encode CTA
constexpr int kPqUpdThreads = 512;
constexpr int kPqScThreads = 256;
constexpr int kPqScPer = 4;           // positions per thread in a score tile
constexpr int kPqScTile = kPqScThreads * kPqScPer;

struct PqScoreParams {
    const __nv_bfloat16 *q;    // [B, 1, H_q, D]
    const float *codebook;     // [B, H_kv, M, C, 8]
    const uint8_t *codes;      // [B, H_kv, L_cap, M]
    const int32_t *len;
    float *score;              // [B, H_q, L_sc]
    int *err;
    int B, H_q, H_kv, G, L_cap, L_sc, C;
    float scale;
};

__device__ __forceinline__ int pq_clamp(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }

__device__ __forceinline__ void bf16x8_to_float(const uint4 u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// ------------------------------------------------------------------ encode
template <int D>
__global__ void __launch_bounds__(kPqEncThreads) pq_encode_kernel(const __nv_bfloat16 *k,
                                                                 const float *codebook,
                                                                 uint8_t *__restrict__ codes, int H_kv, int L_cap,
                                                                 int C) {
    constexpr int M = D / kPqDs;
    extern __shared__ __align__(16) float pq_smem[];
    float *cb = pq_smem;                         // [M][C][8]
    float *nrm = cb + (size_t)M * C * kPqDs;     // [M][C]
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    const float4 *src = reinterpret_cast<const float4 *>(codebook + ((size_t)b * H_kv + h) * M * C * kPqDs);
    for (int i = tid; i < M * C * kPqDs / 4; i += kPqEncThreads) reinterpret_cast<float4 *>(cb)[i] = ld_dep_f4(src + i);
    __syncthreads();
    for (int i = tid; i < M * C; i += kPqEncThreads) {
        const float *c = cb + (size_t)i * kPqDs;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < kPqDs; ++e) s = fmaf(c[e], c[e], s);
        nrm[i] = s;
    }
    __syncthreads();
    const int j0 = chunk * kPqEncChunk, j1 = min(L_cap, j0 + kPqEncChunk);
    // KPT positions j + r * kPqEncThreads together: each centroid read feeds KPT keys
    constexpr int KPT = 4;
    for (int base = j0; base < j1; base += KPT * kPqEncThreads) {
        const uint4 *kr[KPT];
        bool valid[KPT];
#pragma unroll
        for (int r = 0; r < KPT; ++r) {
            const int j = base + r * kPqEncThreads + tid;
            valid[r] = j < j1;
            kr[r] = reinterpret_cast<const uint4 *>(k + (((size_t)b * L_cap + (valid[r] ? j : j0)) * H_kv + h) * D);
        }
        uint32_t packed[KPT][M / 4];
#pragma unroll
        for (int r = 0; r < KPT; ++r)
#pragma unroll
            for (int wi = 0; wi < M / 4; ++wi) packed[r][wi] = 0u;
#pragma unroll 1
        for (int m = 0; m < M; ++m) {
            float x[KPT][8];
#pragma unroll
            for (int r = 0; r < KPT; ++r) bf16x8_to_float(ld_dep_u4(kr[r] + m), x[r]);
            float best[KPT];
            int arg[KPT];
#pragma unroll
            for (int r = 0; r < KPT; ++r) { best[r] = INFINITY; arg[r] = 0; }
            const float *cm = cb + (size_t)m * C * kPqDs;
            const float *nm = nrm + (size_t)m * C;
            for (int c = 0; c < C; ++c) {
                const float4 c0 = *reinterpret_cast<const float4 *>(cm + c * kPqDs);
                const float4 c1 = *reinterpret_cast<const float4 *>(cm + c * kPqDs + 4);
                const float n = nm[c];
#pragma unroll
                for (int r = 0; r < KPT; ++r) {
                    float dd = x[r][0] * c0.x;
                    dd = fmaf(x[r][1], c0.y, dd);
                    dd = fmaf(x[r][2], c0.z, dd);
                    dd = fmaf(x[r][3], c0.w, dd);
                    dd = fmaf(x[r][4], c1.x, dd);
                    dd = fmaf(x[r][5], c1.y, dd);
                    dd = fmaf(x[r][6], c1.z, dd);
                    dd = fmaf(x[r][7], c1.w, dd);
                    const float e = fmaf(-2.f, dd, n);
                    if (e < best[r]) { best[r] = e; arg[r] = c; }   // strict: the smaller index keeps a tie
                }
            }
#pragma unroll
            for (int r = 0; r < KPT; ++r) {
                // byte m of the key's code word (M/4 words of 4 codes)
#pragma unroll
                for (int wi = 0; wi < M / 4; ++wi)
                    if (wi == (m >> 2)) {
                        const uint32_t sh = 8u * (uint32_t)(m & 3);
                        packed[r][wi] = (packed[r][wi] & ~(255u << sh)) | ((uint32_t)arg[r] << sh);
                    }
            }
        }
#pragma unroll
        for (int r = 0; r < KPT; ++r) {
            if (!valid[r]) continue;
            uint32_t *dst = reinterpret_cast<uint32_t *>(
                codes + (((size_t)b * H_kv + h) * L_cap + base + r * kPqEncThreads + tid) * M);
#pragma unroll
            for (int wi = 0; wi < M / 4; ++wi) dst[wi] = packed[r][wi];
        }
    }
}

// ------------------------------------------------------------------ update
template <int D>
__global__ void __launch_bounds__(kPqUpdThreads) pq_update_kernel(const __nv_bfloat16 *k,
                                                                 const int32_t *len_p,
                                                                 const uint8_t *codes,
                                                                 float *__restrict__ codebook, int H_kv, int L_cap,
                                                                 int C) {
    constexpr int M = D / kPqDs;
    constexpr int MH = M / 2;                     // subspaces per CTA (blockIdx.x picks the half)
    extern __shared__ __align__(16) unsigned long long pq_acc[];
    // [MH][8][C]: the code is the fastest index, so lanes with different codes
    // fall in different banks.  2^-32 fixed point (two's complement).
    unsigned long long *sum = pq_acc;
    int *cnt = reinterpret_cast<int *>(sum + (size_t)MH * C * kPqDs);   // [MH][C]
    const int half = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int m0 = half * MH;
    pdl_trigger();
    pdl_wait();
    for (int i = tid; i < MH * C * kPqDs; i += kPqUpdThreads) sum[i] = 0ull;
    for (int i = tid; i < MH * C; i += kPqUpdThreads) cnt[i] = 0;
    __syncthreads();
    const int len = pq_clamp(ld_dep(len_p + b), L_cap);
    for (int j = tid; j < len; j += kPqUpdThreads) {
        const uint8_t *cr = codes + (((size_t)b * H_kv + h) * L_cap + j) * M + m0;
        const uint4 *kr = reinterpret_cast<const uint4 *>(k + (((size_t)b * L_cap + j) * H_kv + h) * D) + m0;
#pragma unroll 1
        for (int mm = 0; mm < MH; ++mm) {
            const int c = ld_dep_u8(cr + mm);
            if (c >= C) continue;
            float x[8];
            bf16x8_to_float(ld_dep_u4(kr + mm), x);
            atomicAdd(cnt + mm * C + c, 1);
            unsigned long long *s = sum + (size_t)mm * kPqDs * C + c;
#pragma unroll
            for (int e = 0; e < kPqDs; ++e)
                atomicAdd(s + (size_t)e * C, (unsigned long long)__float2ll_rn(x[e] * 4294967296.0f));
        }
    }
    __syncthreads();
    float *cbo = codebook + (((size_t)b * H_kv + h) * M + m0) * C * kPqDs;
    for (int t = tid; t < MH * C * kPqDs; t += kPqUpdThreads) {
        const int mc = t / kPqDs, e = t - mc * kPqDs;       // output order [MH][C][8]
        const int mm = mc / C, c = mc - mm * C;
        const int n = cnt[mc];
        if (n == 0) continue;
        const double total = (double)(long long)sum[((size_t)mm * kPqDs + e) * C + c] * (1.0 / 4294967296.0);
        cbo[t] = (float)__ddiv_rn(total, (double)n);
    }
}

// ------------------------------------------------------------------ scores
__device__ __forceinline__ int pq_locate(long long t, const int *prefix, int B, int H_kv, int &h, int &ti) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)H_kv * prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int nt = prefix[lo + 1] - prefix[lo];
    const long long local = t - (long long)H_kv * prefix[lo];
    h = (int)(local / nt);
    ti = (int)(local - (long long)h * nt);
    return lo;
}

// a0 += b0, a1 += b1 as one packed fp32x2 add (two independent round-to-nearest
// single-precision adds, the same results as two scalar adds)
__device__ __forceinline__ void pq_add2(float &a0, float &a1, float b0, float b1) {
    unsigned long long a, b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}

template <int D>
__global__ void __launch_bounds__(kPqScThreads) pq_scores_kernel(const PqScoreParams p) {
    constexpr int M = D / kPqDs;
    extern __shared__ __align__(16) float pq_sm[];
    const int G = p.G, C = p.C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *lut = pq_sm;                                   // [C][M][4] when G == 4, else [M][C][G]
    float *qs = lut + (size_t)M * C * G;                  // [G][D]
    int *prefix = reinterpret_cast<int *>(qs + (size_t)G * D);   // [B + 1]
    pdl_trigger();
    pdl_wait();
    for (int b = tid; b < p.B; b += kPqScThreads)
        prefix[b] = (pq_clamp(checked(ld_dep(p.len + b), 0, p.L_cap, p.err), p.L_cap) + kPqScTile - 1) / kPqScTile;
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
    const long long t0 = T * blockIdx.x / gridDim.x, t1 = T * (blockIdx.x + 1) / gridDim.x;
    int cur_b = -1, cur_h = -1;
    // Location (sequence, KV head, tile) of a flat tile: a binary search at the
    // start of the range and when a step leaves a sequence, else one step on.
    struct Loc { int b, h, ti, nt, len; };
    auto locate = [&](long long tt) {
        Loc l;
        l.b = pq_locate(tt, prefix, p.B, p.H_kv, l.h, l.ti);
        l.nt = prefix[l.b + 1] - prefix[l.b];
        l.len = pq_clamp(ld_dep(p.len + l.b), p.L_cap);
        return l;
    };
    auto advance = [&](const Loc &l, long long tt_next) {
        Loc n = l;
        if (l.ti + 1 < l.nt) {
            n.ti = l.ti + 1;
        } else if (l.h + 1 < p.H_kv) {
            n.h = l.h + 1;
            n.ti = 0;
        } else {
            n = locate(tt_next);
        }
        return n;
    };
    // codes of tile t are loaded during tile t-1 (software pipeline)
    auto load_codes = [&](const Loc &lc, uint4 (&dst)[kPqScPer]) {
        const int bb = lc.b, hh = lc.h, tti = lc.ti, ll = lc.len;
        const uint8_t *cbase = p.codes + ((size_t)bb * p.H_kv + hh) * p.L_cap * M;
#pragma unroll
        for (int i = 0; i < kPqScPer; ++i) {
            const int j = tti * kPqScTile + i * kPqScThreads + tid;
            dst[i] = make_uint4(0u, 0u, 0u, 0u);
            if (j < ll) {
                if (M == 16) {
                    dst[i] = ld_dep_u4(reinterpret_cast<const uint4 *>(cbase + (size_t)j * M));
                } else {
                    const uint2 u = ld_dep_u2(reinterpret_cast<const uint2 *>(cbase + (size_t)j * M));
                    dst[i].x = u.x;
                    dst[i].y = u.y;
                }
            }
        }
    };
    uint4 raw[kPqScPer], nxt[kPqScPer];
#pragma unroll
    for (int i = 0; i < kPqScPer; ++i) raw[i] = nxt[i] = make_uint4(0u, 0u, 0u, 0u);
    Loc cur{};
    if (t0 < t1) {
        cur = locate(t0);
        load_codes(cur, raw);
    }
    for (long long t = t0; t < t1; ++t) {
        const int b = cur.b, h = cur.h, ti = cur.ti, len = cur.len;
        Loc nxl = cur;
        if (t + 1 < t1) {
            nxl = advance(cur, t + 1);
            load_codes(nxl, nxt);
        }
        if (b != cur_b || h != cur_h) {            // lookup table of this (sequence, KV head) for its G query heads
            __syncthreads();
            for (int i = tid; i < G * D; i += kPqScThreads) {
                const int g = i / D, e = i - g * D;
                qs[i] = __bfloat162float(p.q[((size_t)b * p.H_q + (size_t)h * G + g) * D + e]);
            }
            __syncthreads();
            const float *cbh = p.codebook + ((size_t)b * p.H_kv + h) * M * C * kPqDs;
            constexpr int BATCH = 4;
            for (int mc0 = tid; mc0 < M * C; mc0 += BATCH * kPqScThreads) {
                float4 c0[BATCH], c1[BATCH];
#pragma unroll
                for (int u = 0; u < BATCH; ++u) {
                    const int mc = mc0 + u * kPqScThreads;
                    if (mc < M * C) {
                        c0[u] = ld_dep_f4(reinterpret_cast<const float4 *>(cbh + (size_t)mc * kPqDs));
                        c1[u] = ld_dep_f4(reinterpret_cast<const float4 *>(cbh + (size_t)mc * kPqDs + 4));
                    }
                }
#pragma unroll
                for (int u = 0; u < BATCH; ++u) {
                    const int mc = mc0 + u * kPqScThreads;
                    if (mc >= M * C) continue;
                    const int m = mc / C, cc = mc - m * C;
                    // G == 4: entry (c, m) at [c][m][4], so the 16-byte entries of
                    // the M subspaces of one centroid index fill consecutive bank
                    // quads (see the lookups below); otherwise [m][c][G]
                    const size_t at = G == 4 ? ((size_t)cc * M + m) * 4 : (size_t)mc * G;
                    if (G == 4) {
                        // the warp shares m: the query slices are broadcast reads, and
                        // the entry is one 16-byte store
                        float sd[4];
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            const float4 qa = *reinterpret_cast<const float4 *>(qs + g * D + m * kPqDs);
                            const float4 qb4 = *reinterpret_cast<const float4 *>(qs + g * D + m * kPqDs + 4);
                            float sdot = qa.x * c0[u].x;
                            sdot = fmaf(qa.y, c0[u].y, sdot);
                            sdot = fmaf(qa.z, c0[u].z, sdot);
                            sdot = fmaf(qa.w, c0[u].w, sdot);
                            sdot = fmaf(qb4.x, c1[u].x, sdot);
                            sdot = fmaf(qb4.y, c1[u].y, sdot);
                            sdot = fmaf(qb4.z, c1[u].z, sdot);
                            sdot = fmaf(qb4.w, c1[u].w, sdot);
                            sd[g] = sdot * p.scale;
                        }
                        *reinterpret_cast<float4 *>(lut + at) = make_float4(sd[0], sd[1], sd[2], sd[3]);
                        continue;
                    }
                    for (int g = 0; g < G; ++g) {
                        const float *qq = qs + g * D + m * kPqDs;
                        float sdot = qq[0] * c0[u].x;
                        sdot = fmaf(qq[1], c0[u].y, sdot);
                        sdot = fmaf(qq[2], c0[u].z, sdot);
                        sdot = fmaf(qq[3], c0[u].w, sdot);
                        sdot = fmaf(qq[4], c1[u].x, sdot);
                        sdot = fmaf(qq[5], c1[u].y, sdot);
                        sdot = fmaf(qq[6], c1[u].z, sdot);
                        sdot = fmaf(qq[7], c1[u].w, sdot);
                        lut[at + g] = sdot * p.scale;
                    }
                }
            }
            __syncthreads();
            cur_b = b;
            cur_h = h;
        }
        float *srow0 = p.score + ((size_t)b * p.H_q + (size_t)h * G) * p.L_sc;
#pragma unroll
        for (int i = 0; i < kPqScPer; ++i) {
            const int j = ti * kPqScTile + i * kPqScThreads + tid;
            if (j >= len) continue;
            const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
            float *srow = srow0 + j;
            if (G == 4) {
                // A 16-byte lookup is served a quarter-warp (8 lanes) at a time,
                // one wavefront per bank quad touched.  Entry (c, m) lies in bank
                // quad m % 8 whatever c is, and lane l takes the subspaces in the
                // order m = (r + l) mod M (r = 0 .. M-1, l = the position's lane),
                // so the 8 lanes of a quarter-warp always touch 8 different quads:
                // 4 wavefronts per warp-wide lookup instead of about 11 for
                // arbitrary codes.  The codes are rotated once so that step r
                // reads byte r of the rotated vector.
                const int rot = lane & (M - 1);
                uint32_t x0 = w[0], x1 = w[1], x2 = w[2], x3 = w[3];
                uint32_t v[4];
                if (M == 16) {
                    const int sw = rot >> 2;
                    if (sw & 1) { const uint32_t tt = x0; x0 = x1; x1 = x2; x2 = x3; x3 = tt; }
                    if (sw & 2) { const uint32_t t0 = x0, t1 = x1; x0 = x2; x1 = x3; x2 = t0; x3 = t1; }
                    const int sh = (rot & 3) * 8;
                    v[0] = __funnelshift_r(x0, x1, sh);
                    v[1] = __funnelshift_r(x1, x2, sh);
                    v[2] = __funnelshift_r(x2, x3, sh);
                    v[3] = __funnelshift_r(x3, x0, sh);
                } else {                                     // M == 8: codes in w[0], w[1]
                    if (rot >> 2) { const uint32_t tt = x0; x0 = x1; x1 = tt; }
                    const int sh = (rot & 3) * 8;
                    v[0] = __funnelshift_r(x0, x1, sh);
                    v[1] = __funnelshift_r(x1, x0, sh);
                    v[2] = v[3] = 0u;
                }
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M == 16 && C == 256) {
                    // every byte is a valid code: the entry's byte offset c*256 + m*16
                    // is one byte permute (code r into bits 8-15) plus the subspace's
                    // offset, which depends only on r and the lane
                    const char *lutb = reinterpret_cast<const char *>(lut);
                    const uint32_t rot16 = (uint32_t)rot << 4;
#pragma unroll
                    for (int r = 0; r < M; ++r) {
                        const uint32_t off = __byte_perm(v[r >> 2], 0u, 0x4404u | ((uint32_t)(r & 3) << 4)) +
                                             (((uint32_t)r * 16u + rot16) & 0xF0u);
                        const float4 l = *reinterpret_cast<const float4 *>(lutb + off);
                        pq_add2(acc.x, acc.y, l.x, l.y);
                        pq_add2(acc.z, acc.w, l.z, l.w);
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < M; ++r) {
                        const int m = (r + rot) & (M - 1);
                        int c = (int)((v[r >> 2] >> (8 * (r & 3))) & 255u);
                        c = c < C ? c : 0;
                        const float4 l = *reinterpret_cast<const float4 *>(lut + ((size_t)c * M + m) * 4);
                        acc.x += l.x; acc.y += l.y; acc.z += l.z; acc.w += l.w;
                    }
                }
                srow[0] = acc.x;
                srow[(size_t)p.L_sc] = acc.y;
                srow[2 * (size_t)p.L_sc] = acc.z;
                srow[3 * (size_t)p.L_sc] = acc.w;
            } else {
                for (int g = 0; g < G; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        int c = (int)((w[m >> 2] >> (8 * (m & 3))) & 255u);
                        c = c < C ? c : 0;
                        acc += lut[((size_t)m * C + c) * G + g];
                    }
                    srow[(size_t)g * p.L_sc] = acc;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kPqScPer; ++i) raw[i] = nxt[i];
        cur = nxl;
    }
}

// ------------------------------------------------------------------- host side
// Nearest centroid on the tensor cores.  The dot products k_m . c of a
// subspace are a (keys x 8) x (8 x C) contraction; each fp32 centroid is split
// exactly into three bf16 pieces (hi = bf16(c), mid = bf16(c - hi),
// lo = c - hi - mid), stored times -2 (exact), every product of a bf16 key
// value with a piece is exact in fp32, and three m16n8k8 bf16 MMAs into an
// accumulator started at |c|^2 leave |c|^2 - 2 k.c to fp32 accuracy.  The
// argmin (ties: the smaller index) stays in fp32 on the ALU, which now bounds
// the kernel.  Shared memory: the pieces
// [3][M][CP][8] bf16 and the norms [M][CP] fp32 of one (sequence, KV head)
// codebook, CP = C rounded up to 32 (padding centroids have an infinite norm
// and are never chosen).
__device__ __forceinline__ void pq_mma_k8(float (&c)[4], const uint32_t (&a)[2], uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(b0));
}

constexpr int kPqTcThreads = 512;
constexpr int kPqTcKeys = 16;                      // keys per warp batch (one m16 tile)

template <int D>
__global__ void __launch_bounds__(kPqTcThreads, 1)
    pq_encode_tc_kernel(const __nv_bfloat16 *k, const float *codebook,
                        uint8_t *__restrict__ codes, int H_kv, int L_cap, int C, int CP) {
    constexpr int M = D / kPqDs;
    extern __shared__ __align__(128) uint8_t pq_tc_smem[];
    uint8_t *pieces = pq_tc_smem;                                          // [3][M][CP][8] bf16
    float *nrm = reinterpret_cast<float *>(pq_tc_smem + (size_t)3 * M * CP * 16);   // [M][CP]
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    pdl_wait();
    const float *cbh = codebook + ((size_t)b * H_kv + h) * M * C * kPqDs;
    for (int i = tid; i < M * CP; i += kPqTcThreads) {
        const int m = i / CP, c = i - m * CP;
        uint32_t w[3][4];
        float n = INFINITY;
        if (c < C) {
            const float4 u0 = ld_dep_f4(reinterpret_cast<const float4 *>(cbh + ((size_t)m * C + c) * kPqDs));
            const float4 u1 = ld_dep_f4(reinterpret_cast<const float4 *>(cbh + ((size_t)m * C + c) * kPqDs + 4));
            const float x[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            float s2 = 0.f;
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                float hi[2], mi[2], lo[2];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    hi[t] = __bfloat162float(__float2bfloat16_rn(x[e + t]));
                    mi[t] = __bfloat162float(__float2bfloat16_rn(x[e + t] - hi[t]));
                    lo[t] = x[e + t] - hi[t] - mi[t];
                }
                // pieces scaled by -2 (exact): with the accumulator started at
                // |c|^2 the MMAs leave |c|^2 - 2 k.c
                w[0][e / 2] = pack_bf16(-2.f * hi[0], -2.f * hi[1]);
                w[1][e / 2] = pack_bf16(-2.f * mi[0], -2.f * mi[1]);
                w[2][e / 2] = pack_bf16(-2.f * lo[0], -2.f * lo[1]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) s2 = fmaf(x[e], x[e], s2);
            n = s2;
        } else {
#pragma unroll
            for (int pc = 0; pc < 3; ++pc) w[pc][0] = w[pc][1] = w[pc][2] = w[pc][3] = 0u;
        }
#pragma unroll
        for (int pc = 0; pc < 3; ++pc)
            *reinterpret_cast<uint4 *>(pieces + (((size_t)pc * M + m) * CP + c) * 16) =
                make_uint4(w[pc][0], w[pc][1], w[pc][2], w[pc][3]);
        nrm[i] = n;
    }
    __syncthreads();

    const int g = lane >> 2, t4 = lane & 3;
    const int j0 = chunk * kPqEncChunk, j1 = min(L_cap, j0 + kPqEncChunk);
    const uint32_t pbase = smem_u32(pieces);
    const int lrow = (lane >> 3) * 8 + (lane & 7);         // centroid row this lane addresses in an x4 load
    constexpr int STRIDE = (kPqTcThreads / 32) * kPqTcKeys;
    // A fragments (16 keys x 8 channels per subspace): rows g and g+8, channels
    // 2*t4 and 2*t4+1 of each subspace; every subspace's words of a batch are
    // loaded together, and the next batch's while this one is searched
    auto load_a = [&](int base, uint32_t (&dst)[M][2]) {
        const int ja = min(base + g, j1 - 1), jb = min(base + g + 8, j1 - 1);
        const uint32_t *ka = reinterpret_cast<const uint32_t *>(k + (((size_t)b * L_cap + ja) * H_kv + h) * D);
        const uint32_t *kb = reinterpret_cast<const uint32_t *>(k + (((size_t)b * L_cap + jb) * H_kv + h) * D);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            dst[m][0] = ld_dep_u32(ka + m * 4 + t4);
            dst[m][1] = ld_dep_u32(kb + m * 4 + t4);
        }
    };
    uint32_t a_cur[M][2], a_nxt[M][2];
    if (j0 + warp * kPqTcKeys < j1) load_a(j0 + warp * kPqTcKeys, a_cur);
    for (int base = j0 + warp * kPqTcKeys; base < j1; base += STRIDE) {
        const int ja = base + g, jb = base + g + 8;
        if (base + STRIDE < j1) load_a(base + STRIDE, a_nxt);
        uint32_t pk_a[M / 4], pk_b[M / 4];
#pragma unroll
        for (int wi = 0; wi < M / 4; ++wi) pk_a[wi] = pk_b[wi] = 0u;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint32_t a[2] = {a_cur[m][0], a_cur[m][1]};
            // two argmin chains per key row (centroid tiles j = 0, 2 and j = 1, 3 of
            // each group of four), each in ascending centroid order
            float best_a[2] = {INFINITY, INFINITY}, best_b[2] = {INFINITY, INFINITY};
            int arg_a[2] = {0, 0}, arg_b[2] = {0, 0};
            const float *nm = nrm + (size_t)m * CP;
            for (int c4 = 0; c4 < CP; c4 += 32) {
                uint32_t bp[3][4];
#pragma unroll
                for (int pc = 0; pc < 3; ++pc)
                    ldsm_x4(pbase + (uint32_t)((((size_t)pc * M + m) * CP + c4 + lrow) * 16), bp[pc][0], bp[pc][1],
                            bp[pc][2], bp[pc][3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c0 = c4 + j * 8 + 2 * t4;
                    const float2 n = *reinterpret_cast<const float2 *>(nm + c0);
                    float e[4] = {n.x, n.y, n.x, n.y};      // rows g, g+8 x columns c0, c0+1
                    pq_mma_k8(e, a, bp[0][j]);
                    pq_mma_k8(e, a, bp[1][j]);
                    pq_mma_k8(e, a, bp[2][j]);
                    const int ch = j & 1;
                    if (e[0] < best_a[ch]) { best_a[ch] = e[0]; arg_a[ch] = c0; }   // strict: the smaller index keeps a tie
                    if (e[1] < best_a[ch]) { best_a[ch] = e[1]; arg_a[ch] = c0 + 1; }
                    if (e[2] < best_b[ch]) { best_b[ch] = e[2]; arg_b[ch] = c0; }
                    if (e[3] < best_b[ch]) { best_b[ch] = e[3]; arg_b[ch] = c0 + 1; }
                }
            }
            float bst_a = best_a[0], bst_b = best_b[0];
            int ar_a = arg_a[0], ar_b = arg_b[0];
            if (best_a[1] < bst_a || (best_a[1] == bst_a && arg_a[1] < ar_a)) { bst_a = best_a[1]; ar_a = arg_a[1]; }
            if (best_b[1] < bst_b || (best_b[1] == bst_b && arg_b[1] < ar_b)) { bst_b = best_b[1]; ar_b = arg_b[1]; }
            // the four lanes of a quad hold disjoint centroid columns
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                const float ob_a = __shfl_xor_sync(0xffffffffu, bst_a, o);
                const int oa_a = __shfl_xor_sync(0xffffffffu, ar_a, o);
                const float ob_b = __shfl_xor_sync(0xffffffffu, bst_b, o);
                const int oa_b = __shfl_xor_sync(0xffffffffu, ar_b, o);
                if (ob_a < bst_a || (ob_a == bst_a && oa_a < ar_a)) { bst_a = ob_a; ar_a = oa_a; }
                if (ob_b < bst_b || (ob_b == bst_b && oa_b < ar_b)) { bst_b = ob_b; ar_b = oa_b; }
            }
#pragma unroll
            for (int wi = 0; wi < M / 4; ++wi)
                if (wi == (m >> 2)) {
                    const uint32_t sh = 8u * (uint32_t)(m & 3);
                    pk_a[wi] |= (uint32_t)ar_a << sh;
                    pk_b[wi] |= (uint32_t)ar_b << sh;
                }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            a_cur[m][0] = a_nxt[m][0];
            a_cur[m][1] = a_nxt[m][1];
        }
        if (t4 == 0) {
            uint8_t *cbase = codes + ((size_t)b * H_kv + h) * L_cap * M;
            if (M == 16) {
                if (ja < j1) *reinterpret_cast<uint4 *>(cbase + (size_t)ja * M) = make_uint4(pk_a[0], pk_a[1], pk_a[2], pk_a[3 % (M / 4)]);
                if (jb < j1) *reinterpret_cast<uint4 *>(cbase + (size_t)jb * M) = make_uint4(pk_b[0], pk_b[1], pk_b[2], pk_b[3 % (M / 4)]);
            } else {
                if (ja < j1) *reinterpret_cast<uint2 *>(cbase + (size_t)ja * M) = make_uint2(pk_a[0], pk_a[1 % (M / 4)]);
                if (jb < j1) *reinterpret_cast<uint2 *>(cbase + (size_t)jb * M) = make_uint2(pk_b[0], pk_b[1 % (M / 4)]);
            }
        }
    }
}

magicdec_status launch_pq_encode(int B, int H_kv, int D, int L_cap, int C, const void *k, const float *codebook,
                                 uint8_t *codes, cudaStream_t st) {
    const int M = D / kPqDs;
    const char *env = getenv("MAGICDEC_PQ_TC");
    if (!(env && env[0] == '0')) {
        // tensor-core search (MAGICDEC_PQ_TC=0: the FMA kernel below)
        const int CP = (C + 31) & ~31;
        const size_t smem_tc = (size_t)3 * M * CP * 16 + (size_t)M * CP * 4;
        if (smem_tc <= (size_t)magicdec_host::max_smem_optin()) {
            const dim3 grid((L_cap + kPqEncChunk - 1) / kPqEncChunk, H_kv, B);
            auto kb = static_cast<const __nv_bfloat16 *>(k);
            auto kern = D == 128 ? pq_encode_tc_kernel<128> : pq_encode_tc_kernel<64>;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_tc) != cudaSuccess)
                return MAGICDEC_ERR_CUDA;
            return magicdec_host::launch_pdl(kern, grid, dim3(kPqTcThreads), smem_tc, st, kb, codebook, codes, H_kv,
                                             L_cap, C, CP);
        }
    }
    const size_t smem = (size_t)M * C * kPqDs * 4 + (size_t)M * C * 4;
    if (smem > (size_t)magicdec_host::max_smem_optin()) return MAGICDEC_ERR_UNSUPPORTED;
    const dim3 grid((L_cap + kPqEncChunk - 1) / kPqEncChunk, H_kv, B);
    auto kb = static_cast<const __nv_bfloat16 *>(k);
    if (D == 128) {
        if (cudaFuncSetAttribute(pq_encode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return MAGICDEC_ERR_CUDA;
        return magicdec_host::launch_pdl(pq_encode_kernel<128>, grid, dim3(kPqEncThreads), smem, st, kb, codebook,
                                         codes, H_kv, L_cap, C);
    }
    if (cudaFuncSetAttribute(pq_encode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    return magicdec_host::launch_pdl(pq_encode_kernel<64>, grid, dim3(kPqEncThreads), smem, st, kb, codebook, codes,
                                     H_kv, L_cap, C);
}

magicdec_status launch_pq_update(int B, int H_kv, int D, int L_cap, int C, const void *k, const int32_t *len,
                                 const uint8_t *codes, float *codebook, cudaStream_t st) {
    const int MH = D / kPqDs / 2;
    const size_t smem = (size_t)MH * C * kPqDs * 8 + (size_t)MH * C * 4;
    if (smem > (size_t)magicdec_host::max_smem_optin()) return MAGICDEC_ERR_UNSUPPORTED;
    const dim3 grid(2, H_kv, B);
    auto kb = static_cast<const __nv_bfloat16 *>(k);
    if (D == 128) {
        if (cudaFuncSetAttribute(pq_update_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return MAGICDEC_ERR_CUDA;
        return magicdec_host::launch_pdl(pq_update_kernel<128>, grid, dim3(kPqUpdThreads), smem, st, kb, len, codes,
                                         codebook, H_kv, L_cap, C);
    }
    if (cudaFuncSetAttribute(pq_update_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    return magicdec_host::launch_pdl(pq_update_kernel<64>, grid, dim3(kPqUpdThreads), smem, st, kb, len, codes,
                                     codebook, H_kv, L_cap, C);
}

magicdec_status launch_topk_select_attn(int B, int H_q, int H_kv, int D, int L_cap, const void *q, const void *k,
                                        const void *v, const int32_t *len, int top_k, bool exact, const float *score,
                                        void *out, int32_t *idx, cudaStream_t st);

magicdec_status launch_pq_draft_attn(int B, int H_q, int H_kv, int D, int L_cap, int C, const void *q, const void *k,
                                     const void *v, const int32_t *len, const float *codebook, const uint8_t *codes,
                                     int top_k, void *out, int32_t *idx, void *ws, cudaStream_t st) {
    const int M = D / kPqDs, G = H_q / H_kv;
    PqScoreParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.codebook = codebook;
    p.codes = codes;
    p.len = len;
    p.score = static_cast<float *>(ws);
    p.B = B;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.L_cap = L_cap;
    p.L_sc = (L_cap + 3) & ~3;
    p.C = C;
    p.scale = 1.0f / sqrtf((float)D);
    p.err = magicdec_host::device_error_word();
    const size_t smem = (size_t)M * C * G * 4 + (size_t)G * D * 4 + (size_t)(B + 1) * 4;
    if (smem > (size_t)magicdec_host::max_smem_optin()) return MAGICDEC_ERR_UNSUPPORTED;
    auto kern = D == 128 ? pq_scores_kernel<128> : pq_scores_kernel<64>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    // persistent grid: exactly the CTAs that can be resident at once
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPqScThreads, smem) != cudaSuccess ||
        per_sm < 1)
        return MAGICDEC_ERR_UNSUPPORTED;
    const int grid = magicdec_host::sm_count() * per_sm;
    magicdec_status s = magicdec_host::launch_pdl(kern, dim3(grid), dim3(kPqScThreads), smem, st, p);
    if (s != MAGICDEC_OK) return s;
    return launch_topk_select_attn(B, H_q, H_kv, D, L_cap, q, k, v, len, top_k, true, p.score, out, idx, st);
}

}  // namespace magicdec
