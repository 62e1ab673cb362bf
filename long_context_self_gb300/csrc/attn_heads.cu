// attn_heads.cu -- verification attention that streams all eight KV heads of
// a sequence together (d = 128, H_kv = 8, up to 24 query rows per KV head),
// sm_103a.  verify_heads_kernel serves up to 16 rows per KV head,
// verify_heads_t_kernel (below) 17 to 24.
//
// The operation is verification attention (paper section 3.1, T_V(B,S,gamma)):
// the gamma+1 speculated queries of every query head attend to the full KV
// cache [B, L_cap, H_kv, d], causal inside the speculated block.  The general
// kernel (attn.cu) streams one (sequence, KV head) pair at a time, fetching
// 256-byte rows that lie 2 KB apart in the cache; this one reads, per
// pipeline stage, 8 consecutive positions of all 8 heads of one sequence --
// 16 KB of K and 16 KB of V contiguous in HBM.  On GB300 that traversal
// streams 2 % faster (7.47 against 7.32 TB/s for the same bytes with no
// compute), and verification is most of a speculative step.
//
// Design:
//  * Persistent grid, one CTA per SM; the batch is a flat list of 8-position
//    tiles ordered (sequence, tile), split evenly across CTAs.  A sequence split
//    across CTAs leaves per-head partial (max, sum, unnormalised output)
//    triples; the last CTA to finish the sequence (an atomic counter per
//    sequence, no spin-wait) merges them with the log-sum-exp rule.
//  * One producer thread issues per stage four TMA boxes (K and V, two
//    64-channel halves) of 64 channels x 8 positions x 8 heads from a tensor
//    map whose position stride precedes its head stride, so each head's 8 rows
//    are consecutive 128-byte swizzled rows in shared memory (ldmatrix reads
//    conflict-free); plus, per sequence, the query rows of all heads.
//  * Eight consumer warps, warp h owning KV head h and its G*n_q <= 16 query
//    rows: S = Q_h K_h^T (16 x 8) by m16n8k16 over eight k-steps, an fp32
//    online softmax with exp2, then O += P V_h by m16n8k8 with P taken
//    straight from the S accumulator.  A warp owns whole rows, so a sequence
//    ends without any cross-warp combine.
#include "common.cuh"

namespace magicdec {

constexpr int kHdHeads = 8;                        // KV heads, one consumer warp each
constexpr int kHdPos = 8;                          // positions per stage
constexpr int kHdD = 128;
constexpr int kHdHalf = kHdPos * kHdHeads * 128;   // one 64-channel half of K (or V) per stage: 8 KB
constexpr int kHdStage = 4 * kHdHalf;              // K and V, two halves each: 32 KB
constexpr int kHdMaxStages = 8;
constexpr int kHdDefaultStages = 5;               // stage ring depth unless overridden
constexpr int kHdMaxContrib = 512;                 // CTAs at most (a merge lists one slot per CTA in shared memory)
constexpr int kHdRows = 16;                        // query rows per KV head (one m16 tile)

struct HeadsParams {
    const __nv_bfloat16 *q;     // [B, n_q, H_q, 128]
    const int32_t *len;         // [B]
    __nv_bfloat16 *out;         // [B, n_q, H_q, 128]
    float *part_o;              // [2C][8 heads][16 rows][128] partial outputs
    float *part_ml;             // [2C][8][16][2] (max, sum)
    int *counters;              // [B] merge arrivals, zero between calls
    int *err;
    int B, H_q, G, n_q, L_cap, M, stages;
    float scale_log2;           // log2(e) / sqrt(128)
};

__device__ __forceinline__ int hd_clamp(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }

// Sequence holding flat tile t (prefix[b] = tiles of sequences < b).
__device__ __forceinline__ int hd_seq_of(long long t, const int *prefix, int B) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ long long hd_cta_start(int c, long long T, int C) { return T * c / C; }
__device__ __forceinline__ int hd_cta_of(long long t, long long T, int C) {
    return (int)(((t + 1) * (long long)C - 1) / T);
}

// D(16x8 fp32) += A(16x8 bf16, row) * B(8x8 bf16, col)
__device__ __forceinline__ void mma_bf16_k8(float (&c)[4], const uint32_t (&a)[2], uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(b0));
}

__global__ void __launch_bounds__((kHdHeads + 1) * 32, 1)
    verify_heads_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ CUtensorMap tmq, const HeadsParams p) {
    constexpr int NCW = kHdHeads;
    constexpr int KS = kHdD / 16;              // k-steps of Q K^T
    constexpr int ND = kHdD / 8;               // 8-channel n-tiles of P V
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int stages = p.stages;
    const int QHALF = p.H_q * p.n_q * 128;     // one 64-channel half of the query box (a multiple of 1 KB)
    uint8_t *stage_base = smem;
    uint8_t *qslot = smem + (size_t)stages * kHdStage;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(qslot + 2 * QHALF);
    uint64_t *empty_bar = full_bar + kHdMaxStages;
    uint64_t *qfull = empty_bar + kHdMaxStages;
    uint64_t *qempty = qfull + 1;
    int *flag = reinterpret_cast<int *>(qempty + 1);
    int *contrib = flag + 4;                   // [gridDim.x + 1]
    int *prefix = contrib + gridDim.x + 1;     // [B+1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NCW);
        }
        mbar_init(qfull, 1);
        mbar_init(qempty, NCW);
        mbar_fence_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        prefetch_tensormap(&tmq);
    }
    pdl_wait();
    // 8-position tiles per sequence, loaded in parallel, then an exclusive scan by warp 0.
    for (int b = tid; b < p.B; b += blockDim.x)
        prefix[b] = (hd_clamp(checked(ld_dep(p.len + b), 0, p.L_cap, p.err), p.L_cap) + kHdPos - 1) / kHdPos;
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

    const long long T = prefix[p.B];
    const int C = gridDim.x, c = blockIdx.x;
    const long long t_begin = hd_cta_start(c, T, C), t_end = hd_cta_start(c + 1, T, C);
    const long long q_tok_stride = (long long)p.H_q * kHdD;   // between query tokens of one sequence

    if (warp == NCW) {
        // ------------------------------------------------------- producer (1 thread)
        if (lane != 0) return;
        const uint64_t pol = policy_evict_normal();
        const uint64_t pol_q = policy_evict_first();
        int stage = 0, seg_no = 0, issued = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long t = t_begin; t < t_end && ok; ++seg_no) {
            const int b = hd_seq_of(t, prefix, p.B);
            const int ti0 = (int)(t - prefix[b]);
            const int nseg = (int)min((long long)prefix[b + 1] - t, t_end - t);
            // the query rows of all heads; the slot is free once every consumer
            // warp has taken the previous sequence's rows into registers
            if (!mbar_wait(qempty, (uint32_t)(seg_no & 1) ^ 1u, p.err)) { ok = false; break; }
            mbar_arrive_expect_tx(qfull, 2 * QHALF);
            tma_load_4d(qslot, &tmq, 0, 0, 0, b, qfull, pol_q);
            tma_load_4d(qslot + QHALF, &tmq, 64, 0, 0, b, qfull, pol_q);
            for (int i = 0; i < nseg; ++i) {
                if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) { ok = false; break; }
                mbar_arrive_expect_tx(&full_bar[stage], kHdStage);
                uint8_t *sk = stage_base + (size_t)stage * kHdStage;
                uint8_t *sv = sk + 2 * kHdHalf;
                const int pos0 = (ti0 + i) * kHdPos;
                tma_load_4d(sk, &tmk, 0, pos0, 0, b, &full_bar[stage], pol);
                tma_load_4d(sk + kHdHalf, &tmk, 64, pos0, 0, b, &full_bar[stage], pol);
                tma_load_4d(sv, &tmv, 0, pos0, 0, b, &full_bar[stage], pol);
                tma_load_4d(sv + kHdHalf, &tmv, 64, pos0, 0, b, &full_bar[stage], pol);
                ++issued;
                if (++stage == stages) { stage = 0; phase ^= 1u; }
            }
            t += nseg;
        }
        // Drain: do not leave the CTA while copies issued here may still land.
        int st = stage;
        uint32_t ph = phase;
        for (int k = 0; k < min(issued, stages); ++k) {
            if (st == 0) { st = stages - 1; ph ^= 1u; } else { --st; }
            mbar_wait(&full_bar[st], ph, p.err);
        }
        if (seg_no > 0) mbar_wait(qfull, (uint32_t)((seg_no - 1) & 1), p.err);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int h = warp;                                // KV head of this warp
    const int g = lane >> 2, t4 = lane & 3;
    const float sl = p.scale_log2;
    const float NEG_INF = -INFINITY;

    // Sequences with nothing to attend produce zero rows.
    for (int b = c; b < p.B; b += C) {
        if (prefix[b + 1] != prefix[b]) continue;
        uint4 *o = reinterpret_cast<uint4 *>(p.out + (long long)b * p.n_q * q_tok_stride);
        const int n16 = p.n_q * p.H_q * kHdD / 8;
        for (int i = tid; i < n16; i += NCW * 32) o[i] = make_uint4(0, 0, 0, 0);
    }

    // Rows owned by this thread: r0 = g, r1 = g + 8.  Row r < M is query token
    // r / G of query head h*G + r % G; rows past M are zero.
    const int r0 = g, r1 = g + 8;
    const bool v0 = r0 < p.M, v1 = r1 < p.M;
    // query-slot row (within a 64-channel half) of A-row r: [token][query head]
    auto qrow = [&](int r) {
        r = r < p.M ? r : 0;
        return (r / p.G) * p.H_q + h * p.G + r % p.G;
    };

    int stage = 0, seg_no = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (long long t = t_begin; t < t_end; ++seg_no) {
        const int b = hd_seq_of(t, prefix, p.B);
        const int ti0 = (int)(t - prefix[b]);
        const int nseg = (int)min((long long)prefix[b + 1] - t, t_end - t);
        const int len = hd_clamp(ld_dep(p.len + b), p.L_cap);
        const int lim0 = v0 ? len - p.n_q + r0 / p.G : len - 1;   // last position row r may see
        const int lim1 = v1 ? len - p.n_q + r1 / p.G : len - 1;

        uint32_t qa[KS][4];
        {
            if (ok) ok = mbar_wait(qfull, (uint32_t)(seg_no & 1), p.err);
            const uint32_t qbase = smem_u32(qslot);
            const int mat = lane >> 3, rr = lane & 7;
            const int srow = qrow(rr + 8 * (mat & 1));
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int ch = ks * 2 + (mat >> 1);
                ldsm_x4(qbase + (ch >> 3) * QHALF + swz128(srow, ch & 7), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
                if (!v0) qa[ks][0] = qa[ks][2] = 0u;
                if (!v1) qa[ks][1] = qa[ks][3] = 0u;
            }
            fence_proxy_async_smem();   // reads done before TMA may refill the buffer
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty);
        }

        float o[ND][4];
#pragma unroll
        for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;

        for (int i = 0; i < nseg; ++i) {
            if (ok) ok = mbar_wait(&full_bar[stage], phase, p.err);
            if (ok) {
                uint8_t *kt = stage_base + (size_t)stage * kHdStage;
                uint8_t *vt = kt + 2 * kHdHalf;
                const int pos0 = (ti0 + i) * kHdPos;
                if (pos0 + kHdPos > len) {
                    // rows at or past the sequence end hold whatever the cache holds
                    // there: zero this head's V rows so P = 0 meets finite values
                    for (int idx = lane; idx < kHdPos * 16; idx += 32) {
                        const int pp = idx >> 4, ch = idx & 15;
                        if (pos0 + pp >= len)
                            *reinterpret_cast<uint4 *>(vt + (ch >> 3) * kHdHalf + swz128(h * kHdPos + pp, ch & 7)) =
                                make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
                const int mat = lane >> 3, pp = lane & 7;
                const int krow = h * kHdPos + pp;
                // S = Q_h K_h^T: 16 rows x 8 positions
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k2 = 0; k2 < KS / 2; ++k2) {
                    const int ch = k2 * 4 + mat;             // 16-byte channel chunk 0..15
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + (ch >> 3) * kHdHalf + swz128(krow, ch & 7), b0, b1, b2, b3);
                    mma_bf16(sc, qa[2 * k2], b0, b1);
                    mma_bf16(sc, qa[2 * k2 + 1], b2, b3);
                }
                if (pos0 + kHdPos - 1 > len - p.n_q) {
                    const int pb = pos0 + 2 * t4;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (pb + e > lim0) sc[e] = NEG_INF;
                        if (pb + e > lim1) sc[2 + e] = NEG_INF;
                    }
                }
                float mx0 = fmaxf(sc[0], sc[1]), mx1 = fmaxf(sc[2], sc[3]);
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float mu0 = mn0 == NEG_INF ? 0.f : mn0, mu1 = mn1 == NEG_INF ? 0.f : mn1;
                const float al0 = fast_exp2((m0 - mu0) * sl), al1 = fast_exp2((m1 - mu1) * sl);
                const float ms0 = mu0 * sl, ms1 = mu1 * sl;
                sc[0] = fast_exp2(fmaf(sc[0], sl, -ms0));
                sc[1] = fast_exp2(fmaf(sc[1], sl, -ms0));
                sc[2] = fast_exp2(fmaf(sc[2], sl, -ms1));
                sc[3] = fast_exp2(fmaf(sc[3], sl, -ms1));
                l0 = l0 * al0 + (sc[0] + sc[1]);
                l1 = l1 * al1 + (sc[2] + sc[3]);
                m0 = mn0;
                m1 = mn1;
#pragma unroll
                for (int n = 0; n < ND; ++n) {
                    o[n][0] *= al0; o[n][1] *= al0;
                    o[n][2] *= al1; o[n][3] *= al1;
                }
                // O += P V_h: P (16 x 8) is the S accumulator re-packed as the A operand
                const uint32_t pa[2] = {pack_bf16(sc[0], sc[1]), pack_bf16(sc[2], sc[3])};
#pragma unroll
                for (int n4 = 0; n4 < ND / 4; ++n4) {
                    const int ch = n4 * 4 + mat;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(vbase + (ch >> 3) * kHdHalf + swz128(krow, ch & 7), b0, b1, b2, b3);
                    mma_bf16_k8(o[4 * n4], pa, b0);
                    mma_bf16_k8(o[4 * n4 + 1], pa, b1);
                    mma_bf16_k8(o[4 * n4 + 2], pa, b2);
                    mma_bf16_k8(o[4 * n4 + 3], pa, b3);
                }
            }
            fence_proxy_async_smem();   // reads done before TMA may refill the buffer
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            if (++stage == stages) { stage = 0; phase ^= 1u; }
        }

        // ------------------------------------------------ end of this CTA's run of the sequence
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        const long long seq_t0 = prefix[b];
        const int ntiles = prefix[b + 1] - prefix[b];
        const int c_first = hd_cta_of(seq_t0, T, C), c_last = hd_cta_of(seq_t0 + ntiles - 1, T, C);
        // contributors: the CTAs whose ranges overlap the sequence (with fewer
        // tiles than CTAs some ranges are empty, so at most `ntiles` of them)
        const int n_contrib = min(c_last - c_first + 1, ntiles);
        __nv_bfloat16 *ob = p.out + (long long)b * p.n_q * q_tok_stride + (long long)h * p.G * kHdD;
        if (n_contrib == 1) {
            const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
            __nv_bfloat16 *o0 = ob + (r0 / p.G) * q_tok_stride + (r0 % p.G) * kHdD;
            __nv_bfloat16 *o1 = ob + (r1 / p.G) * q_tok_stride + (r1 % p.G) * kHdD;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                const int col = n * 8 + 2 * t4;
                if (v0) *reinterpret_cast<uint32_t *>(o0 + col) = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
                if (v1) *reinterpret_cast<uint32_t *>(o1 + col) = pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
            }
        } else {
            // Partial slots: CTA c keeps 2c (its first run, when its range starts
            // inside a sequence split across CTAs) and 2c+1 (its last run).
            const int slot = 2 * c + (t_begin >= seq_t0 ? 0 : 1);
            float *po = p.part_o + ((long long)slot * kHdHeads + h) * kHdRows * kHdD;
            float *pml = p.part_ml + ((long long)slot * kHdHeads + h) * kHdRows * 2;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                const int col = n * 8 + 2 * t4;
                *reinterpret_cast<float2 *>(po + r0 * kHdD + col) = make_float2(o[n][0], o[n][1]);
                *reinterpret_cast<float2 *>(po + r1 * kHdD + col) = make_float2(o[n][2], o[n][3]);
            }
            if (t4 == 0) {
                *reinterpret_cast<float2 *>(pml + r0 * 2) = make_float2(m0, l0);
                *reinterpret_cast<float2 *>(pml + r1 * 2) = make_float2(m1, l1);
            }
            named_bar_sync(1, NCW * 32);
            if (tid == 0) {
                // release: this CTA's partials (ordered by the barrier above);
                // acquire: for the last arriver, every other contributor's partials
                const int old = atomic_add_acq_rel_gpu(p.counters + b, 1);
                const int last = (old == n_contrib - 1);
                if (old >= n_contrib) raise_error(p.err, kErrState);
                if (last) p.counters[b] = 0;
                *flag = last;
            }
            named_bar_sync(1, NCW * 32);
            if (*flag) {
                // The last arriver lists the contributors' slots (CTAs ascending;
                // -1 for an empty range) and each warp merges its head's rows with
                // the running log-sum-exp rule, four rows' loads in flight per lane.
                const int n_list = c_last - c_first + 1;
                for (int i = tid; i < n_list; i += NCW * 32) {
                    const int cc = c_first + i;
                    const long long st0 = hd_cta_start(cc, T, C);
                    contrib[i] = hd_cta_start(cc + 1, T, C) == st0 ? -1 : 2 * cc + (st0 >= seq_t0 ? 0 : 1);
                }
                named_bar_sync(1, NCW * 32);
                constexpr int MR = 4;
                for (int rb = 0; rb < p.M; rb += MR) {
                    float Mr[MR], Lr[MR];
                    float4 acc[MR];
#pragma unroll
                    for (int k = 0; k < MR; ++k) {
                        Mr[k] = NEG_INF;
                        Lr[k] = 0.f;
                        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    for (int j = 0; j < n_list; ++j) {
                        const int sj = contrib[j];
                        if (sj < 0) continue;
                        const long long base = ((long long)sj * kHdHeads + h) * kHdRows;
                        float2 ml[MR];
                        float4 oc[MR];
#pragma unroll
                        for (int k = 0; k < MR; ++k) {
                            const int r = min(rb + k, kHdRows - 1);
                            ml[k] = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + (base + r) * 2));
                            oc[k] = __ldcg(reinterpret_cast<const float4 *>(p.part_o + (base + r) * kHdD + 4 * lane));
                        }
#pragma unroll
                        for (int k = 0; k < MR; ++k) {
                            const float mn = fmaxf(Mr[k], ml[k].x);
                            const float mu = mn == NEG_INF ? 0.f : mn;
                            const float fa = fast_exp2((Mr[k] - mu) * sl), fb = fast_exp2((ml[k].x - mu) * sl);
                            Lr[k] = Lr[k] * fa + ml[k].y * fb;
                            acc[k].x = acc[k].x * fa + oc[k].x * fb;
                            acc[k].y = acc[k].y * fa + oc[k].y * fb;
                            acc[k].z = acc[k].z * fa + oc[k].z * fb;
                            acc[k].w = acc[k].w * fa + oc[k].w * fb;
                            Mr[k] = mn;
                        }
                    }
#pragma unroll
                    for (int k = 0; k < MR; ++k) {
                        const int r = rb + k;
                        if (r >= p.M) continue;
                        const float inv = Lr[k] > 0.f ? 1.f / Lr[k] : 0.f;
                        uint2 pk;
                        pk.x = pack_bf16(acc[k].x * inv, acc[k].y * inv);
                        pk.y = pack_bf16(acc[k].z * inv, acc[k].w * inv);
                        *reinterpret_cast<uint2 *>(ob + (r / p.G) * q_tok_stride + (r % p.G) * kHdD + 4 * lane) = pk;
                    }
                }
            }
            named_bar_sync(1, NCW * 32);
        }
        t += nseg;
    }
}

// ---------------------------------------------------------------------------
// 17 to 24 query rows per KV head (G * n_q, e.g. 20 rows for 4 query heads and
// 5 speculated tokens): the same traversal and schedule, with the operands of
// both products swapped so that the query rows fill 8-wide n-tiles instead of
// 16-row m-tiles (20 rows cost 24 rather than 32).  A tile is 16 positions
// (two 8-position stages).  Warp h, KV head h:
//   S^T (16 positions x 8 NT rows) = K_h (m16, k = channels) x Q_h^T, the
//   query fragments held in registers for the sequence's run;
//   the row maxima reduce over the 8 lanes holding a row's 16 positions;
//   P^T is the S^T accumulator re-packed and transposed in registers
//   (movmatrix) into the B operand of O^T (128 channels x 8 NT rows) +=
//   V_h^T (m16 per 16 channels, k = positions) x P^T.
// Three warpgroups: two of consumers (warps 0-7) and one whose first thread is
// the producer.  The consumers' O^T takes 32 NT registers per thread, so the
// producer warpgroup hands its registers over: at launch 384 threads x 168,
// then 128 x 24 (producer group) + 256 x 232 (consumers) = 62464 <= 64512, and
// per sub-partition (two consumer warps and one producer-group warp)
// 2 x 32 x 232 + 32 x 24 = 15616 <= 16384.
constexpr int kHdTThreads = 3 * 128;
constexpr int kHdTRegsProducer = 24;
constexpr int kHdTRegsConsumer = 232;

template <int NT>
__global__ void __launch_bounds__(kHdTThreads, 1)
    verify_heads_t_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                          const __grid_constant__ CUtensorMap tmq, const HeadsParams p) {
    constexpr int NCW = kHdHeads;
    constexpr int KS = kHdD / 16;              // k-steps of S^T = K Q^T
    constexpr int MTD = kHdD / 16;             // 16-channel m-tiles of O^T
    constexpr int TP = 2 * kHdPos;             // positions per tile
    constexpr int RW = 8 * NT;                 // rows a warp holds (padded)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int stages = p.stages;
    const int QHALF = p.H_q * p.n_q * 128;     // one 64-channel half of the query box (a multiple of 1 KB)
    uint8_t *stage_base = smem;
    uint8_t *qslot = smem + (size_t)stages * kHdStage;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(qslot + 2 * QHALF);
    uint64_t *empty_bar = full_bar + kHdMaxStages;
    uint64_t *qfull = empty_bar + kHdMaxStages;
    uint64_t *qempty = qfull + 1;
    int *flag = reinterpret_cast<int *>(qempty + 1);
    int *contrib = flag + 4;                   // [gridDim.x + 1]
    int *prefix = contrib + gridDim.x + 1;     // [B+1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NCW);
        }
        mbar_init(qfull, 1);
        mbar_init(qempty, NCW);
        mbar_fence_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        prefetch_tensormap(&tmq);
    }
    pdl_wait();
    // 16-position tiles per sequence, loaded in parallel, then an exclusive scan by warp 0.
    for (int b = tid; b < p.B; b += blockDim.x)
        prefix[b] = (hd_clamp(checked(ld_dep(p.len + b), 0, p.L_cap, p.err), p.L_cap) + TP - 1) / TP;
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

    const long long T = prefix[p.B];
    const int C = gridDim.x, c = blockIdx.x;
    const long long t_begin = hd_cta_start(c, T, C), t_end = hd_cta_start(c + 1, T, C);
    const long long q_tok_stride = (long long)p.H_q * kHdD;

    if (warp >= NCW) {
        // ------------------------------------------------------- producer (1 thread)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kHdTRegsProducer));
        if (warp != NCW || lane != 0) return;
        const uint64_t pol = policy_evict_normal();
        const uint64_t pol_q = policy_evict_first();
        int stage = 0, seg_no = 0, issued = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long t = t_begin; t < t_end && ok; ++seg_no) {
            const int b = hd_seq_of(t, prefix, p.B);
            const int ti0 = (int)(t - prefix[b]);
            const int nseg = (int)min((long long)prefix[b + 1] - t, t_end - t);
            // the query rows of all heads; the slot is free once every consumer
            // warp has taken the previous sequence's rows into registers
            if (!mbar_wait(qempty, (uint32_t)(seg_no & 1) ^ 1u, p.err)) { ok = false; break; }
            mbar_arrive_expect_tx(qfull, 2 * QHALF);
            tma_load_4d(qslot, &tmq, 0, 0, 0, b, qfull, pol_q);
            tma_load_4d(qslot + QHALF, &tmq, 64, 0, 0, b, qfull, pol_q);
            for (int i = 0; i < 2 * nseg; ++i) {        // two 8-position stages per tile
                if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) { ok = false; break; }
                mbar_arrive_expect_tx(&full_bar[stage], kHdStage);
                uint8_t *sk = stage_base + (size_t)stage * kHdStage;
                uint8_t *sv = sk + 2 * kHdHalf;
                const int pos0 = ti0 * TP + i * kHdPos;
                tma_load_4d(sk, &tmk, 0, pos0, 0, b, &full_bar[stage], pol);
                tma_load_4d(sk + kHdHalf, &tmk, 64, pos0, 0, b, &full_bar[stage], pol);
                tma_load_4d(sv, &tmv, 0, pos0, 0, b, &full_bar[stage], pol);
                tma_load_4d(sv + kHdHalf, &tmv, 64, pos0, 0, b, &full_bar[stage], pol);
                ++issued;
                if (++stage == stages) { stage = 0; phase ^= 1u; }
            }
            t += nseg;
        }
        // Drain: do not leave the CTA while copies issued here may still land.
        int st = stage;
        uint32_t ph = phase;
        for (int k = 0; k < min(issued, stages); ++k) {
            if (st == 0) { st = stages - 1; ph ^= 1u; } else { --st; }
            mbar_wait(&full_bar[st], ph, p.err);
        }
        if (seg_no > 0) mbar_wait(qfull, (uint32_t)((seg_no - 1) & 1), p.err);
        return;
    }

    // ---------------------------------------------------------------- consumers
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kHdTRegsConsumer));
    const int h = warp;                                // KV head of this warp
    const int g = lane >> 2, t4 = lane & 3;
    const int mat = lane >> 3, rr = lane & 7;          // ldmatrix: matrix and row this lane addresses
    const float sl = p.scale_log2;
    const float NEG_INF = -INFINITY;

    // Sequences with nothing to attend produce zero rows.
    for (int b = c; b < p.B; b += C) {
        if (prefix[b + 1] != prefix[b]) continue;
        uint4 *o = reinterpret_cast<uint4 *>(p.out + (long long)b * p.n_q * q_tok_stride);
        const int n16 = p.n_q * p.H_q * kHdD / 8;
        for (int i = tid; i < n16; i += NCW * 32) o[i] = make_uint4(0, 0, 0, 0);
    }

    // Row r < M of this head is query token r / G of query head h*G + r % G.
    // The B-operand rows a lane supplies to ldmatrix: row nt*8 + rr (rows past
    // M read row 0 and are zeroed); the rows whose S^T / O^T columns it holds:
    // nt*8 + 2*t4 + e, e = 0, 1.
    // The query slot of this kernel is head-major: row (query head, token).
    auto qrow = [&](int r) { return (h * p.G + r % p.G) * p.n_q + r / p.G; };
    const uint32_t qbase = smem_u32(qslot);

    int stage = 0, seg_no = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (long long t = t_begin; t < t_end; ++seg_no) {
        const int b = hd_seq_of(t, prefix, p.B);
        const int ti0 = (int)(t - prefix[b]);
        const int nseg = (int)min((long long)prefix[b + 1] - t, t_end - t);
        const int len = hd_clamp(ld_dep(p.len + b), p.L_cap);
        // The query rows as B fragments (k = channels, n = rows), held in registers
        // for the run (the slot is released at once).  Lanes address rows nt*8 + rr
        // of the slot; the lanes whose fragments hold a row past M zero them.
        uint32_t qb[KS][NT][2];
        if (ok) ok = mbar_wait(qfull, (uint32_t)(seg_no & 1), p.err);
        {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int qr = nt * 8 + rr < p.M ? qrow(nt * 8 + rr) : 0;
                const bool valid = nt * 8 + g < p.M;
#pragma unroll
                for (int k2 = 0; k2 < KS / 2; ++k2) {
                    // chunks 4*k2 .. 4*k2+3 = k-steps 2*k2 (b0, b1) and 2*k2 + 1
                    const int ch = 4 * k2 + mat;
                    uint32_t q0, q1, q2, q3;
                    ldsm_x4(qbase + (ch >> 3) * QHALF + swz128(qr, ch & 7), q0, q1, q2, q3);
                    qb[2 * k2][nt][0] = valid ? q0 : 0u;
                    qb[2 * k2][nt][1] = valid ? q1 : 0u;
                    qb[2 * k2 + 1][nt][0] = valid ? q2 : 0u;
                    qb[2 * k2 + 1][nt][1] = valid ? q3 : 0u;
                }
            }
            fence_proxy_async_smem();   // reads done before TMA may refill the slot
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty);
        }

        float o[MTD][NT][4];
#pragma unroll
        for (int mt = 0; mt < MTD; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        float m_r[NT][2], l_r[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) m_r[nt][0] = m_r[nt][1] = NEG_INF, l_r[nt][0] = l_r[nt][1] = 0.f;

        for (int i = 0; i < nseg; ++i) {
            int st2[2];
            uint32_t ph2[2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                st2[x] = stage;
                ph2[x] = phase;
                if (++stage == stages) { stage = 0; phase ^= 1u; }
            }
            if (ok) ok = mbar_wait(&full_bar[st2[0]], ph2[0], p.err);
            if (ok) ok = mbar_wait(&full_bar[st2[1]], ph2[1], p.err);
            if (ok) {
                uint8_t *ktA = stage_base + (size_t)st2[0] * kHdStage, *ktB = stage_base + (size_t)st2[1] * kHdStage;
                uint8_t *vtA = ktA + 2 * kHdHalf, *vtB = ktB + 2 * kHdHalf;
                const int pos0 = (ti0 + i) * TP;
                if (pos0 + TP > len) {
                    // rows at or past the sequence end hold whatever the cache holds
                    // there: zero this head's V rows so P = 0 meets finite values
                    for (int idx = lane; idx < TP * 16; idx += 32) {
                        const int pp = idx >> 4, ch = idx & 15;
                        if (pos0 + pp >= len)
                            *reinterpret_cast<uint4 *>((pp < kHdPos ? vtA : vtB) + (ch >> 3) * kHdHalf +
                                                       swz128(h * kHdPos + (pp & (kHdPos - 1)), ch & 7)) =
                                make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                // K rows of this lane's ldmatrix: positions (mat & 1) * 8 + rr (stage A or B)
                const uint32_t kb = smem_u32((mat & 1) ? ktB : ktA);
                // S^T = K Q^T: 16 positions x 8 NT rows
                float s[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    // channel chunks 2*ks (matrices 0, 1) and 2*ks + 1 (2, 3)
                    uint32_t a[4];
                    {
                        const int ch = 2 * ks + (mat >> 1);
                        ldsm_x4(kb + (ch >> 3) * kHdHalf + swz128(h * kHdPos + rr, ch & 7), a[0], a[1], a[2], a[3]);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16(s[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
                }
                // S^T element (position pos0 + g + 8*(j>>1), row nt*8 + 2*t4 + (j&1))
                if (pos0 + TP - 1 > len - p.n_q) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            // the last position row nt*8 + 2*t4 + (j&1) may see
                            const int r = nt * 8 + 2 * t4 + (j & 1);
                            const int lim = r < p.M ? len - p.n_q + r / p.G : len - 1;
                            if (pos0 + g + 8 * (j >> 1) > lim) s[nt][j] = NEG_INF;
                        }
                }
                // online softmax per row: the 16 positions of a row are held by the 8
                // lanes sharing t4 (two each)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float al[2];
                    bool moved = false;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float mx = fmaxf(s[nt][e], s[nt][2 + e]);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float mn = fmaxf(m_r[nt][e], mx);
                        const float mu = mn == NEG_INF ? 0.f : mn;
                        al[e] = fast_exp2((m_r[nt][e] - mu) * sl);
                        moved |= al[e] != 1.f;
                        const float ms = mu * sl;
                        s[nt][e] = fast_exp2(fmaf(s[nt][e], sl, -ms));
                        s[nt][2 + e] = fast_exp2(fmaf(s[nt][2 + e], sl, -ms));
                        l_r[nt][e] = l_r[nt][e] * al[e] + (s[nt][e] + s[nt][2 + e]);
                        m_r[nt][e] = mn;
                    }
                    // once a row's maximum settles its factor is exactly 1
                    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                        for (int mt = 0; mt < MTD; ++mt) {
                            o[mt][nt][0] *= al[0];
                            o[mt][nt][1] *= al[1];
                            o[mt][nt][2] *= al[0];
                            o[mt][nt][3] *= al[1];
                        }
                    }
                }
                // P^T as the B operand (k = positions, n = rows): the accumulator's
                // (position g, rows 2t4, 2t4+1) pairs, transposed in registers
                uint32_t pb[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    pb[nt][0] = movmatrix_trans(pack_bf16(s[nt][0], s[nt][1]));   // positions 0-7
                    pb[nt][1] = movmatrix_trans(pack_bf16(s[nt][2], s[nt][3]));   // positions 8-15
                }
                // O^T += V^T P^T: per 16-channel m-tile, V rows of positions 0-7
                // (matrices 0, 1) and 8-15 (2, 3), channels lo (0, 2) and hi (1, 3)
                const uint32_t vb = smem_u32((mat >> 1) ? vtB : vtA);
#pragma unroll
                for (int mt = 0; mt < MTD; ++mt) {
                    const int ch = 2 * mt + (mat & 1);
                    uint32_t a[4];
                    ldsm_x4_trans(vb + (ch >> 3) * kHdHalf + swz128(h * kHdPos + rr, ch & 7), a[0], a[1], a[2], a[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16(o[mt][nt], a, pb[nt][0], pb[nt][1]);
                }
            }
            fence_proxy_async_smem();   // reads done before TMA may refill the buffers
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty_bar[st2[0]]);
                mbar_arrive(&empty_bar[st2[1]]);
            }
        }

        // ------------------------------------------------ end of this CTA's run of the sequence
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = l_r[nt][e];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                l_r[nt][e] = l;
            }
        const long long seq_t0 = prefix[b];
        const int ntiles = prefix[b + 1] - prefix[b];
        const int c_first = hd_cta_of(seq_t0, T, C), c_last = hd_cta_of(seq_t0 + ntiles - 1, T, C);
        const int n_contrib = min(c_last - c_first + 1, ntiles);
        __nv_bfloat16 *ob = p.out + (long long)b * p.n_q * q_tok_stride + (long long)h * p.G * kHdD;
        if (n_contrib == 1) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = nt * 8 + 2 * t4 + e;
                    if (r >= p.M) continue;
                    const float inv = l_r[nt][e] > 0.f ? 1.f / l_r[nt][e] : 0.f;
                    __nv_bfloat16 *orow = ob + (r / p.G) * q_tok_stride + (r % p.G) * kHdD;
#pragma unroll
                    for (int mt = 0; mt < MTD; ++mt) {
                        orow[16 * mt + g] = __float2bfloat16(o[mt][nt][e] * inv);
                        orow[16 * mt + 8 + g] = __float2bfloat16(o[mt][nt][2 + e] * inv);
                    }
                }
        } else {
            // Partial slots: CTA c keeps 2c (its first run, when its range starts
            // inside a sequence split across CTAs) and 2c+1 (its last run); a
            // warp's slot holds its head's rows (up to RW) x 128 channels.
            const int slot = 2 * c + (t_begin >= seq_t0 ? 0 : 1);
            float *po = p.part_o + ((long long)slot * kHdHeads + h) * RW * kHdD;
            float *pml = p.part_ml + ((long long)slot * kHdHeads + h) * RW * 2;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = nt * 8 + 2 * t4 + e;
#pragma unroll
                    for (int mt = 0; mt < MTD; ++mt) {
                        po[r * kHdD + 16 * mt + g] = o[mt][nt][e];
                        po[r * kHdD + 16 * mt + 8 + g] = o[mt][nt][2 + e];
                    }
                    if (g == 0) *reinterpret_cast<float2 *>(pml + r * 2) = make_float2(m_r[nt][e], l_r[nt][e]);
                }
            named_bar_sync(1, NCW * 32);
            if (tid == 0) {
                const int old = atomic_add_acq_rel_gpu(p.counters + b, 1);
                const int last = (old == n_contrib - 1);
                if (old >= n_contrib) raise_error(p.err, kErrState);
                if (last) p.counters[b] = 0;
                *flag = last;
            }
            named_bar_sync(1, NCW * 32);
            if (*flag) {
                const int n_list = c_last - c_first + 1;
                for (int i = tid; i < n_list; i += NCW * 32) {
                    const int cc = c_first + i;
                    const long long st0 = hd_cta_start(cc, T, C);
                    contrib[i] = hd_cta_start(cc + 1, T, C) == st0 ? -1 : 2 * cc + (st0 >= seq_t0 ? 0 : 1);
                }
                named_bar_sync(1, NCW * 32);
                constexpr int MR = 4;
                for (int rb = 0; rb < p.M; rb += MR) {
                    float Mr[MR], Lr[MR];
                    float4 acc[MR];
#pragma unroll
                    for (int k = 0; k < MR; ++k) {
                        Mr[k] = NEG_INF;
                        Lr[k] = 0.f;
                        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    for (int j = 0; j < n_list; ++j) {
                        const int sj = contrib[j];
                        if (sj < 0) continue;
                        const long long base = ((long long)sj * kHdHeads + h) * RW;
                        float2 ml[MR];
                        float4 oc[MR];
#pragma unroll
                        for (int k = 0; k < MR; ++k) {
                            const int r = min(rb + k, RW - 1);
                            ml[k] = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + (base + r) * 2));
                            oc[k] = __ldcg(reinterpret_cast<const float4 *>(p.part_o + (base + r) * kHdD + 4 * lane));
                        }
#pragma unroll
                        for (int k = 0; k < MR; ++k) {
                            const float mn = fmaxf(Mr[k], ml[k].x);
                            const float mu = mn == NEG_INF ? 0.f : mn;
                            const float fa = fast_exp2((Mr[k] - mu) * sl), fb = fast_exp2((ml[k].x - mu) * sl);
                            Lr[k] = Lr[k] * fa + ml[k].y * fb;
                            acc[k].x = acc[k].x * fa + oc[k].x * fb;
                            acc[k].y = acc[k].y * fa + oc[k].y * fb;
                            acc[k].z = acc[k].z * fa + oc[k].z * fb;
                            acc[k].w = acc[k].w * fa + oc[k].w * fb;
                            Mr[k] = mn;
                        }
                    }
#pragma unroll
                    for (int k = 0; k < MR; ++k) {
                        const int r = rb + k;
                        if (r >= p.M) continue;
                        const float inv = Lr[k] > 0.f ? 1.f / Lr[k] : 0.f;
                        uint2 pk;
                        pk.x = pack_bf16(acc[k].x * inv, acc[k].y * inv);
                        pk.y = pack_bf16(acc[k].z * inv, acc[k].w * inv);
                        *reinterpret_cast<uint2 *>(ob + (r / p.G) * q_tok_stride + (r % p.G) * kHdD + 4 * lane) = pk;
                    }
                }
            }
            named_bar_sync(1, NCW * 32);
        }
        t += nseg;
    }
}

// ------------------------------------------------------------------- host side

static int hd_env_int(const char *name, int dflt) {
    const char *s = getenv(name);
    if (!s || !*s) return dflt;
    return atoi(s);
}

// Shapes these kernels cover: d = 128, eight KV heads, G * n_q <= 24 query rows
// per KV head (verify_heads_kernel up to 16, verify_heads_t_kernel 17 to 24).
constexpr int kHdRowsT = 24;
bool verify_heads_supported(int H_kv, int D, int M) { return H_kv == kHdHeads && D == kHdD && M >= 1 && M <= kHdRowsT; }

// Rows of a warp's partial slot: 16, or 8 per n-tile of the swapped kernel.
static int hd_slot_rows(int M) { return M <= kHdRows ? kHdRows : (M + 7) / 8 * 8; }

// Workspace for `ctas` CTAs: [counters | scheduler] (kAttnCounterBytes, left
// zero by every call), then part_o [2*ctas][8][rows][128] fp32 and part_ml
// [2*ctas][8][rows][2] fp32, rows = 16 for up to 16 query rows per KV head,
// else the rows rounded up to 8.
size_t verify_heads_ws_bytes(int ctas, int M) {
    const size_t rows = (size_t)2 * ctas * kHdHeads * hd_slot_rows(M);
    return kAttnCounterBytes + rows * kHdD * 4 + rows * 2 * 4;
}

// MAGICDEC_ERR_WORKSPACE when `ws_bytes` cannot hold this kernel's partials
// (the caller then runs the per-pair kernel).
magicdec_status launch_verify_heads(int B, int H_q, int L_cap, int n_q, const void *q, const void *k, const void *v,
                                    const int32_t *len, void *out, void *ws, size_t ws_bytes, cudaStream_t st) {
    HeadsParams prm{};
    prm.G = H_q / kHdHeads;
    prm.M = prm.G * n_q;
    int ctas_per_sm = hd_env_int("MAGICDEC_ATTN_CTAS_PER_SM", 1);
    ctas_per_sm = ctas_per_sm < 1 ? 1 : (ctas_per_sm > 2 ? 2 : ctas_per_sm);
    const int C = magicdec_host::sm_count() * ctas_per_sm;
    if (C + 1 > kHdMaxContrib) return MAGICDEC_ERR_UNSUPPORTED;
    if (ws_bytes < verify_heads_ws_bytes(C, prm.M)) return MAGICDEC_ERR_WORKSPACE;
    const size_t qhalf = (size_t)H_q * n_q * 128;
    const size_t fixed = 1024 /* alignment slack */ + 2 * qhalf + (2 * kHdMaxStages + 2) * 8 + 16 +
                         (size_t)(C + 1) * 4 + (size_t)(B + 1) * 4;
    const int smem_cap = magicdec_host::max_smem_optin();
    const size_t per_cta_cap = ctas_per_sm == 1 ? (size_t)smem_cap : (size_t)(smem_cap / 2 - 1024);
    if (per_cta_cap <= fixed) return MAGICDEC_ERR_UNSUPPORTED;
    // Five stages (160 KB of K/V in flight per SM) unless MAGICDEC_ATTN_STAGES asks
    // otherwise.  Measured at B=32 and 128 with 2, 3 and 4 query tokens: a sixth
    // stage, where shared memory has room for it, is 4-5 % slower; four are
    // within 1.5 % (slower at B=32 and with 4 tokens); three are 4-5 % slower.
    int stages = (int)((per_cta_cap - fixed) / kHdStage);
    const int want = hd_env_int("MAGICDEC_ATTN_STAGES", 0);
    const int cap = want > 0 ? want : kHdDefaultStages;
    if (cap < stages) stages = cap;
    if (stages > kHdMaxStages) stages = kHdMaxStages;
    if (stages < 2) return MAGICDEC_ERR_UNSUPPORTED;
    const size_t smem = fixed + (size_t)stages * kHdStage;
    // 17 to 24 rows: the swapped-operand kernel (three 8-row n-tiles)
    const bool swapped = prm.M > kHdRows;
    auto kern_t = verify_heads_t_kernel<3>;
    if (cudaFuncSetAttribute(swapped ? kern_t : verify_heads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;

    prm.q = static_cast<const __nv_bfloat16 *>(q);
    prm.len = len;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    uint8_t *w = static_cast<uint8_t *>(ws);
    prm.counters = reinterpret_cast<int *>(w);
    prm.part_o = reinterpret_cast<float *>(w + kAttnCounterBytes);
    prm.part_ml = prm.part_o + (size_t)2 * C * kHdHeads * hd_slot_rows(prm.M) * kHdD;
    prm.err = magicdec_host::device_error_word();
    prm.B = B;
    prm.H_q = H_q;
    prm.n_q = n_q;
    prm.L_cap = L_cap;
    prm.stages = stages;
    prm.scale_log2 = kLog2e / sqrtf((float)kHdD);

    // K, V as (d, L_cap, H_kv, B): the position stride (H_kv*d) precedes the head
    // stride (d), so a box of 64 channels x 8 positions x 8 heads lands head by head.
    CUtensorMap tmk, tmv, tmq;
    const uint64_t e = 2;
    const uint64_t dims[4] = {(uint64_t)kHdD, (uint64_t)L_cap, (uint64_t)kHdHeads, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)kHdHeads * kHdD * e, (uint64_t)kHdD * e,
                                 (uint64_t)L_cap * kHdHeads * kHdD * e};
    const uint32_t box[4] = {64, (uint32_t)kHdPos, (uint32_t)kHdHeads, 1};
    if (!magicdec_host::encode_tmap_bf16_4d(&tmk, k, dims, strides, box) ||
        !magicdec_host::encode_tmap_bf16_4d(&tmv, v, dims, strides, box))
        return MAGICDEC_ERR_CUDA;
    // Queries as (d, H_q, n_q, B); one box = every query row of the sequence,
    // token-major.  The swapped-operand kernel takes them as (d, n_q, H_q, B),
    // head-major: a head's rows then sit at consecutive slot rows, whose
    // swizzle phases differ, so its 8-row ldmatrix reads meet few bank conflicts.
    const uint64_t qdims[4] = {(uint64_t)kHdD, (uint64_t)(swapped ? n_q : H_q), (uint64_t)(swapped ? H_q : n_q),
                               (uint64_t)B};
    const uint64_t qstrides[3] = {swapped ? (uint64_t)H_q * kHdD * e : (uint64_t)kHdD * e,
                                  swapped ? (uint64_t)kHdD * e : (uint64_t)H_q * kHdD * e,
                                  (uint64_t)n_q * H_q * kHdD * e};
    const uint32_t qbox[4] = {64, (uint32_t)(swapped ? n_q : H_q), (uint32_t)(swapped ? H_q : n_q), 1};
    if (!magicdec_host::encode_tmap_bf16_4d(&tmq, q, qdims, qstrides, qbox)) return MAGICDEC_ERR_CUDA;
    if (swapped)
        return magicdec_host::launch_pdl(kern_t, dim3(C), dim3(kHdTThreads), smem, st, tmk, tmv, tmq, prm);
    return magicdec_host::launch_pdl(verify_heads_kernel, dim3(C), dim3((kHdHeads + 1) * 32), smem, st, tmk, tmv, tmq,
                                     prm);
}

}  // namespace magicdec
