// snapkv_tc.cu -- SnapKV observation-window scoring on the fifth-generation
// tensor cores (tcgen05 + TMEM), sm_103a.
//
// SnapKV selection (MagicDec paper section 4.4 / section 5.2) scores every
// prefix position j of a (sequence, KV head) pair by the softmax probability
// that the w observation-window queries of the G query heads of the group put
// on it.  With M = w*G = 128..160 query rows and d = 128 channels, each
// 128-key tile of K is a real 128 x 128 x 128 contraction (128 flop per K
// byte), which the warp-level mma.sync path cannot feed from shared memory at
// HBM speed.  Here one thread issues tcgen05.mma from shared-memory
// descriptors into a double-buffered TMEM accumulator, and four epilogue
// warps drain it with tcgen05.ld while the next tile's MMAs run:
//
//   pass 1  S = Q K^T   (M = 128 query rows per row block, N = 128 keys):
//           thread = query row; online max / sum of exp2 over the chunk's keys
//           (causal mask inside the window), one (max, sum) partial per row
//           and chunk;
//   pass 2  S^T = K Q^T (M = 128 keys, N = rows padded to 32): thread = key;
//           the score of the key is the sum over rows of exp2(s - lse_row),
//           a per-thread loop, no cross-thread reduction.
//
// Roles (192 threads): warp 0 issues TMA boxes (the window queries once, then
// 128-key x 64-channel K boxes, 128-byte swizzled, into a 4-stage ring);
// warp 1 owns the TMEM allocation and its lane 0 issues the MMAs; warps 2-5
// are the epilogue (warp w reads TMEM lanes 32*(w%4)..+31).  Every wait is
// bounded; on a timeout each role stops, the MMA issuer waits (bounded) for
// its MMAs, and the TMEM columns are always released.
#include "common.cuh"

namespace magicdec {

constexpr int kTcKeys = 128;                 // keys per K tile
constexpr int kTcChunk = 4096;               // positions per CTA
constexpr int kTcStages = 2;           // 2 stages: two CTAs per SM, one streams while the other sets up
constexpr int kTcThreads = 192;
constexpr int kTcHalf = kTcKeys * 128;       // one 128-key x 64-channel swizzled box (16 KB)

struct SnapTcParams {
    const int32_t *len;
    float *part;       // [B, H_kv, n_chunks, RP, 2]: pass-1 (max, sum) per window row and chunk
    float *score;      // [B, H_kv, L_cap]
    int *err;
    int B, H_q, H_kv, G, w, L_cap, M, n_chunks;
    int RB;            // pass-1 row blocks of 128 rows (RP = 128 * RB)
    int NR;            // pass-2 rows padded to a multiple of 32 (the MMA's N)
    float scale_log2;  // log2(e) / sqrt(d)
};

__device__ __forceinline__ int clamp_len_tc(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }

// Lane 0 waits (bounded) and the warp agrees on the outcome, so the
// .sync.aligned TMEM loads that follow always run with the full warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int *err, bool ok, int lane) {
    int got = ok ? 1 : 0;
    if (ok && lane == 0) got = mbar_wait(bar, parity, err) ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    return got != 0;
}

__host__ __device__ constexpr uint32_t tc_pow2_cols(int cols) {
    return cols <= 32 ? 32u : cols <= 64 ? 64u : cols <= 128 ? 128u : cols <= 256 ? 256u : 512u;
}

template <int D, int PASS>
__global__ void __launch_bounds__(kTcThreads, 1)
    snapkv_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
                     const SnapTcParams p) {
    constexpr int HALVES = D / 64;
    constexpr int KT = HALVES * kTcHalf;
    constexpr int KS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int QR = PASS == 1 ? p.RB * 128 : p.NR;        // query rows held in shared memory
    const int QH = QR * 128;                              // bytes of one 64-channel half
    uint8_t *kbuf = smem;
    uint8_t *qbuf = smem + kTcStages * KT;
    float *lse2 = reinterpret_cast<float *>(qbuf + HALVES * QH);     // [256]
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(lse2 + 256);
    uint64_t *empty_bar = full_bar + kTcStages;
    uint64_t *acc_full = empty_bar + kTcStages;          // [2]
    uint64_t *acc_empty = acc_full + 2;                  // [2]
    uint64_t *q_full = acc_empty + 2;
    uint64_t *mma_done = q_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);

    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    pdl_wait();
    const int L = clamp_len_tc(checked(ld_dep(p.len + b), 0, p.L_cap, p.err), p.L_cap);
    if (L < p.w) return;
    const int end = PASS == 1 ? L : L - p.w;
    const int pos_begin = chunk * kTcChunk;
    const int pos_end = min(pos_begin + kTcChunk, end);
    if (pos_begin >= pos_end) return;
    const int ntiles = (pos_end - pos_begin + kTcKeys - 1) / kTcKeys;
    const uint32_t tmem_cols = PASS == 1 ? tc_pow2_cols(p.RB * 2 * 128) : tc_pow2_cols(2 * p.NR);
    const float sl = p.scale_log2;
    const int RP = p.RB * 128;

    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 4);
        }
        mbar_init(q_full, 1);
        mbar_init(mma_done, 1);
        mbar_fence_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmq);
    }
    if (warp == 1) tmem_alloc(tmem_slot, tmem_cols);
    // Query rows M..QR-1 are padding: zero them (the TMA box writes rows < M).
    {
        const int pad = QR - p.M;
        for (int i = tid; i < HALVES * pad * 8; i += kTcThreads) {
            const int hf = i / (pad * 8), rem = i - hf * pad * 8;
            *reinterpret_cast<uint4 *>(qbuf + hf * QH + (p.M + rem / 8) * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (PASS == 2) {
        // log2-sum-exp2 of every window row from the pass-1 partials; padding rows +inf (weight 0)
        const int nvalid = (L + kTcChunk - 1) / kTcChunk;
        const float *pb = p.part + ((long long)b * p.H_kv + h) * p.n_chunks * RP * 2;
        for (int r = tid; r < 256; r += kTcThreads) {
            if (r >= p.M) { lse2[r] = INFINITY; continue; }
            float mx = -INFINITY;
            for (int cc = 0; cc < nvalid; ++cc) mx = fmaxf(mx, pb[((long long)cc * RP + r) * 2]);
            float sm = 0.f;
            for (int cc = 0; cc < nvalid; ++cc)
                sm += pb[((long long)cc * RP + r) * 2 + 1] * fast_exp2((pb[((long long)cc * RP + r) * 2] - mx) * sl);
            lse2[r] = mx * sl + __log2f(sm);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            bool ok = true;
            // window queries of KV head h: rows r = wr*G + g
            mbar_arrive_expect_tx(q_full, (uint32_t)(HALVES * p.M * 128));
#pragma unroll
            for (int hf = 0; hf < HALVES; ++hf) tma_load_4d(qbuf + hf * QH, &tmq, hf * 64, h * p.G, 0, b, q_full, pol);
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            for (int ti = 0; ti < ntiles && ok; ++ti) {
                if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) { ok = false; break; }
                mbar_arrive_expect_tx(&full_bar[stage], KT);
                const int pos0 = pos_begin + ti * kTcKeys;
#pragma unroll
                for (int hf = 0; hf < HALVES; ++hf)
                    tma_load_4d(kbuf + stage * KT + hf * kTcHalf, &tmk, hf * 64, h, pos0, b, &full_bar[stage], pol);
                ++issued;
                if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
            }
            int st = stage;
            uint32_t ph = phase;
            for (int k = 0; k < min(issued, kTcStages); ++k) {
                if (st == 0) { st = kTcStages - 1; ph ^= 1u; } else { --st; }
                mbar_wait(&full_bar[st], ph, p.err);
            }
            mbar_wait(q_full, 0, p.err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = PASS == 1 ? umma_idesc_bf16(128, kTcKeys) : umma_idesc_bf16(128, p.NR);
            bool ok = mbar_wait(q_full, 0, p.err);
            tc_fence_after();
            const uint32_t qb = smem_u32(qbuf);
            int stage = 0;
            uint32_t phase = 0;
            for (int ti = 0; ti < ntiles && ok; ++ti) {
                const int buf = ti & 1;
                const uint32_t acc_phase = (ti >> 1) & 1;
                if (!mbar_wait(&full_bar[stage], phase, p.err)) { ok = false; break; }
                if (!mbar_wait(&acc_empty[buf], acc_phase ^ 1u, p.err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t kt = smem_u32(kbuf + stage * KT);
                if (PASS == 1) {
                    for (int rb = 0; rb < p.RB; ++rb) {
                        const uint32_t d = tmem_base + (uint32_t)((rb * 2 + buf) * 128);
#pragma unroll
                        for (int ks = 0; ks < KS; ++ks) {
                            const uint64_t a = umma_desc_sw128(qb + (ks >> 2) * QH + rb * 128 * 128 + (ks & 3) * 32);
                            const uint64_t bd = umma_desc_sw128(kt + (ks >> 2) * kTcHalf + (ks & 3) * 32);
                            umma_bf16(d, a, bd, idesc, ks > 0);
                        }
                    }
                } else {
                    const uint32_t d = tmem_base + (uint32_t)(buf * p.NR);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const uint64_t a = umma_desc_sw128(kt + (ks >> 2) * kTcHalf + (ks & 3) * 32);
                        const uint64_t bd = umma_desc_sw128(qb + (ks >> 2) * QH + (ks & 3) * 32);
                        umma_bf16(d, a, bd, idesc, ks > 0);
                    }
                }
                umma_commit(&empty_bar[stage]);   // the K stage is free once these MMAs are done
                umma_commit(&acc_full[buf]);      // the accumulator is ready for the epilogue
                if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
            }
            umma_commit(mma_done);
            mbar_wait(mma_done, 0, p.err);
        }
    } else {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;                           // TMEM lane quadrant
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        bool ok = true;
        if (PASS == 1) {
            float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
            int lim[2];
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
                const int r = rb * 128 + 32 * q + lane;
                lim[rb] = r < p.M ? L - p.w + r / p.G : -1;
            }
            for (int ti = 0; ti < ntiles; ++ti) {
                const int buf = ti & 1;
                ok = warp_wait(&acc_full[buf], (ti >> 1) & 1, p.err, ok, lane);
                tc_fence_after();
                const int tile_pos = pos_begin + ti * kTcKeys;
                const bool edge = tile_pos + kTcKeys - 1 > L - p.w || tile_pos + kTcKeys > pos_end;
                for (int rb = 0; rb < p.RB && ok; ++rb) {
#pragma unroll 1
                    for (int c0 = 0; c0 < kTcKeys; c0 += 32) {
                        float v[32];
                        tmem_ld32(tmem_base + lane_addr + (uint32_t)((rb * 2 + buf) * 128 + c0), v);
                        if (edge) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int pos = tile_pos + c0 + j;
                                if (pos > lim[rb] || pos >= pos_end) v[j] = -INFINITY;
                            }
                        }
                        float cm = v[0];
#pragma unroll
                        for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
                        const float mn = fmaxf(m[rb], cm);
                        const float mu = mn == -INFINITY ? 0.f : mn;
                        const float ms = mu * sl;
                        float s = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) s += fast_exp2(fmaf(v[j], sl, -ms));
                        l[rb] = l[rb] * fast_exp2((m[rb] - mu) * sl) + s;
                        m[rb] = mn;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
            float *pb = p.part + (((long long)b * p.H_kv + h) * p.n_chunks + chunk) * RP * 2;
            for (int rb = 0; rb < p.RB; ++rb) {
                const int r = rb * 128 + 32 * q + lane;
                pb[r * 2] = m[rb];
                pb[r * 2 + 1] = l[rb];
            }
        } else {
            float *score_row = p.score + ((long long)b * p.H_kv + h) * p.L_cap;
            for (int ti = 0; ti < ntiles; ++ti) {
                const int buf = ti & 1;
                ok = warp_wait(&acc_full[buf], (ti >> 1) & 1, p.err, ok, lane);
                tc_fence_after();
                float sum = 0.f;
                if (ok) {
#pragma unroll 1
                    for (int c0 = 0; c0 < p.NR; c0 += 32) {
                        float v[32];
                        tmem_ld32(tmem_base + lane_addr + (uint32_t)(buf * p.NR + c0), v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) sum += fast_exp2(fmaf(v[j], sl, -lse2[c0 + j]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
                const int key = pos_begin + ti * kTcKeys + 32 * q + lane;
                if (ok && key < pos_end) score_row[key] = sum;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

// ------------------------------------------------------------------- host side
static size_t align256t(size_t x) { return (x + 255) & ~(size_t)255; }

int snapkv_tc_row_blocks(int M) { return (M + 127) / 128; }

size_t snapkv_tc_workspace_bytes(int B, int H_q, int H_kv, int L_cap, int w) {
    const int M = w * (H_q / H_kv);
    const int RP = snapkv_tc_row_blocks(M) * 128;
    const int n_chunks = (L_cap + kTcChunk - 1) / kTcChunk;
    return align256t((size_t)B * H_kv * n_chunks * RP * 2 * 4) + align256t((size_t)B * H_kv * L_cap * 4) +
           align256t((size_t)B * H_kv * (size_t)((L_cap + 3) & ~3) * 4);
}

template <int D, int PASS>
static magicdec_status launch_tc_pass(const CUtensorMap &tmk, const CUtensorMap &tmq, const SnapTcParams &prm,
                                      cudaStream_t st) {
    const int QR = PASS == 1 ? prm.RB * 128 : prm.NR;
    const size_t smem = 1024 + (size_t)kTcStages * (D / 64) * kTcHalf + (size_t)(D / 64) * QR * 128 + 256 * 4 +
                        (2 * kTcStages + 6) * 8 + 16;
    auto kern = snapkv_tc_kernel<D, PASS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    return magicdec_host::launch_pdl(kern, dim3(prm.n_chunks, prm.H_kv, prm.B), dim3(kTcThreads), smem, st, tmk, tmq,
                                     prm);
}

// Passes 1 and 2 of SnapKV scoring; fills `score` ([B, H_kv, L_cap], the
// prefix [0, L-w) of every pair) for the top-k kernel.
magicdec_status launch_snapkv_scores_tc(int B, int H_q, int H_kv, int D, int L_cap, const void *q_win, const void *k,
                                        const int32_t *seq_len, int w, void *ws, float **score_out,
                                        cudaStream_t st) {
    SnapTcParams prm{};
    prm.len = seq_len;
    prm.B = B;
    prm.H_q = H_q;
    prm.H_kv = H_kv;
    prm.G = H_q / H_kv;
    prm.w = w;
    prm.L_cap = L_cap;
    prm.M = w * prm.G;
    prm.RB = snapkv_tc_row_blocks(prm.M);
    prm.NR = ((prm.M + 31) / 32) * 32;
    if (prm.RB > 2 || prm.NR > 256) return MAGICDEC_ERR_UNSUPPORTED;
    prm.n_chunks = (L_cap + kTcChunk - 1) / kTcChunk;
    prm.scale_log2 = kLog2e / sqrtf((float)D);
    prm.err = magicdec_host::device_error_word();
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    prm.part = reinterpret_cast<float *>(wsb);
    wsb += align256t((size_t)B * H_kv * prm.n_chunks * prm.RB * 128 * 2 * 4);
    prm.score = reinterpret_cast<float *>(wsb);
    *score_out = prm.score;

    // K as (d, H_kv, L_cap, B), boxes of 64 channels x 128 keys; window queries
    // as (d, H_q, w, B), one box = the w*G rows of a KV group (rows wr*G + g).
    CUtensorMap tmk, tmq;
    const uint64_t kd[4] = {(uint64_t)D, (uint64_t)H_kv, (uint64_t)L_cap, (uint64_t)B};
    const uint64_t ks[3] = {(uint64_t)D * 2, (uint64_t)H_kv * D * 2, (uint64_t)L_cap * H_kv * D * 2};
    const uint32_t kb[4] = {64, 1, (uint32_t)kTcKeys, 1};
    const uint64_t qd[4] = {(uint64_t)D, (uint64_t)H_q, (uint64_t)w, (uint64_t)B};
    const uint64_t qs[3] = {(uint64_t)D * 2, (uint64_t)H_q * D * 2, (uint64_t)w * H_q * D * 2};
    const uint32_t qbx[4] = {64, (uint32_t)prm.G, (uint32_t)w, 1};
    if (!magicdec_host::encode_tmap_bf16_4d(&tmk, k, kd, ks, kb) ||
        !magicdec_host::encode_tmap_bf16_4d(&tmq, q_win, qd, qs, qbx))
        return MAGICDEC_ERR_CUDA;
    magicdec_status s;
    if (D == 128) {
        if ((s = launch_tc_pass<128, 1>(tmk, tmq, prm, st)) != MAGICDEC_OK) return s;
        return launch_tc_pass<128, 2>(tmk, tmq, prm, st);
    }
    if (D == 64) {
        if ((s = launch_tc_pass<64, 1>(tmk, tmq, prm, st)) != MAGICDEC_OK) return s;
        return launch_tc_pass<64, 2>(tmk, tmq, prm, st);
    }
    return MAGICDEC_ERR_UNSUPPORTED;
}

}  // namespace magicdec
