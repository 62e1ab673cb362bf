// attn.cu -- batched GQA decode attention for the draft and verification
// passes of MagicDec self-speculative decoding, sm_103a.
//
// Verification (paper section 3.1, T_V(B,S,gamma)): the gamma+1 speculated
// queries of every query head in a KV group attend to the full KV cache
// [B, L_cap, H_kv, d], causal inside the speculated block.  Draft (section
// 4.1, Eq. 3, T_D(B,K)): one query per head over the compact draft cache
// [B, H_kv, cap, d].  Both are the same problem -- M = G * n_q query rows per
// (sequence, KV head) pair streaming that pair's K/V rows once -- so one kernel
// serves both; only the tensor maps (and the order of their coordinates)
// differ.  Verification with d = 128, eight KV heads and M <= 16 runs the
// kernel of attn_heads.cu instead, which streams all heads of a sequence per
// stage (launch_decode_attn below picks it).
//
// Design (HBM-bound: every K/V byte is read exactly once):
//  * Persistent grid, one CTA per SM.  The whole batch's work is a flat list of
//    64-row tiles ordered (sequence, KV head, tile); CTA c takes the contiguous
//    range [c*T/C, (c+1)*T/C), so every SM streams the same number of bytes
//    whatever the length mix.  A pair split across CTAs produces partial
//    (max, sum, unnormalised output) triples that the last CTA to finish the
//    pair merges with the log-sum-exp rule (flash-decoding split-KV; the paper
//    cites flash decoding in section 2).  "Last arriver merges": an atomic
//    counter per pair, never a spin-wait.  The producer hands each run of a
//    pair's tiles (a segment) to the consumers as a descriptor in a two-entry
//    shared-memory ring beside the query slots.  Optional dynamic tails
//    (MAGICDEC_ATTN_TAILS=1): pairs of >= 64 tiles leave their last 1/16 to a
//    pool that CTAs claim after their static share.
//  * One producer thread issues TMA tiled copies: per 64-row tile, one 4-D box
//    of 64 rows x 64 channels per 128-byte half of K and of V, 128-byte
//    swizzled so ldmatrix reads are bank-conflict free, into a ring of STAGES
//    slots guarded by full/empty mbarriers.  Rows past the sequence end are
//    masked (and their V rows zeroed in shared memory, so stale or
//    uninitialised cache rows can never reach the output).
//  * L2 priority of the K/V copies.  Draft: evict_first, so the copies do not
//    push out the part of the compact cache (written by the gather or the
//    draft-cache update just before, larger than L2) that stays resident
//    across the gamma draft calls.  Verify: evict_normal.  The full cache is
//    read once and gains nothing from L2, but with evict_first its lines may
//    only take the ways that normal-priority lines (the draft cache the
//    gather just wrote back, still dirty) leave free, which measurably slowed
//    verification right after a gather (2.57 ms against 2.37 ms per call at
//    B=128, L=32000).
//  * 4*MT consumer warps: warp (mt, pq) owns query rows mt*16..mt*16+15 and
//    key columns pq*16..pq*16+15 of each tile.  S = Q K^T and O += P V run on
//    bf16 mma.sync m16n8k16 with fp32 accumulation (the contraction is
//    16 flop/byte, far below the tensor ridge); the online softmax runs in
//    fp32 with exp2.  At the end of a pair the four column warps of a row tile
//    merge in a fixed order through shared memory (deterministic).
#include "common.cuh"

namespace magicdec {

constexpr int kTileN = 64;      // KV rows per pipeline stage
constexpr int kMaxStages = 8;
constexpr int kHalfBytes = kTileN * 128;   // one 64-row x 64-channel swizzled box
constexpr int kMaxContrib = 512;           // contributors a merge lists in shared memory (CTAs + tail)
constexpr int kTailMinTiles = 64;          // pairs of at least this many tiles have a dynamic tail
constexpr int kTailDiv = 16;               // ... of n / kTailDiv tiles
constexpr int kPrefetchTiles = 5;          // draft tiles per CTA prefetched into L2 before the dependency wait
constexpr int kDraftStages = 4;   // stage ring depth of the draft (head-major) launches

struct AttnParams {
    const __nv_bfloat16 *q;     // [B, n_q, H_q, D]
    const int32_t *len;         // [B]
    __nv_bfloat16 *out;         // [B, n_q, H_q, D]
    float *part_o;              // [2*C + (tails ? 2*B*H_kv : 0), MT*16, D] partial outputs
    float *part_ml;             // same slots, [.., MT*16, 2] (max, sum)
    int *counters;              // [B * H_kv] merge arrivals, zero between calls
    int *sched;                 // [0] tail claims, [1] CTAs finished; zero between calls
    int tails;                  // 1: pairs of >= kTailMinTiles tiles hand their last n/kTailDiv to the pool
    int *err;
    int B, H_q, H_kv, G, n_q, L_cap, M;
    int head_major;             // 0: verify layout [B, L_cap, H_kv, D]; 1: draft [B, H_kv, cap, D]
    int prefetch;               // draft: tiles prefetched into L2 before the dependency wait (0: none)
    int stages;
    float scale_log2;           // log2(e) / sqrt(D)
};

struct Segment {
    int b, h, ti0, ntiles, len;
    long long pair_t0;          // global index of the pair's first tile
};

// One run of consecutive tiles of one pair, handed from the producer to the
// consumer warps through a two-entry ring in shared memory.
struct SegDesc {
    int b, h;                   // the pair
    int ti0, nseg;              // first tile (within the pair) and tile count
    int len;                    // the sequence's clamped length
    int kind;                   // 0: part of the pair's head; 1: its whole tail; -1: no more work
};

__device__ __forceinline__ int clamp_len(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }
__device__ __forceinline__ int tiles_of(int len) { return (len + kTileN - 1) / kTileN; }
// Tiles at the end of an n-tile pair that go to the dynamic pool.
__device__ __forceinline__ int tail_tiles(int n, int tails) { return (tails && n >= kTailMinTiles) ? n / kTailDiv : 0; }

// Pair and tile holding global head tile t.  prefix[b] = head tiles of
// sequences < b (per KV head); the heads of sequence b's pairs occupy
// [H_kv*prefix[b], H_kv*prefix[b+1]).
__device__ __forceinline__ Segment decode_tile(long long t, const int *prefix, const AttnParams &p) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)p.H_kv * prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    Segment s;
    s.b = lo;
    s.ntiles = prefix[lo + 1] - prefix[lo];
    const long long local = t - (long long)p.H_kv * prefix[lo];
    s.h = (int)(local / s.ntiles);
    s.ti0 = (int)(local - (long long)s.h * s.ntiles);
    s.pair_t0 = (long long)p.H_kv * prefix[lo] + (long long)s.h * s.ntiles;
    s.len = clamp_len(ld_dep(p.len + lo), p.L_cap);
    return s;
}

// CTA whose range [c*T/C, (c+1)*T/C) contains tile t.
__device__ __forceinline__ int cta_of(long long t, long long T, int C) {
    return (int)(((t + 1) * (long long)C - 1) / T);
}

__device__ __forceinline__ long long cta_start(int c, long long T, int C) { return T * c / C; }

// The last arriver's merge of a pair's partials (slots contrib[0..n_merge),
// -1 = none): one pass with the running log-sum-exp rule.  Each thread loads
// two contributors' partials of its output vector before using either, so
// their L2 round trips overlap (more in flight costs the streaming loop
// registers: at 201 for D = 128 two CTAs still fit on an SM).
template <int D, int MT>
__device__ __forceinline__ void merge_partials(const AttnParams &p, const int *contrib, int n_merge,
                                            __nv_bfloat16 *ob, long long q_head_stride, int ctid, int NT) {
    const float sl = p.scale_log2;
    const float NEG_INF = -INFINITY;
    constexpr int MP = 1;
    const int n_items = p.M * (D / 4);
    for (int base = 0; base < n_items; base += NT * MP) {
        int ro[MP], co[MP];
        float Mr[MP], Lr[MP];
        float4 acc[MP];
#pragma unroll
        for (int k = 0; k < MP; ++k) {
            const int idx = min(base + ctid + k * NT, n_items - 1);   // clamped duplicates are not stored
            ro[k] = idx / (D / 4);
            co[k] = (idx % (D / 4)) * 4;
            Mr[k] = NEG_INF;
            Lr[k] = 0.f;
            acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int j0 = 0; j0 < n_merge; j0 += 2) {
            int sj[2];
            float2 ml[2][MP];
            float4 oc[2][MP];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                sj[u] = j0 + u < n_merge ? contrib[j0 + u] : -1;
                if (sj[u] < 0) continue;
#pragma unroll
                for (int k = 0; k < MP; ++k) {
                    const long long row = (long long)sj[u] * (MT * 16) + ro[k];
                    ml[u][k] = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + row * 2));
                    oc[u][k] = __ldcg(reinterpret_cast<const float4 *>(p.part_o + row * D + co[k]));
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (sj[u] < 0) continue;
#pragma unroll
                for (int k = 0; k < MP; ++k) {
                    const float mn = fmaxf(Mr[k], ml[u][k].x);
                    const float mu = mn == NEG_INF ? 0.f : mn;
                    const float fa = fast_exp2((Mr[k] - mu) * sl), fb = fast_exp2((ml[u][k].x - mu) * sl);
                    Lr[k] = Lr[k] * fa + ml[u][k].y * fb;
                    acc[k].x = acc[k].x * fa + oc[u][k].x * fb;
                    acc[k].y = acc[k].y * fa + oc[u][k].y * fb;
                    acc[k].z = acc[k].z * fa + oc[u][k].z * fb;
                    acc[k].w = acc[k].w * fa + oc[u][k].w * fb;
                    Mr[k] = mn;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < MP; ++k) {
            if (base + ctid + k * NT >= n_items) continue;
            const int r = ro[k];
            const float inv = Lr[k] > 0.f ? 1.f / Lr[k] : 0.f;
            uint2 pk;
            pk.x = pack_bf16(acc[k].x * inv, acc[k].y * inv);
            pk.y = pack_bf16(acc[k].z * inv, acc[k].w * inv);
            *reinterpret_cast<uint2 *>(ob + (r / p.G) * q_head_stride + (r % p.G) * D + co[k]) = pk;
        }
    }
}

template <int D, int MT>
__global__ void __launch_bounds__((4 * MT + 1) * 32, 1)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmq, const AttnParams p) {
    constexpr int HALVES = D / 64;
    constexpr int TILE_BYTES = HALVES * kHalfBytes;
    constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    constexpr uint32_t TX_BYTES = STAGE_BYTES;
    constexpr int QHALF = MT * 16 * 128;           // one 64-channel half of the query rows
    constexpr int QSLOT = HALVES * QHALF;
    constexpr int NCW = 4 * MT;                    // consumer warps
    constexpr int CS = D + 4;                      // combine buffer row stride (floats)
    constexpr int KS = D / 16;                     // k-steps of QK^T
    constexpr int ND = D / 8;                      // n-tiles of PV

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int stages = p.stages;
    uint8_t *stage_base = smem;
    uint8_t *qslots = smem + (size_t)stages * STAGE_BYTES;   // 2 slots, ring of segment queries
    float *comb = reinterpret_cast<float *>(qslots + 2 * QSLOT);   // [MT][4 warps][16][CS] partial outputs
    float *red_m = comb + MT * 4 * 16 * CS;        // [MT][4][16]
    float *red_l = red_m + MT * 64;
    float *row_m = red_l + MT * 64;                // [MT*16]
    float *row_l = row_m + MT * 16;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(row_l + MT * 16);
    uint64_t *empty_bar = full_bar + kMaxStages;
    uint64_t *qfull_bar = empty_bar + kMaxStages;  // [2]
    uint64_t *qempty_bar = qfull_bar + 2;          // [2]
    int *flag = reinterpret_cast<int *>(qempty_bar + 2);
    SegDesc *desc = reinterpret_cast<SegDesc *>(flag + 4);   // [2] ring beside the query slots
    int *contrib = reinterpret_cast<int *>(desc + 2);        // [kMaxContrib] partial slots of a merged pair
    int *prefix = contrib + kMaxContrib;           // [B+1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NCW);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull_bar[s], 1);
            mbar_init(&qempty_bar[s], NCW);
        }
        mbar_fence_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        prefetch_tensormap(&tmq);
        if (p.prefetch) {
            // While the previous kernel drains (it may be writing this very
            // cache: L2 keeps the prefetched lines coherent), start the first
            // `prefetch` tiles of this CTA's range on their way into L2.  The
            // range is the stream-K split computed as if every sequence had
            // sequence 0's length (read before the wait, so possibly stale: a
            // hint that only picks what to prefetch; the real schedule is
            // computed after the wait).  The draft caches of a step usually
            // have one length for the whole batch, and then the guess is exact.
            const int n = tiles_of(clamp_len(ld_dep(p.len), p.L_cap));
            if (n > 0) {
                const long long T = (long long)p.B * p.H_kv * n;
                const long long t0 = cta_start(blockIdx.x, T, gridDim.x);
                const long long t1 = min(cta_start(blockIdx.x + 1, T, gridDim.x), t0 + p.prefetch);
                for (long long t = t0; t < t1; ++t) {
                    const long long pair = t / n;
                    const int ti = (int)(t - pair * n), b = (int)(pair / p.H_kv), h = (int)(pair - (long long)b * p.H_kv);
#pragma unroll
                    for (int hf = 0; hf < HALVES; ++hf) {
                        tma_prefetch_4d(&tmk, hf * 64, ti * kTileN, h, b);
                        tma_prefetch_4d(&tmv, hf * 64, ti * kTileN, h, b);
                    }
                }
            }
        }
    }
    // Query rows past M stay zero in both slots (the TMA box writes rows < M only).
    for (int i = tid; i < 2 * QSLOT / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(qslots)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    pdl_wait();
    // Head tiles per sequence (all tiles less the dynamic tail), loaded in
    // parallel, then an exclusive scan by warp 0.
    for (int b = tid; b < p.B; b += blockDim.x) {
        const int n = tiles_of(clamp_len(checked(ld_dep(p.len + b), 0, p.L_cap, p.err), p.L_cap));
        prefix[b] = n - tail_tiles(n, p.tails);
    }
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
    const long long t_begin = cta_start(c, T, C), t_end = cta_start(c + 1, T, C);
    const long long q_head_stride = (long long)p.H_q * D;   // between query tokens of one sequence

    if (warp == NCW) {
        // ------------------------------------------------------- producer (1 thread)
        if (lane != 0) return;
        const uint64_t pol = p.head_major ? policy_evict_first() : policy_evict_normal();
        const uint64_t pol_q = policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0, seg_no = 0;
        bool ok = true;
        // Hand one segment to the consumers: its descriptor, and for work its
        // G*n_q query rows (one box per 64-channel half) on the same barrier.
        auto publish = [&](const SegDesc &d) -> bool {
            const int qs = seg_no & 1;
            if (!mbar_wait(&qempty_bar[qs], ((seg_no >> 1) & 1) ^ 1u, p.err)) return false;
            desc[qs] = d;
            if (d.kind >= 0) {
                mbar_arrive_expect_tx(&qfull_bar[qs], HALVES * p.M * 128);
#pragma unroll
                for (int hf = 0; hf < HALVES; ++hf)
                    tma_load_4d(qslots + qs * QSLOT + hf * QHALF, &tmq, hf * 64, d.h * p.G, 0, d.b, &qfull_bar[qs],
                                pol_q);
            } else {
                mbar_arrive(&qfull_bar[qs]);
            }
            ++seg_no;
            return true;
        };
        auto load_tiles = [&](const SegDesc &d) -> bool {
            for (int i = 0; i < d.nseg; ++i) {
                if (!mbar_wait(&empty_bar[stage], phase ^ 1u, p.err)) return false;
                mbar_arrive_expect_tx(&full_bar[stage], TX_BYTES);
                uint8_t *sk = stage_base + (size_t)stage * STAGE_BYTES;
                uint8_t *sv = sk + TILE_BYTES;
                const int pos0 = (d.ti0 + i) * kTileN;
#pragma unroll
                for (int hf = 0; hf < HALVES; ++hf) {
                    if (p.head_major) {
                        tma_load_4d(sk + hf * kHalfBytes, &tmk, hf * 64, pos0, d.h, d.b, &full_bar[stage], pol);
                        tma_load_4d(sv + hf * kHalfBytes, &tmv, hf * 64, pos0, d.h, d.b, &full_bar[stage], pol);
                    } else {
                        tma_load_4d(sk + hf * kHalfBytes, &tmk, hf * 64, d.h, pos0, d.b, &full_bar[stage], pol);
                        tma_load_4d(sv + hf * kHalfBytes, &tmv, hf * 64, d.h, pos0, d.b, &full_bar[stage], pol);
                    }
                }
                ++issued;
                if (++stage == stages) { stage = 0; phase ^= 1u; }
            }
            return true;
        };
        // This CTA's static share of the heads ...
        for (long long t = t_begin; t < t_end && ok;) {
            const Segment s = decode_tile(t, prefix, p);
            const int nseg = (int)min((long long)(s.ntiles - s.ti0), t_end - t);
            const SegDesc d{s.b, s.h, s.ti0, nseg, s.len, 0};
            ok = publish(d) && load_tiles(d);
            t += nseg;
        }
        // ... then tails claimed one pair at a time until none is left.
        if (p.tails) {
            const int n_pairs = p.B * p.H_kv;
            while (ok) {
                const int j = atomicAdd(p.sched, 1);
                if (j >= n_pairs) break;
                const int b = j / p.H_kv, h = j - b * p.H_kv;
                const int len = clamp_len(ld_dep(p.len + b), p.L_cap);
                const int n = tiles_of(len), tl = tail_tiles(n, 1);
                if (tl == 0) continue;
                const SegDesc d{b, h, n - tl, tl, len, 1};
                ok = publish(d) && load_tiles(d);
            }
        }
        if (ok) ok = publish(SegDesc{0, 0, 0, 0, 0, -1});
        // Drain: do not leave the CTA while copies issued here may still land.
        int st = stage;
        uint32_t ph = phase;
        for (int k = 0; k < min(issued, stages); ++k) {
            if (st == 0) { st = stages - 1; ph ^= 1u; } else { --st; }
            mbar_wait(&full_bar[st], ph, p.err);
        }
        // The query slots: the last two published segments hold the only copies
        // that may still be in flight (the end marker's phase completes at once).
        for (int k = max(0, seg_no - 2); k < seg_no; ++k) mbar_wait(&qfull_bar[k & 1], (k >> 1) & 1, p.err);
        if (p.tails) {
            // Every CTA has made its last claim before it counts itself here; the
            // last one leaves both words zero for the next call.
            const int old = atomic_add_acq_rel_gpu(p.sched + 1, 1);
            if (old == (int)gridDim.x - 1) {
                atomicExch(p.sched, 0);
                atomicExch(p.sched + 1, 0);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int mt = warp >> 2, pq = warp & 3;
    const int g = lane >> 2, t4 = lane & 3;
    const int ctid = tid;                          // 0 .. NCW*32-1
    const int gtid = pq * 32 + lane;               // within the row tile's 4 warps
    const float sl = p.scale_log2;
    const float NEG_INF = -INFINITY;

    // Sequences with nothing to attend produce zero rows.
    for (int b = c; b < p.B; b += C) {
        if (prefix[b + 1] != prefix[b]) continue;
        uint4 *o = reinterpret_cast<uint4 *>(p.out + (long long)b * p.n_q * q_head_stride);
        const int n16 = p.n_q * p.H_q * D / 8;
        for (int i = ctid; i < n16; i += NCW * 32) o[i] = make_uint4(0, 0, 0, 0);
    }

    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int seg_no = 0;; ++seg_no) {
        // The next segment from the producer (its wait failing has raised the
        // error word; nothing more can be trusted, so stop).
        const int qs = seg_no & 1;
        if (!mbar_wait(&qfull_bar[qs], (seg_no >> 1) & 1, p.err)) break;
        const SegDesc d = desc[qs];
        if (d.kind < 0) break;
        const int nseg = d.nseg;

        // Rows owned by this thread: r0 = mt*16+g, r1 = r0+8.  Row r is query
        // token r / G of head h*G + r % G and sees positions <= len-n_q+r/G.
        const int r0 = mt * 16 + g, r1 = r0 + 8;
        const int lim0 = r0 < p.M ? d.len - p.n_q + r0 / p.G : d.len - 1;
        const int lim1 = r1 < p.M ? d.len - p.n_q + r1 / p.G : d.len - 1;
        uint32_t qa[KS][4];
        {
            const uint32_t qbase = smem_u32(qslots + qs * QSLOT);
            const int mat = lane >> 3, rr = lane & 7;
            const int row = mt * 16 + (mat & 1) * 8 + rr;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int ch = ks * 2 + (mat >> 1);
                ldsm_x4(qbase + (ch >> 3) * QHALF + swz128(row, ch & 7), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
            }
            fence_proxy_async_smem();   // reads done before TMA may refill the buffer
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty_bar[qs]);
        }

        float o[ND][4];
#pragma unroll
        for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;

        for (int i = 0; i < nseg; ++i) {
            if (ok) ok = mbar_wait(&full_bar[stage], phase, p.err);
            if (ok) {
                uint8_t *kt = stage_base + (size_t)stage * STAGE_BYTES;
                uint8_t *vt = kt + TILE_BYTES;
                const int tile_pos = (d.ti0 + i) * kTileN;
                if (tile_pos + kTileN > d.len) {
                    // Rows at or past the sequence end hold whatever the cache holds
                    // there: zero this warp's V rows so P = 0 meets finite values.
                    for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
                        const int r = pq * 16 + idx / (D / 8), ch = idx % (D / 8);
                        if (tile_pos + r >= d.len)
                            *reinterpret_cast<uint4 *>(vt + (ch >> 3) * kHalfBytes + swz128(r, ch & 7)) =
                                make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
                float sc[2][4];
#pragma unroll
                for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                {
                    const int mat = lane >> 3, rr = lane & 7;
                    const int row = pq * 16 + (mat >> 1) * 8 + rr;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int ch = ks * 2 + (mat & 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kbase + (ch >> 3) * kHalfBytes + swz128(row, ch & 7), b0, b1, b2, b3);
                        mma_bf16(sc[0], qa[ks], b0, b1);
                        mma_bf16(sc[1], qa[ks], b2, b3);
                    }
                }
                if (tile_pos + kTileN - 1 > d.len - p.n_q) {
                    const int pb = tile_pos + pq * 16 + 2 * t4;
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int pos = pb + n * 8 + e;
                            if (pos > lim0) sc[n][e] = NEG_INF;
                            if (pos > lim1) sc[n][2 + e] = NEG_INF;
                        }
                }
                float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
                float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float mu0 = mn0 == NEG_INF ? 0.f : mn0, mu1 = mn1 == NEG_INF ? 0.f : mn1;
                const float al0 = fast_exp2((m0 - mu0) * sl), al1 = fast_exp2((m1 - mu1) * sl);
                const float ms0 = mu0 * sl, ms1 = mu1 * sl;
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    sc[n][0] = fast_exp2(fmaf(sc[n][0], sl, -ms0));
                    sc[n][1] = fast_exp2(fmaf(sc[n][1], sl, -ms0));
                    sc[n][2] = fast_exp2(fmaf(sc[n][2], sl, -ms1));
                    sc[n][3] = fast_exp2(fmaf(sc[n][3], sl, -ms1));
                }
                l0 = l0 * al0 + (sc[0][0] + sc[0][1] + sc[1][0] + sc[1][1]);
                l1 = l1 * al1 + (sc[0][2] + sc[0][3] + sc[1][2] + sc[1][3]);
                m0 = mn0;
                m1 = mn1;
#pragma unroll
                for (int n = 0; n < ND; ++n) {
                    o[n][0] *= al0; o[n][1] *= al0;
                    o[n][2] *= al1; o[n][3] *= al1;
                }
                uint32_t pa[4];
                pa[0] = pack_bf16(sc[0][0], sc[0][1]);
                pa[1] = pack_bf16(sc[0][2], sc[0][3]);
                pa[2] = pack_bf16(sc[1][0], sc[1][1]);
                pa[3] = pack_bf16(sc[1][2], sc[1][3]);
                {
                    const int mat = lane >> 3, rr = lane & 7;
                    const int row = pq * 16 + (mat & 1) * 8 + rr;
#pragma unroll
                    for (int n2 = 0; n2 < D / 16; ++n2) {
                        const int ch = n2 * 2 + (mat >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(vbase + (ch >> 3) * kHalfBytes + swz128(row, ch & 7), b0, b1, b2, b3);
                        mma_bf16(o[2 * n2], pa, b0, b1);
                        mma_bf16(o[2 * n2 + 1], pa, b2, b3);
                    }
                }
            }
            fence_proxy_async_smem();   // reads done before TMA may refill the buffer
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            if (++stage == stages) { stage = 0; phase ^= 1u; }
        }

        // ----------------------------------------------- merge the 4 column warps
        // Each warp leaves its unnormalised partial (o, m, l) in shared memory;
        // after one barrier every thread of the row tile combines the four
        // partials of its output elements with the log-sum-exp weights.
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        float *rm = red_m + mt * 64, *rl = red_l + mt * 64;
        if (t4 == 0) {
            rm[pq * 16 + g] = m0; rm[pq * 16 + g + 8] = m1;
            rl[pq * 16 + g] = l0; rl[pq * 16 + g + 8] = l1;
        }
        float *cbase = comb + mt * 4 * 16 * CS;
        {
            float *pw = cbase + pq * 16 * CS;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                *reinterpret_cast<float2 *>(pw + g * CS + n * 8 + 2 * t4) = make_float2(o[n][0], o[n][1]);
                *reinterpret_cast<float2 *>(pw + (g + 8) * CS + n * 8 + 2 * t4) = make_float2(o[n][2], o[n][3]);
            }
        }
        named_bar_sync(2 + mt, 128);

        // The pair's contributors: the CTAs whose static ranges overlap its head
        // (with fewer head tiles than CTAs some ranges are empty, so at most
        // `head` of them), plus its tail when it has one.
        const int n_all = tiles_of(d.len), tl = tail_tiles(n_all, p.tails), head = n_all - tl;
        const long long pair_t0 = (long long)p.H_kv * prefix[d.b] + (long long)d.h * head;
        const int c_first = cta_of(pair_t0, T, C);
        const int c_last = cta_of(pair_t0 + head - 1, T, C);
        const int n_static = min(c_last - c_first + 1, head);
        const int n_contrib = n_static + (tl > 0 ? 1 : 0);
        const bool whole = n_contrib == 1;
        const int pair = d.b * p.H_kv + d.h;
        // Partial slots: CTA c keeps 2c (its first segment, when its range
        // starts inside a head split across CTAs) and 2c+1 (its last segment);
        // pair P keeps 2C+2P (its head, when one CTA holds all of it) and
        // 2C+2P+1 (its tail).
        const int slot_id = d.kind == 1 ? 2 * C + 2 * pair + 1
                            : n_static == 1 ? 2 * C + 2 * pair
                                            : 2 * c + (t_begin >= pair_t0 ? 0 : 1);
        __nv_bfloat16 *ob = p.out + (long long)d.b * p.n_q * q_head_stride + (long long)d.h * p.G * D;
        float *po = p.part_o + (long long)slot_id * (MT * 16) * D;
        float *pml = p.part_ml + (long long)slot_id * (MT * 16) * 2;
        for (int idx = gtid; idx < 16 * (D / 8); idx += 128) {
            const int row = idx / (D / 8), col = (idx % (D / 8)) * 8;
            const int r = mt * 16 + row;
            if (whole && r >= p.M) continue;
            float mw[4], Mx = NEG_INF;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                mw[w] = rm[w * 16 + row];
                Mx = fmaxf(Mx, mw[w]);
            }
            const float Mu = Mx == NEG_INF ? 0.f : Mx;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            float Lr = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float f = fast_exp2((mw[w] - Mu) * sl);
                Lr += f * rl[w * 16 + row];
                const float4 a = *reinterpret_cast<const float4 *>(cbase + (w * 16 + row) * CS + col);
                const float4 bq = *reinterpret_cast<const float4 *>(cbase + (w * 16 + row) * CS + col + 4);
                acc[0] += f * a.x; acc[1] += f * a.y; acc[2] += f * a.z; acc[3] += f * a.w;
                acc[4] += f * bq.x; acc[5] += f * bq.y; acc[6] += f * bq.z; acc[7] += f * bq.w;
            }
            if (whole) {
                const float inv = Lr > 0.f ? 1.f / Lr : 0.f;
                uint4 pk;
                pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
                pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
                pk.z = pack_bf16(acc[4] * inv, acc[5] * inv);
                pk.w = pack_bf16(acc[6] * inv, acc[7] * inv);
                *reinterpret_cast<uint4 *>(ob + (r / p.G) * q_head_stride + (r % p.G) * D + col) = pk;
            } else {
                *reinterpret_cast<float4 *>(po + r * D + col) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4 *>(po + r * D + col + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                if (col == 0) {
                    pml[r * 2] = Mx;
                    pml[r * 2 + 1] = Lr;
                }
            }
        }
        if (whole) {
            named_bar_sync(2 + mt, 128);
        } else {
            named_bar_sync(1, NCW * 32);
            if (ctid == 0) {
                // release: this CTA's partial (ordered by the barrier above);
                // acquire: for the last arriver, every other contributor's partial
                const int old = atomic_add_acq_rel_gpu(p.counters + pair, 1);
                const int last = (old == n_contrib - 1);
                if (old >= n_contrib) raise_error(p.err, kErrState);
                if (last) p.counters[pair] = 0;
                *flag = last;
            }
            named_bar_sync(1, NCW * 32);
            if (*flag) {
                // The last arriver lists the contributors' slots in a fixed order
                // (CTAs ascending, then the tail; -1 for an empty CTA range) ...
                const int n_list = n_static == 1 ? 1 : c_last - c_first + 1;
                for (int i = ctid; i < n_list; i += NCW * 32) {
                    int v = 2 * C + 2 * pair;
                    if (n_static != 1) {
                        const int cc = c_first + i;
                        const long long st0 = cta_start(cc, T, C);
                        v = cta_start(cc + 1, T, C) == st0 ? -1 : 2 * cc + (st0 >= pair_t0 ? 0 : 1);
                    }
                    contrib[i] = v;
                }
                if (ctid == 0 && tl > 0) contrib[n_list] = 2 * C + 2 * pair + 1;
                named_bar_sync(1, NCW * 32);
                const int n_merge = n_list + (tl > 0 ? 1 : 0);
                // ... and merges them.
                merge_partials<D, MT>(p, contrib, n_merge, ob, q_head_stride, ctid, NCW * 32);
            }
            named_bar_sync(1, NCW * 32);
        }
    }
}

// ------------------------------------------------------------------- host side

static int env_int(const char *name, int dflt) {
    const char *s = getenv(name);
    if (!s || !*s) return dflt;
    return atoi(s);
}

template <int D, int MT>
static size_t attn_fixed_smem(int B) {
    return 1024 /* alignment slack */ + 2 * (size_t)(D / 64) * MT * 16 * 128 /* query ring */ +
           (size_t)MT * 4 * 16 * (D + 4) * 4 + (size_t)MT * 64 * 4 * 2 + (size_t)MT * 16 * 4 * 2 +
           (2 * kMaxStages + 4) * 8 + 16 + 2 * sizeof(SegDesc) + kMaxContrib * 4 + (size_t)(B + 1) * 4;
}

template <int D>
static constexpr size_t attn_stage_bytes() {
    return 2 * (size_t)(D / 64) * kHalfBytes;
}

// Workspace layout: [counters: kAttnMaxPairs int32 | scheduler: 64 int32],
// always left zero, then the partial slots, part_o [n_slots][rows][D] fp32
// and part_ml [n_slots][rows][2] fp32, rows = M rounded up to 16.  n_slots:
// two per CTA (up to two CTAs per SM) and, when tails are on, two per pair.
// The counter head has a fixed size so that calls of any shape can share
// one workspace; every call leaves it zeroed.
static size_t attn_slots(int B, int H_kv, bool tails) {
    return (size_t)4 * magicdec_host::sm_count() + (tails ? (size_t)2 * B * H_kv : 0);
}

static size_t attn_ws_bytes(int B, int H_kv, int D, int M, bool tails) {
    const size_t rows = (size_t)((M + 15) / 16) * 16, n = attn_slots(B, H_kv, tails);
    return kAttnCounterBytes + n * rows * D * 4 + n * rows * 2 * 4;
}

bool verify_heads_supported(int H_kv, int D, int M);
size_t verify_heads_ws_bytes(int ctas, int M);
magicdec_status launch_verify_heads(int B, int H_q, int L_cap, int n_q, const void *q, const void *k, const void *v,
                                    const int32_t *len, void *out, void *ws, size_t ws_bytes, cudaStream_t st);

// What the entry points ask of callers: room for tails and, where the shape
// allows it, for the all-heads verification kernel at two CTAs per SM.
size_t attn_workspace_bytes(int B, int H_kv, int D, int M) {
    const size_t per_pair = attn_ws_bytes(B, H_kv, D, M, true);
    const size_t heads = verify_heads_supported(H_kv, D, M) ? verify_heads_ws_bytes(2 * magicdec_host::sm_count(), M) : 0;
    return per_pair > heads ? per_pair : heads;
}
// The least the kernel can run with (no tails).
size_t attn_workspace_bytes_min(int B, int H_kv, int D, int M) { return attn_ws_bytes(B, H_kv, D, M, false); }

template <int D, int MT>
static magicdec_status launch_impl(AttnParams prm, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   const CUtensorMap &tmq, int B, void *ws, bool tails, cudaStream_t st) {
    const size_t fixed = attn_fixed_smem<D, MT>(B);
    const size_t sb = attn_stage_bytes<D>();
    const int smem_cap = magicdec_host::max_smem_optin();
    int ctas_per_sm = env_int("MAGICDEC_ATTN_CTAS_PER_SM", 1);
    if (ctas_per_sm < 1) ctas_per_sm = 1;
    if (ctas_per_sm > 2) ctas_per_sm = 2;
    const size_t per_cta_cap = ctas_per_sm == 1 ? (size_t)smem_cap : (size_t)(smem_cap / 2 - 1024);
    if (per_cta_cap <= fixed) return MAGICDEC_ERR_UNSUPPORTED;
    int stages = (int)((per_cta_cap - fixed) / sb);
    const int want = env_int("MAGICDEC_ATTN_STAGES", 0);
    if (want > 0 && want < stages) stages = want;
    // The draft (head-major compact cache) measured 0.3-1 % faster with four
    // stages than with the five that fit, on every draft shape of the bench
    // (B=32..128, budgets 512..4096; CUDA graphs of 96 calls, same GPU).
    else if (want <= 0 && prm.head_major && stages > kDraftStages) stages = kDraftStages;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return MAGICDEC_ERR_UNSUPPORTED;
    const size_t smem = fixed + (size_t)stages * sb;

    auto kern = decode_attn_kernel<D, MT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MAGICDEC_ERR_CUDA;
    const int C = magicdec_host::sm_count() * ctas_per_sm;
    if (C + 1 > kMaxContrib) return MAGICDEC_ERR_UNSUPPORTED;   // a merge lists every CTA and a tail
    // One tail per pair: with fewer than two per CTA the few CTAs that take one
    // finish after everyone else's static share, so the pool would unbalance.
    if ((long long)B * prm.H_kv < 2LL * C) tails = false;
    uint8_t *w = static_cast<uint8_t *>(ws);
    prm.counters = reinterpret_cast<int *>(w);
    prm.sched = prm.counters + kAttnMaxPairs;
    prm.part_o = reinterpret_cast<float *>(w + kAttnCounterBytes);
    prm.part_ml = prm.part_o + attn_slots(B, prm.H_kv, tails) * (MT * 16) * D;
    prm.tails = tails ? 1 : 0;
    prm.stages = stages;
    prm.err = magicdec_host::device_error_word();
    return magicdec_host::launch_pdl(kern, dim3(C), dim3((4 * MT + 1) * 32), smem, st, tmk, tmv, tmq, prm);
}

// Shared launcher for draft (head_major = 1, n_q = 1) and verify attention.
magicdec_status launch_decode_attn(int B, int H_q, int H_kv, int D, int L_cap, int n_q, int head_major,
                                   const void *q, const void *k, const void *v, const int32_t *len, void *out,
                                   void *ws, size_t ws_bytes, cudaStream_t st) {
    AttnParams prm{};
    prm.q = static_cast<const __nv_bfloat16 *>(q);
    prm.len = len;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.B = B;
    prm.H_q = H_q;
    prm.H_kv = H_kv;
    prm.G = H_q / H_kv;
    prm.n_q = n_q;
    prm.L_cap = L_cap;
    prm.M = prm.G * n_q;
    prm.head_major = head_major;
    prm.prefetch = head_major ? env_int("MAGICDEC_ATTN_PREFETCH", kPrefetchTiles) : 0;
    prm.scale_log2 = kLog2e / sqrtf((float)D);

    // Verification of d = 128, eight KV heads and at most 16 query rows per KV
    // head streams all heads of a sequence together (attn_heads.cu) unless the
    // workspace cannot hold its partials (MAGICDEC_ATTN_HEADS=0 turns it off).
    if (!head_major && verify_heads_supported(H_kv, D, prm.M) && env_int("MAGICDEC_ATTN_HEADS", 1) != 0) {
        const magicdec_status s = launch_verify_heads(B, H_q, L_cap, n_q, q, k, v, len, out, ws, ws_bytes, st);
        if (s != MAGICDEC_ERR_WORKSPACE) return s;
    }

    // 4-D views, innermost first.  Verify: (d, H_kv, L_cap, B); draft: (d, cap, H_kv, B).
    CUtensorMap tmk, tmv;
    const uint64_t e = 2;
    uint64_t dims[4], strides[3];
    uint32_t box[4];
    if (head_major) {
        dims[0] = D; dims[1] = L_cap; dims[2] = H_kv; dims[3] = B;
        strides[0] = D * e; strides[1] = (uint64_t)L_cap * D * e; strides[2] = (uint64_t)H_kv * L_cap * D * e;
        box[0] = 64; box[1] = kTileN; box[2] = 1; box[3] = 1;
    } else {
        dims[0] = D; dims[1] = H_kv; dims[2] = L_cap; dims[3] = B;
        strides[0] = D * e; strides[1] = (uint64_t)H_kv * D * e; strides[2] = (uint64_t)L_cap * H_kv * D * e;
        box[0] = 64; box[1] = 1; box[2] = kTileN; box[3] = 1;
    }
    if (!magicdec_host::encode_tmap_bf16_4d(&tmk, k, dims, strides, box) ||
        !magicdec_host::encode_tmap_bf16_4d(&tmv, v, dims, strides, box))
        return MAGICDEC_ERR_CUDA;
    // Queries as (d, H_q, n_q, B); one box = the G*n_q rows of a KV group, rows ordered i*G + g.
    CUtensorMap tmq;
    const uint64_t qdims[4] = {(uint64_t)D, (uint64_t)H_q, (uint64_t)n_q, (uint64_t)B};
    const uint64_t qstrides[3] = {(uint64_t)D * e, (uint64_t)H_q * D * e, (uint64_t)n_q * H_q * D * e};
    const uint32_t qbox[4] = {64, (uint32_t)prm.G, (uint32_t)n_q, 1};
    if (!magicdec_host::encode_tmap_bf16_4d(&tmq, q, qdims, qstrides, qbox)) return MAGICDEC_ERR_CUDA;

    // Dynamic tails are opt-in (MAGICDEC_ATTN_TAILS=1): measured, they tighten
    // the CTAs' finishing times but cost one more partial epilogue per pair, a
    // wash at B=128 and 2.6 % slower at B=64 with 20 rows per KV head.  Only
    // where some pair can have one and the workspace has their slots.
    if (ws_bytes < attn_ws_bytes(B, H_kv, D, prm.M, false)) return MAGICDEC_ERR_WORKSPACE;
    const bool tails = L_cap >= kTailMinTiles * kTileN && ws_bytes >= attn_ws_bytes(B, H_kv, D, prm.M, true) &&
                       env_int("MAGICDEC_ATTN_TAILS", 0) != 0;
    const int MT = (prm.M + 15) / 16;
    if (D == 128) {
        if (MT == 1) return launch_impl<128, 1>(prm, tmk, tmv, tmq, B, ws, tails, st);
        if (MT == 2) return launch_impl<128, 2>(prm, tmk, tmv, tmq, B, ws, tails, st);
    } else if (D == 64) {
        if (MT == 1) return launch_impl<64, 1>(prm, tmk, tmv, tmq, B, ws, tails, st);
        if (MT == 2) return launch_impl<64, 2>(prm, tmk, tmv, tmq, B, ws, tails, st);
    }
    return MAGICDEC_ERR_UNSUPPORTED;
}

}  // namespace magicdec
