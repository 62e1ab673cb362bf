// Draft-cache update: append, post-verification refresh and rollback of the
// compact draft cache.
//
// MagicDec (arXiv 2408.11049) section 4.4: the static drafts (StreamingLLM,
// SnapKV) select their KV once and afterwards only take in new tokens;
// section 3.1: after verification the sequence keeps the accepted prefix, so
// rows the sparse draft wrote for rejected or re-verified positions are
// replaced.  The compact cache kc/vc [B, H_kv, cap, d] has one of two layouts:
//   ring > 0 (StreamingLLM): position q < origin[b] (a sink) at slot q,
//     position q >= origin[b] at slot origin[b] + (q - origin[b]) mod ring;
//   ring == 0 (SnapKV): the selected rows at slots [0, base[b]), position
//     q >= origin[b] at slot base[b] + q - origin[b].
// Per sequence the copies form at most three contiguous ranges of positions
// (see dc_ranges below), so a warp takes (copy, KV head) items and moves one
// K row and one V row with 16-byte lanes.
//
// The step-length kernel below turns (length, accepted count) into the next
// step's lengths, so a multi-step loop keeps its bookkeeping on the device.
#include "common.cuh"

namespace magicdec {

constexpr int kDcThreads = 256;
constexpr int kDcCtasPerSeq = 4;

struct DcParams {
    const uint4 *k, *v;               // [B, L_cap, H_kv, d] as 16-byte chunks
    uint4 *kc, *vc;                   // [B, H_kv, cap, d]
    const int32_t *len_valid, *len_old, *len_new, *origin, *base;
    int32_t *draft_len;
    int *err;
    int B, H_kv, L_cap, ring, cap, cpr;   // cpr = 16-byte chunks per row
};

__device__ __forceinline__ int dc_clamp(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }

// The copies of one sequence, as ranges of source positions:
//   r0 = [a0, a1): sinks (ring) or appended positions (linear), slot by layout;
//   r1 = [b0, b1): ring positions of the new window;
//   r2 = [c0, c1): ring slots to restore: slot(p) <- row p - ring.
struct DcRanges {
    int a0, a1, b0, b1, c0, c1, o, bs, draft_len;
};

__device__ __forceinline__ DcRanges dc_ranges(const DcParams &p, int b) {
    DcRanges r;
    const int lo = dc_clamp(checked(ld_dep(p.len_old + b), 0, p.L_cap, p.err), p.L_cap);
    const int ln = dc_clamp(checked(ld_dep(p.len_new + b), 0, p.L_cap, p.err), p.L_cap);
    const int lv = min(dc_clamp(checked(ld_dep(p.len_valid + b), 0, p.L_cap, p.err), p.L_cap), min(lo, ln));
    const int o = max(0, ld_dep(p.origin + b));
    r.o = o;
    if (p.ring > 0) {
        const int R = p.ring;
        r.bs = o;
        r.a0 = lv;
        r.a1 = max(lv, min(ln, o));
        r.b0 = max(max(lv, o), ln - R);
        r.b1 = max(r.b0, ln);
        r.c0 = max(ln, o + R);
        r.c1 = max(r.c0, min(lo, min(ln + R, lv + R)));
        r.draft_len = ln <= o ? ln : o + min(ln - o, R);
    } else {
        r.bs = max(0, ld_dep(p.base + b));
        r.a0 = max(lv, o);
        r.a1 = max(r.a0, ln);
        r.b0 = r.b1 = r.c0 = r.c1 = 0;
        r.draft_len = r.bs + max(0, ln - o);
    }
    return r;
}

__global__ void __launch_bounds__(kDcThreads) draft_cache_update_kernel(const DcParams p) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DcRanges r = dc_ranges(p, b);
    const int na = r.a1 - r.a0, nb = r.b1 - r.b0, nc = r.c1 - r.c0;
    const long long items = (long long)(na + nb + nc) * p.H_kv;
    const int stride = kDcCtasPerSeq * (kDcThreads / 32);
    for (long long it = (long long)blockIdx.y * (kDcThreads / 32) + warp; it < items; it += stride) {
        const int op = (int)(it / p.H_kv), h = (int)(it - (long long)op * p.H_kv);
        int src, slot;
        if (op < na) {
            src = r.a0 + op;
            slot = p.ring > 0 ? src : r.bs + (src - r.o);
        } else if (op < na + nb) {
            src = r.b0 + (op - na);
            slot = r.o + (src - r.o) % p.ring;
        } else {
            const int pos = r.c0 + (op - na - nb);
            src = pos - p.ring;
            slot = r.o + (pos - r.o) % p.ring;
        }
        if (slot >= p.cap) {
            if (lane == 0) raise_error(p.err, kErrCapacity);
            continue;
        }
        const long long from = (((long long)b * p.L_cap + src) * p.H_kv + h) * p.cpr;
        const long long to = (((long long)b * p.H_kv + h) * p.cap + slot) * p.cpr;
        if (lane < p.cpr) {
            p.kc[to + lane] = ld_dep_u4(p.k + from + lane);
        } else if (lane < 2 * p.cpr) {
            p.vc[to + lane - p.cpr] = ld_dep_u4(p.v + from + lane - p.cpr);
        }
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) p.draft_len[b] = min(r.draft_len, p.cap);
}

magicdec_status launch_draft_cache_update(int B, int H_kv, int D, int L_cap, const void *k, const void *v,
                                          const int32_t *len_valid, const int32_t *len_old, const int32_t *len_new,
                                          const int32_t *origin, const int32_t *base, int ring, int cap, void *kc,
                                          void *vc, int32_t *draft_len, cudaStream_t st) {
    DcParams p{};
    p.k = static_cast<const uint4 *>(k);
    p.v = static_cast<const uint4 *>(v);
    p.kc = static_cast<uint4 *>(kc);
    p.vc = static_cast<uint4 *>(vc);
    p.len_valid = len_valid;
    p.len_old = len_old;
    p.len_new = len_new;
    p.origin = origin;
    p.base = base;
    p.draft_len = draft_len;
    p.err = magicdec_host::device_error_word();
    p.B = B;
    p.H_kv = H_kv;
    p.L_cap = L_cap;
    p.ring = ring;
    p.cap = cap;
    p.cpr = D * 2 / 16;
    return magicdec_host::launch_pdl(draft_cache_update_kernel, dim3(B, kDcCtasPerSeq), dim3(kDcThreads), 0, st, p);
}

// ---------------------------------------------------------------- step lengths
// Per sequence: len = clamp(len_in + (n_acc ? n_acc + 1 : 0), 0, L_cap), then
// len_out = len and table[j][b] = min(len + j, L_cap) for j = 0 .. gamma+1:
// the lengths one speculative step's calls take (draft step g appends
// position len + g; verification sees len + gamma + 1).  len_out may alias
// len_in (each thread reads its element before writing it).
__global__ void step_lengths_kernel(int B, int gamma, int L_cap, const int32_t *len_in, const int32_t *n_acc,
                                    int32_t *len_out, int32_t *table) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    long long len = ld_dep(len_in + b);
    if (n_acc) len += (long long)ld_dep(n_acc + b) + 1;
    const int l = (int)(len < 0 ? 0 : (len > L_cap ? L_cap : len));
    len_out[b] = l;
    for (int j = 0; j <= gamma + 1; ++j) table[(long long)j * B + b] = min(l + j, L_cap);
}

magicdec_status launch_step_lengths(int B, int gamma, int L_cap, const int32_t *len_in, const int32_t *n_acc,
                                    int32_t *len_out, int32_t *table, cudaStream_t st) {
    const int threads = 256;
    return magicdec_host::launch_pdl(step_lengths_kernel, dim3((unsigned)((B + threads - 1) / threads)),
                                     dim3(threads), 0, st, B, gamma, L_cap, len_in, n_acc, len_out, table);
}

}  // namespace magicdec
