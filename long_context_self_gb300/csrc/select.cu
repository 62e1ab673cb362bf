// select.cu -- draft-KV selection and gather for MagicDec self-speculation,
// sm_103a.
//
//  * StreamingLLM selection (paper section 4.4 / section 5.1): attention sinks
//    plus a recent window; pure index arithmetic.
//  * SnapKV selection (paper section 4.4 / section 5.2), once after prefill:
//    the observation-window scores come from the two tcgen05 passes in
//    snapkv_tc.cu; here
//      top-k   one CTA per (sequence, KV head): max-pool (kernel k, clipped),
//              an 8-bit-digit MSB-first radix select of the k-th largest
//              pooled score, then an order-preserving block compaction that
//              keeps everything above the threshold and the smallest
//              positions among ties; the window is appended.
//  * Gather of the selected rows into the compact cache (section 4.4): 16-byte vector
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
// A warp moves rows: each lane owns one 16-byte chunk of K or V of a row
// (2*CPR lanes per row), and each iteration moves RPI rows per row slot so
// that RPI loads per lane are in flight.  The row -> (sequence, head, slot)
// decode is done once per row by one lane and broadcast.
template <int CPR, int RPI>
__global__ void __launch_bounds__(256) gather_kv_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                       const int32_t *__restrict__ idx, int H_kv, int L_cap,
                                                       int n_idx, int cap, int rows, uint4 *__restrict__ kc,
                                                       uint4 *__restrict__ vc) {
    constexpr int LPR = 2 * CPR;                 // lanes per row (K and V)
    constexpr int SLOTS = 32 / LPR;              // rows side by side in a warp
    constexpr int RPW = SLOTS * RPI;             // rows per warp per iteration
    static_assert(RPW <= 32, "one decoding lane per row");
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int slot = lane / LPR, sub = lane % LPR;
    const int kv = sub / CPR, ch = sub % CPR;
    const long long warp0 = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long base = warp0 * RPW; base < rows; base += nwarps * RPW) {
        // lane j < RPW decodes row base + j
        long long src_off = -1, dst_off = -1;
        {
            const long long row = base + lane;
            if (lane < RPW && row < rows) {
                const int bh = (int)(row / n_idx);
                const int i = (int)(row - (long long)bh * n_idx);
                const int h = bh % H_kv, b = bh / H_kv;
                const int pos = __ldg(idx + row);
                dst_off = ((long long)bh * cap + i) * CPR;
                if (pos >= 0 && pos < L_cap) src_off = (((long long)b * L_cap + pos) * H_kv + h) * CPR;
            }
        }
        uint4 val[RPI];
        long long dsto[RPI];
#pragma unroll
        for (int r = 0; r < RPI; ++r) {
            const int j = r * SLOTS + slot;
            const long long so = __shfl_sync(0xffffffffu, src_off, j);
            dsto[r] = __shfl_sync(0xffffffffu, dst_off, j);
            val[r] = make_uint4(0, 0, 0, 0);
            if (dsto[r] >= 0 && so >= 0) {
                const uint4 *src = (kv ? v : k) + so + ch;
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(val[r].x), "=r"(val[r].y), "=r"(val[r].z), "=r"(val[r].w)
                             : "l"(src));
            }
        }
#pragma unroll
        for (int r = 0; r < RPI; ++r)
            if (dsto[r] >= 0) (kv ? vc : kc)[dsto[r] + ch] = val[r];
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
    const long long rows = (long long)B * H_kv * n_idx;
    if (rows >= (1ll << 31)) return MAGICDEC_ERR_UNSUPPORTED;
    const int threads = 256;
    const long long want = (rows + 8 * 8 - 1) / (8 * 8);                // 8 warps x 8 rows per CTA iteration
    const int blocks = (int)std::max<long long>(1, std::min<long long>(want, (long long)magicdec_host::sm_count() * 8));
    const uint4 *k4 = static_cast<const uint4 *>(k), *v4 = static_cast<const uint4 *>(v);
    uint4 *kc4 = static_cast<uint4 *>(kc), *vc4 = static_cast<uint4 *>(vc);
    if (D == 128)
        return magicdec_host::launch_pdl(gather_kv_kernel<16, 8>, dim3(blocks), dim3(threads), 0, st, k4, v4, idx,
                                         H_kv, L_cap, n_idx, cap, (int)rows, kc4, vc4);
    return magicdec_host::launch_pdl(gather_kv_kernel<8, 4>, dim3(blocks), dim3(threads), 0, st, k4, v4, idx, H_kv,
                                     L_cap, n_idx, cap, (int)rows, kc4, vc4);
}

size_t snapkv_tc_workspace_bytes(int B, int H_q, int H_kv, int L_cap, int w);
magicdec_status launch_snapkv_scores_tc(int B, int H_q, int H_kv, int D, int L_cap, const void *q_win, const void *k,
                                        const int32_t *seq_len, int w, void *ws, float **score_out, cudaStream_t st);

// Workspace: [pass-1 partials][scores B x H_kv x L_cap fp32][pooled keys B x H_kv x L_cap u32]
size_t snapkv_workspace_bytes(int B, int H_q, int H_kv, int D, int L_cap, int w) {
    (void)D;
    return snapkv_tc_workspace_bytes(B, H_q, H_kv, L_cap, w);
}

magicdec_status launch_snapkv_select(int B, int H_q, int H_kv, int D, int L_cap, const void *q_win, const void *k,
                                     const int32_t *seq_len, int w, int pool, int budget, int32_t *idx,
                                     int32_t *n_sel, void *ws, cudaStream_t st) {
    float *score = nullptr;
    magicdec_status s = launch_snapkv_scores_tc(B, H_q, H_kv, D, L_cap, q_win, k, seq_len, w, ws, &score, st);
    if (s != MAGICDEC_OK) return s;
    uint32_t *keys = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(score) +
                                                  (((size_t)B * H_kv * L_cap * 4 + 255) & ~(size_t)255));
    return magicdec_host::launch_pdl(snapkv_topk_kernel, dim3(H_kv, B), dim3(1024), 0, st,
                                     static_cast<const float *>(score), keys, seq_len, H_kv, L_cap, w, pool, budget,
                                     idx, n_sel);
}

}  // namespace magicdec
