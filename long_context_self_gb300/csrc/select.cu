// select.cu -- draft-KV selection and gather for MagicDec self-speculation,
// sm_103a.
//
//  * StreamingLLM selection (paper section 4.4 / section 5.1): attention sinks
//    plus a recent window; pure index arithmetic.
//  * SnapKV selection (paper section 4.4 / section 5.2), once after prefill:
//    the observation-window scores come from the two tcgen05 passes in
//    snapkv_tc.cu; here the prefix scores are max-pooled (kernel k, clipped),
//    and the select kernel of topk.cu (selection-only mode) keeps the
//    budget - window largest pooled positions (ties: the smaller position)
//    in ascending order and appends the window.
//  * Gather of the selected rows into the compact cache (section 4.4): 16-byte vector
//    row copies into the head-major compact draft cache.
#include <algorithm>

#include "common.cuh"

namespace magicdec {

__device__ __forceinline__ int clamp_len_s(int v, int hi) { return v < 0 ? 0 : (v > hi ? hi : v); }

// ------------------------------------------------------------ StreamingLLM
__global__ void streaming_select_kernel(const int32_t *seq_len, int H_kv, int n_sink, int n_recent, int32_t *idx,
                                        int32_t *n_sel) {
    // grid (index tiles, KV head, sequence): no index arithmetic beyond the tile
    pdl_trigger();
    pdl_wait();
    // 64-bit: the width may come within a block of INT_MAX
    const long long width = (long long)n_sink + n_recent;
    const long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int len = max(ld_dep(seq_len + b), 0);
    const int sinks = min(n_sink, len);
    const int rec0 = max(n_sink, len - n_recent);
    const int n = sinks + max(0, len - rec0);
    if (j < width) {
        int v = -1;
        if (j < sinks) v = (int)j;
        else if (j < n) v = rec0 + (int)(j - sinks);
        idx[((long long)b * H_kv + h) * width + j] = v;
    }
    if (j == 0 && h == 0) n_sel[b] = n;
}

// ------------------------------------------------------------------ gather
// A warp moves rows: each lane owns one 16-byte chunk of K or V of a row
// (2*CPR lanes per row), and each iteration moves RPI rows per row slot so
// that RPI loads per lane are in flight.  The row -> (sequence, head, slot)
// decode is done once per row by one lane and broadcast.
template <int CPR, int RPI>
__global__ void __launch_bounds__(256) gather_kv_kernel(const uint4 *k, const uint4 *v,
                                                       const int32_t *idx, int H_kv, int L_cap,
                                                       int n_idx, int cap, int rows, uint4 *__restrict__ kc,
                                                       uint4 *__restrict__ vc, int *err) {
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
                // rows < 2^31 (checked at launch): 32-bit divisions
                const int r32 = (int)row;
                const int bh = r32 / n_idx;
                const int i = r32 - bh * n_idx;
                const int h = bh % H_kv, b = bh / H_kv;
                // -1 marks padding; any other index outside [0, L_cap) is a
                // caller error, gathered as a zero row (recorded in the debug build)
                const int pos = ld_dep(idx + row);
                if (pos != -1) checked(pos, 0, L_cap - 1, err);
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

// ------------------------------------------------------------------ pooling
// pooled[j] = max of the prefix scores in [j - half, j + half] clipped to
// [0, m), m = len - w (half <= 4); row stride L_sc (a multiple of 4 floats).
// A thread pools 4 consecutive positions 4t..4t+3 from the three aligned
// float4 groups around them.
__global__ void __launch_bounds__(256) snapkv_pool_kernel(const float *score,
                                                         const int32_t *seq_len, int H_kv, int L_cap,
                                                         int L_sc, int w, int half, float *__restrict__ pooled) {
    pdl_trigger();
    pdl_wait();
    const int h = blockIdx.y, b = blockIdx.z;
    const int m = clamp_len_s(ld_dep(seq_len + b), L_cap) - w;
    const float *sc = score + ((long long)b * H_kv + h) * L_cap;
    float *out = pooled + ((long long)b * H_kv + h) * L_sc;
    for (int g = blockIdx.x * blockDim.x + threadIdx.x; 4 * g < m; g += gridDim.x * blockDim.x) {
        const int j0 = 4 * g;
        float x[12];                                  // positions j0-4 .. j0+7, -inf outside [0, m)
#pragma unroll
        for (int e = 0; e < 12; ++e) {
            const int t = j0 - 4 + e;
            x[e] = (t >= 0 && t < m) ? ld_dep_f(sc + t) : -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (j0 + e >= m) break;
            float mx = -INFINITY;
#pragma unroll
            for (int o = -4; o <= 4; ++o)
                if (o >= -half && o <= half) mx = fmaxf(mx, x[4 + e + o]);
            out[j0 + e] = mx;
        }
    }
}

// ------------------------------------------------------------------- host side
magicdec_status launch_streaming_select(const int32_t *seq_len, int B, int H_kv, int n_sink, int n_recent,
                                        int32_t *idx, int32_t *n_sel, cudaStream_t st) {
    const long long width = (long long)n_sink + n_recent;
    if (B <= 0 || H_kv <= 0 || width <= 0) return MAGICDEC_OK;
    if (B > 65535 || H_kv > 65535) return MAGICDEC_ERR_UNSUPPORTED;
    const int threads = 256;
    const dim3 grid((unsigned)((width + threads - 1) / threads), H_kv, B);
    return magicdec_host::launch_pdl(streaming_select_kernel, grid, dim3(threads), 0, st, seq_len, H_kv, n_sink,
                                     n_recent, idx, n_sel);
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
                                         H_kv, L_cap, n_idx, cap, (int)rows, kc4, vc4,
                                         magicdec_host::device_error_word());
    return magicdec_host::launch_pdl(gather_kv_kernel<8, 4>, dim3(blocks), dim3(threads), 0, st, k4, v4, idx, H_kv,
                                     L_cap, n_idx, cap, (int)rows, kc4, vc4, magicdec_host::device_error_word());
}

size_t snapkv_tc_workspace_bytes(int B, int H_q, int H_kv, int L_cap, int w);
magicdec_status launch_snapkv_scores_tc(int B, int H_q, int H_kv, int D, int L_cap, const void *q_win, const void *k,
                                        const int32_t *seq_len, int w, void *ws, float **score_out, cudaStream_t st);

// Workspace: [pass-1 partials][scores B x H_kv x L_cap fp32][pooled B x H_kv x L_sc fp32]
size_t snapkv_workspace_bytes(int B, int H_q, int H_kv, int D, int L_cap, int w) {
    (void)D;
    return snapkv_tc_workspace_bytes(B, H_q, H_kv, L_cap, w);
}

magicdec_status launch_snapkv_pick(int B, int H_kv, int L_cap, const float *pooled, const int32_t *len, int window,
                                   int budget, const int32_t *budgets, int32_t *idx, int32_t *n_sel, cudaStream_t st);

magicdec_status launch_snapkv_select(int B, int H_q, int H_kv, int D, int L_cap, const void *q_win, const void *k,
                                     const int32_t *seq_len, int w, int pool, int budget, const int32_t *budgets,
                                     int32_t *idx, int32_t *n_sel, void *ws, cudaStream_t st) {
    if (pool / 2 > 4) return MAGICDEC_ERR_UNSUPPORTED;   // before anything is launched
    float *score = nullptr;
    magicdec_status s = launch_snapkv_scores_tc(B, H_q, H_kv, D, L_cap, q_win, k, seq_len, w, ws, &score, st);
    if (s != MAGICDEC_OK) return s;
    const int L_sc = (L_cap + 3) & ~3;
    float *pooled = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(score) +
                                              (((size_t)B * H_kv * L_cap * 4 + 255) & ~(size_t)255));
    const int per = 256 * 4 * 4;                      // positions per CTA: 4 per thread, 4 grid-stride steps
    s = magicdec_host::launch_pdl(snapkv_pool_kernel, dim3((L_cap + per - 1) / per, H_kv, B), dim3(256), 0, st,
                                  static_cast<const float *>(score), seq_len, H_kv, L_cap, L_sc, w, pool / 2, pooled);
    if (s != MAGICDEC_OK) return s;
    return launch_snapkv_pick(B, H_kv, L_cap, pooled, seq_len, w, budget, budgets, idx, n_sel, st);
}

}  // namespace magicdec
