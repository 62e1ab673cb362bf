// api.cu -- the extern "C" boundary of libmagicdec: argument validation,
// workspace sizing and dispatch to the sm_103a kernels.  Declarations and the
// contract of every entry point are in include/magicdec.h.
#include <cudaTypedefs.h>

#include <climits>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace magicdec {
magicdec_status launch_decode_attn(int B, int H_q, int H_kv, int D, int L_cap, int n_q, int head_major,
                                   const void *q, const void *k, const void *v, const int32_t *len, void *out,
                                   void *ws, size_t ws_bytes, cudaStream_t st);
size_t attn_workspace_bytes(int B, int H_kv, int D, int M);
size_t topk_workspace_bytes(int B, int H_q, int L_cap);
magicdec_status launch_pq_encode(int B, int H_kv, int D, int L_cap, int C, const void *k, const float *codebook,
                                 uint8_t *codes, cudaStream_t st);
magicdec_status launch_pq_update(int B, int H_kv, int D, int L_cap, int C, const void *k, const int32_t *len,
                                 const uint8_t *codes, float *codebook, cudaStream_t st);
magicdec_status launch_pq_draft_attn(int B, int H_q, int H_kv, int D, int L_cap, int C, const void *q, const void *k,
                                     const void *v, const int32_t *len, const float *codebook, const uint8_t *codes,
                                     int top_k, void *out, int32_t *idx, void *ws, cudaStream_t st);
magicdec_status launch_draft_cache_update(int B, int H_kv, int D, int L_cap, const void *k, const void *v,
                                          const int32_t *len_valid, const int32_t *len_old, const int32_t *len_new,
                                          const int32_t *origin, const int32_t *base, int ring, int cap, void *kc,
                                          void *vc, int32_t *draft_len, cudaStream_t st);
magicdec_status launch_step_lengths(int B, int gamma, int L_cap, const int32_t *len_in, const int32_t *n_acc,
                                    int32_t *len_out, int32_t *table, cudaStream_t st);
magicdec_status launch_topk_draft_attn(int B, int H_q, int H_kv, int D, int L_cap, const void *q, const void *k,
                                       const void *v, const int32_t *len, int top_k, void *out, int32_t *idx,
                                       void *ws, cudaStream_t st);
magicdec_status launch_streaming_select(const int32_t *seq_len, int B, int H_kv, int n_sink, int n_recent,
                                        int32_t *idx, int32_t *n_sel, cudaStream_t st);
magicdec_status launch_gather_kv(int B, int H_kv, int D, int L_cap, const void *k, const void *v,
                                 const int32_t *idx, int n_idx, int cap, void *kc, void *vc, cudaStream_t st);
size_t snapkv_workspace_bytes(int B, int H_q, int H_kv, int D, int L_cap, int w);
magicdec_status launch_snapkv_select(int B, int H_q, int H_kv, int D, int L_cap, const void *q_win, const void *k,
                                     const int32_t *seq_len, int w, int pool, int budget, const int32_t *budgets,
                                     int32_t *idx, int32_t *n_sel, void *ws, cudaStream_t st);
size_t accept_workspace_bytes(int B, int gamma, int V);
magicdec_status launch_spec_accept(int B, int gamma, int V, const float *target, const float *draft,
                                   const int32_t *draft_tok, const float *u_acc, const float *u_res, int greedy,
                                   int32_t *n_acc, int32_t *out_tok, int32_t *n_amb, void *ws, cudaStream_t st);

// The library's device error word (one per device that loads the library).
__device__ int g_error_word;
}  // namespace magicdec

namespace magicdec_host {

constexpr int kMaxDevices = 64;

static int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

int sm_count() {
    static int cache[kMaxDevices] = {0};
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 1;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

int max_smem_optin() {
    static int cache[kMaxDevices] = {0};
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 48 * 1024;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cache[dev] = n > 0 ? n : 48 * 1024;
    }
    return cache[dev];
}

int *device_error_word() {
    static int *cache[kMaxDevices] = {nullptr};
    static std::mutex mu;
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, magicdec::g_error_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int *>(ptr);
    }
    return cache[dev];
}

bool encode_tmap_bf16_4d(CUtensorMap *map, const void *base, const uint64_t dims[4], const uint64_t strides[3],
                         const uint32_t box[4]) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!encode) return false;
    cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
    cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace magicdec_host

using magicdec_host::aligned16;

static bool shape_ok(const magicdec_kv_shape &s) {
    return s.B > 0 && s.H_q > 0 && s.H_kv > 0 && s.H_q % s.H_kv == 0 && (s.d == 64 || s.d == 128) &&
           s.L_cap > 0 && s.B <= 4096;
}

extern "C" {

const char *magicdec_status_string(int status) {
    switch (status) {
        case MAGICDEC_OK: return "ok";
        case MAGICDEC_ERR_NULL: return "null pointer";
        case MAGICDEC_ERR_SHAPE: return "invalid shape";
        case MAGICDEC_ERR_ALIGN: return "pointer not 16-byte aligned";
        case MAGICDEC_ERR_WORKSPACE: return "workspace too small";
        case MAGICDEC_ERR_UNSUPPORTED: return "unsupported shape";
        case MAGICDEC_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

magicdec_status magicdec_device_error(int32_t *out) {
    if (!out) return MAGICDEC_ERR_NULL;
    int *w = magicdec_host::device_error_word();
    if (!w) return MAGICDEC_ERR_CUDA;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return MAGICDEC_ERR_CUDA;
    if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MAGICDEC_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return MAGICDEC_ERR_CUDA;
    *out = v;
    return MAGICDEC_OK;
}

magicdec_status magicdec_streaming_select(const int32_t *seq_len, int B, int H_kv, int n_sink, int n_recent,
                                          int32_t *idx, int32_t *n_sel, void *stream) {
    if (!seq_len || !idx || !n_sel) return MAGICDEC_ERR_NULL;
    if (B <= 0 || H_kv <= 0 || n_sink < 0 || n_recent < 0) return MAGICDEC_ERR_SHAPE;
    const long long width = (long long)n_sink + n_recent;   // the row width of idx must be a positive int
    if (width <= 0 || width > INT_MAX) return MAGICDEC_ERR_SHAPE;
    return magicdec::launch_streaming_select(seq_len, B, H_kv, n_sink, n_recent, idx, n_sel,
                                             static_cast<cudaStream_t>(stream));
}

size_t magicdec_snapkv_workspace_size(magicdec_kv_shape shape, int window) {
    if (!shape_ok(shape) || window <= 0) return 0;
    return magicdec::snapkv_workspace_bytes(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, window);
}

static magicdec_status snapkv_common(const magicdec_kv_shape &shape, const uint16_t *q_win, const uint16_t *k,
                                     const int32_t *seq_len, int window, int pool_kernel, int budget,
                                     const int32_t *idx, const int32_t *n_sel, const void *ws, size_t ws_bytes) {
    if (!q_win || !k || !seq_len || !idx || !n_sel || !ws) return MAGICDEC_ERR_NULL;
    if (!shape_ok(shape) || window <= 0 || budget < window || pool_kernel <= 0 || (pool_kernel & 1) == 0)
        return MAGICDEC_ERR_SHAPE;
    if (pool_kernel > 9) return MAGICDEC_ERR_UNSUPPORTED;
    if ((long long)window * (shape.H_q / shape.H_kv) > 256) return MAGICDEC_ERR_UNSUPPORTED;
    if (!aligned16(q_win) || !aligned16(k) || !aligned16(ws)) return MAGICDEC_ERR_ALIGN;
    if (ws_bytes < magicdec_snapkv_workspace_size(shape, window)) return MAGICDEC_ERR_WORKSPACE;
    return MAGICDEC_OK;
}

magicdec_status magicdec_snapkv_select(magicdec_kv_shape shape, const uint16_t *q_win, const uint16_t *k,
                                       const int32_t *seq_len, int window, int pool_kernel, int budget,
                                       int32_t *idx, int32_t *n_sel, void *ws, size_t ws_bytes, void *stream) {
    magicdec_status s = snapkv_common(shape, q_win, k, seq_len, window, pool_kernel, budget, idx, n_sel, ws, ws_bytes);
    if (s != MAGICDEC_OK) return s;
    return magicdec::launch_snapkv_select(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, q_win, k, seq_len,
                                          window, pool_kernel, budget, nullptr, idx, n_sel, ws,
                                          static_cast<cudaStream_t>(stream));
}

magicdec_status magicdec_snapkv_select_budgets(magicdec_kv_shape shape, const uint16_t *q_win, const uint16_t *k,
                                               const int32_t *seq_len, int window, int pool_kernel,
                                               const int32_t *budgets, int max_budget, int32_t *idx, int32_t *n_sel,
                                               void *ws, size_t ws_bytes, void *stream) {
    if (!budgets) return MAGICDEC_ERR_NULL;
    magicdec_status s =
        snapkv_common(shape, q_win, k, seq_len, window, pool_kernel, max_budget, idx, n_sel, ws, ws_bytes);
    if (s != MAGICDEC_OK) return s;
    return magicdec::launch_snapkv_select(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, q_win, k, seq_len,
                                          window, pool_kernel, max_budget, budgets, idx, n_sel, ws,
                                          static_cast<cudaStream_t>(stream));
}

magicdec_status magicdec_gather_kv(magicdec_kv_shape shape, const uint16_t *k, const uint16_t *v,
                                   const int32_t *idx, int n_idx, int cap, uint16_t *kc, uint16_t *vc,
                                   void *stream) {
    if (!k || !v || !idx || !kc || !vc) return MAGICDEC_ERR_NULL;
    if (!shape_ok(shape) || n_idx < 0 || cap <= 0 || n_idx > cap) return MAGICDEC_ERR_SHAPE;
    if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(vc)) return MAGICDEC_ERR_ALIGN;
    return magicdec::launch_gather_kv(shape.B, shape.H_kv, shape.d, shape.L_cap, k, v, idx, n_idx, cap, kc, vc,
                                      static_cast<cudaStream_t>(stream));
}

size_t magicdec_attn_workspace_size(magicdec_kv_shape shape, int n_q) {
    if (!shape_ok(shape) || n_q <= 0) return 0;
    return magicdec::attn_workspace_bytes(shape.B, shape.H_kv, shape.d, (shape.H_q / shape.H_kv) * n_q);
}

static magicdec_status attn_common(const magicdec_kv_shape &shape, int n_q, const uint16_t *q, const uint16_t *k,
                                   const uint16_t *v, const int32_t *len, uint16_t *out, void *ws,
                                   size_t ws_bytes) {
    if (!q || !k || !v || !len || !out || !ws) return MAGICDEC_ERR_NULL;
    if (!shape_ok(shape) || n_q <= 0) return MAGICDEC_ERR_SHAPE;
    if ((shape.H_q / shape.H_kv) * n_q > 32) return MAGICDEC_ERR_UNSUPPORTED;
    if ((long long)shape.B * shape.H_kv > magicdec::kAttnMaxPairs) return MAGICDEC_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws))
        return MAGICDEC_ERR_ALIGN;
    if (ws_bytes < magicdec_attn_workspace_size(shape, n_q)) return MAGICDEC_ERR_WORKSPACE;
    return MAGICDEC_OK;
}

magicdec_status magicdec_draft_attn(magicdec_kv_shape shape, const uint16_t *q, const uint16_t *kc,
                                    const uint16_t *vc, const int32_t *draft_len, uint16_t *out, void *ws,
                                    size_t ws_bytes, void *stream) {
    magicdec_status s = attn_common(shape, 1, q, kc, vc, draft_len, out, ws, ws_bytes);
    if (s != MAGICDEC_OK) return s;
    return magicdec::launch_decode_attn(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, 1, 1, q, kc, vc,
                                        draft_len, out, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

magicdec_status magicdec_verify_attn(magicdec_kv_shape shape, int n_q, const uint16_t *q, const uint16_t *k,
                                     const uint16_t *v, const int32_t *seq_len, uint16_t *out, void *ws,
                                     size_t ws_bytes, void *stream) {
    magicdec_status s = attn_common(shape, n_q, q, k, v, seq_len, out, ws, ws_bytes);
    if (s != MAGICDEC_OK) return s;
    return magicdec::launch_decode_attn(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, n_q, 0, q, k, v,
                                        seq_len, out, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

magicdec_status magicdec_draft_cache_update(magicdec_kv_shape shape, const uint16_t *k, const uint16_t *v,
                                            const int32_t *len_valid, const int32_t *len_old, const int32_t *len_new,
                                            const int32_t *origin, const int32_t *base, int ring, int cap,
                                            uint16_t *kc, uint16_t *vc, int32_t *draft_len, void *stream) {
    if (!k || !v || !len_valid || !len_old || !len_new || !origin || !kc || !vc || !draft_len)
        return MAGICDEC_ERR_NULL;
    if (ring == 0 && !base) return MAGICDEC_ERR_NULL;
    if (!shape_ok(shape) || ring < 0 || cap <= 0 || ring > cap) return MAGICDEC_ERR_SHAPE;
    if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(vc)) return MAGICDEC_ERR_ALIGN;
    return magicdec::launch_draft_cache_update(shape.B, shape.H_kv, shape.d, shape.L_cap, k, v, len_valid, len_old,
                                               len_new, origin, base, ring, cap, kc, vc, draft_len,
                                               static_cast<cudaStream_t>(stream));
}

magicdec_status magicdec_step_lengths(int B, int gamma, int L_cap, const int32_t *len_in, const int32_t *n_acc,
                                      int32_t *len_out, int32_t *table, void *stream) {
    if (!len_in || !len_out || !table) return MAGICDEC_ERR_NULL;
    if (B <= 0 || gamma < 0 || L_cap <= 0 || gamma > 1024) return MAGICDEC_ERR_SHAPE;
    return magicdec::launch_step_lengths(B, gamma, L_cap, len_in, n_acc, len_out, table,
                                         static_cast<cudaStream_t>(stream));
}

static magicdec_status pq_common(const magicdec_kv_shape &shape, const void *k, int M, int C, const void *codebook,
                                 const void *codes) {
    if (!k || !codebook || !codes) return MAGICDEC_ERR_NULL;
    if (!shape_ok(shape) || M * 8 != shape.d || C < 1 || C > 256) return MAGICDEC_ERR_SHAPE;
    if (!aligned16(k) || !aligned16(codebook) || !aligned16(codes)) return MAGICDEC_ERR_ALIGN;
    return MAGICDEC_OK;
}

magicdec_status magicdec_pq_encode(magicdec_kv_shape shape, const uint16_t *k, int M, int C, const float *codebook,
                                   uint8_t *codes, void *stream) {
    magicdec_status s = pq_common(shape, k, M, C, codebook, codes);
    if (s != MAGICDEC_OK) return s;
    return magicdec::launch_pq_encode(shape.B, shape.H_kv, shape.d, shape.L_cap, C, k, codebook, codes,
                                      static_cast<cudaStream_t>(stream));
}

magicdec_status magicdec_pq_update(magicdec_kv_shape shape, const uint16_t *k, const int32_t *seq_len, int M, int C,
                                   const uint8_t *codes, float *codebook, void *stream) {
    if (!seq_len) return MAGICDEC_ERR_NULL;
    magicdec_status s = pq_common(shape, k, M, C, codebook, codes);
    if (s != MAGICDEC_OK) return s;
    return magicdec::launch_pq_update(shape.B, shape.H_kv, shape.d, shape.L_cap, C, k, seq_len, codes, codebook,
                                      static_cast<cudaStream_t>(stream));
}

size_t magicdec_pq_attn_workspace_size(magicdec_kv_shape shape) {
    if (!shape_ok(shape)) return 0;
    return magicdec::topk_workspace_bytes(shape.B, shape.H_q, shape.L_cap);
}

magicdec_status magicdec_pq_draft_attn(magicdec_kv_shape shape, const uint16_t *q, const uint16_t *k,
                                       const uint16_t *v, const int32_t *seq_len, int M, int C, const float *codebook,
                                       const uint8_t *codes, int top_k, uint16_t *out, int32_t *idx, void *ws,
                                       size_t ws_bytes, void *stream) {
    if (!q || !v || !seq_len || !out || !ws) return MAGICDEC_ERR_NULL;
    magicdec_status s = pq_common(shape, k, M, C, codebook, codes);
    if (s != MAGICDEC_OK) return s;
    if (top_k <= 0) return MAGICDEC_ERR_SHAPE;
    if (top_k > 8192) return MAGICDEC_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(v) || !aligned16(out) || !aligned16(ws)) return MAGICDEC_ERR_ALIGN;
    if (ws_bytes < magicdec_pq_attn_workspace_size(shape)) return MAGICDEC_ERR_WORKSPACE;
    return magicdec::launch_pq_draft_attn(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, C, q, k, v, seq_len,
                                          codebook, codes, top_k, out, idx, ws, static_cast<cudaStream_t>(stream));
}

size_t magicdec_topk_attn_workspace_size(magicdec_kv_shape shape) {
    if (!shape_ok(shape)) return 0;
    return magicdec::topk_workspace_bytes(shape.B, shape.H_q, shape.L_cap);
}

magicdec_status magicdec_topk_draft_attn(magicdec_kv_shape shape, const uint16_t *q, const uint16_t *k,
                                         const uint16_t *v, const int32_t *seq_len, int top_k, uint16_t *out,
                                         int32_t *idx, void *ws, size_t ws_bytes, void *stream) {
    if (!q || !k || !v || !seq_len || !out || !ws) return MAGICDEC_ERR_NULL;
    if (!shape_ok(shape) || top_k <= 0) return MAGICDEC_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws))
        return MAGICDEC_ERR_ALIGN;
    if (ws_bytes < magicdec_topk_attn_workspace_size(shape)) return MAGICDEC_ERR_WORKSPACE;
    return magicdec::launch_topk_draft_attn(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, q, k, v, seq_len,
                                            top_k, out, idx, ws, static_cast<cudaStream_t>(stream));
}

size_t magicdec_spec_accept_workspace_size(int B, int gamma, int V) {
    if (B <= 0 || gamma < 0 || V <= 0) return 0;
    return magicdec::accept_workspace_bytes(B, gamma, V);
}

magicdec_status magicdec_spec_accept(int B, int gamma, int V, const float *target_logits,
                                     const float *draft_logits, const int32_t *draft_tok, const float *u_acc,
                                     const float *u_res, int greedy, int32_t *n_acc, int32_t *out_tok,
                                     int32_t *n_ambiguous, void *ws, size_t ws_bytes, void *stream) {
    if (!target_logits || !n_acc || !out_tok || !ws) return MAGICDEC_ERR_NULL;
    if (gamma > 0 && !draft_tok) return MAGICDEC_ERR_NULL;
    if (!greedy && (!u_res || (gamma > 0 && (!draft_logits || !u_acc)))) return MAGICDEC_ERR_NULL;
    if (B <= 0 || gamma < 0 || V <= 0) return MAGICDEC_ERR_SHAPE;
    if (V > 256 * 4096 || B > magicdec::kAcceptMaxBatch || gamma > 32) return MAGICDEC_ERR_UNSUPPORTED;
    if (!aligned16(target_logits) || (draft_logits && !aligned16(draft_logits)) || !aligned16(ws))
        return MAGICDEC_ERR_ALIGN;
    if (ws_bytes < magicdec_spec_accept_workspace_size(B, gamma, V)) return MAGICDEC_ERR_WORKSPACE;
    return magicdec::launch_spec_accept(B, gamma, V, target_logits, draft_logits, draft_tok, u_acc, u_res, greedy,
                                        n_acc, out_tok, n_ambiguous, ws, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
