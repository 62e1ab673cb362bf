// noalloc.cu -- magicdec_verify_attn_noalloc: verification attention for
// callers that cannot allocate device memory.
//
// Some callers of this library are handed only their input and output
// buffers: a plug-in running inside another runtime's custom-operator
// interface, an engine whose memory plan is fixed before it starts, or a
// process whose device memory belongs entirely to a framework allocator.
// They cannot call cudaMalloc for the workspace that magicdec_verify_attn
// takes.  This entry point runs the same kernel with its scratch (the
// per-pair merge counters and the split partials) in a fixed-size array that
// lives in this file, so the call allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  Host
// code cannot use the array's name as a device address; the first call on a
// device (with that device current) resolves the address with
// cudaGetSymbolAddress, and later calls reuse the cached address.  Every
// call first clears the array's counter region with cudaMemsetAsync on the
// caller's stream (no allocation), so the kernel always starts from zeroed
// counters -- also after an earlier call that gave up on a bounded wait and
// left counters behind -- and the clear is ordered with the launch on that
// stream.  All calls on a device share the one array: calls that overlap on
// the GPU race and must be ordered (for example on one stream).
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace magicdec {
magicdec_status launch_decode_attn(int B, int H_q, int H_kv, int D, int L_cap, int n_q, int head_major,
                                   const void *q, const void *k, const void *v, const int32_t *len, void *out,
                                   void *ws, size_t ws_bytes, cudaStream_t st);
size_t attn_workspace_bytes_min(int B, int H_kv, int D, int M);
}  // namespace magicdec

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;   // 32 MiB

// The scratch itself (zero at module load).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDev] = {nullptr};

// Device address of the scratch array on the current device, resolved the
// first time the device is seen.
magicdec_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MAGICDEC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return MAGICDEC_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return MAGICDEC_OK;
}

}  // namespace

extern "C" magicdec_status magicdec_verify_attn_noalloc(magicdec_kv_shape shape, int n_q, const uint16_t *q,
                                                        const uint16_t *k, const uint16_t *v,
                                                        const int32_t *seq_len, uint16_t *out, void *stream) {
    if (!q || !k || !v || !seq_len || !out) return MAGICDEC_ERR_NULL;
    if (shape.B <= 0 || shape.H_q <= 0 || shape.H_kv <= 0 || shape.H_q % shape.H_kv != 0 ||
        (shape.d != 64 && shape.d != 128) || shape.L_cap <= 0 || shape.B > 4096 || n_q <= 0)
        return MAGICDEC_ERR_SHAPE;
    if ((shape.H_q / shape.H_kv) * n_q > 32) return MAGICDEC_ERR_UNSUPPORTED;
    if ((long long)shape.B * shape.H_kv > magicdec::kAttnMaxPairs) return MAGICDEC_ERR_UNSUPPORTED;
    if (!magicdec_host::aligned16(q) || !magicdec_host::aligned16(k) || !magicdec_host::aligned16(v) ||
        !magicdec_host::aligned16(out))
        return MAGICDEC_ERR_ALIGN;
    // The kernel runs without dynamic tails when their slots do not fit.
    const size_t need =
        magicdec::attn_workspace_bytes_min(shape.B, shape.H_kv, shape.d, (shape.H_q / shape.H_kv) * n_q);
    if (need > kNoAllocScratchBytes) return MAGICDEC_ERR_UNSUPPORTED;   // more SMs than the array covers
    void *ws = nullptr;
    const magicdec_status s = scratch_address(&ws);
    if (s != MAGICDEC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // merge counters and scheduler words start at zero whatever an earlier call left
    if (cudaMemsetAsync(ws, 0, magicdec::kAttnCounterBytes, st) != cudaSuccess) return MAGICDEC_ERR_CUDA;
    return magicdec::launch_decode_attn(shape.B, shape.H_q, shape.H_kv, shape.d, shape.L_cap, n_q, 0, q, k, v,
                                        seq_len, out, ws, kNoAllocScratchBytes, st);
}
