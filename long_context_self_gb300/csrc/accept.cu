// accept.cu -- speculative-sampling accept / resample (Leviathan et al., the
// rule behind Eq. 1 of the MagicDec paper, section 3.1) and greedy
// verification (paper section 5.1), sm_103a.
//
// The step streams the target logits [B, gamma+1, V] and draft logits
// [B, gamma, V] once (fp32, HBM-bound) and then touches one row pair per
// sequence again for the resample.  Three launches:
//   stats  per (row, 16K-logit chunk): chunk max, sum of exp(x - max) in
//          double-float (an fp32 pair, ~48-bit significand), top-1 (smallest
//          index among equals) and top-2 logits;
//   chain  one thread per sequence: merge the chunk stats of its rows in
//          fp64, evaluate p(x)/q(x) for each draft token in fp64, run the
//          sequential accept chain (or the greedy argmax chain) and record the
//          row to resample from;
//   sample per (sequence, chunk): the chunk's sum of resample weights
//          max(0, p - q) (or p for the bonus token), normalised in
//          double-float; the last CTA of a sequence (atomic counter, no
//          waiting) locates the chunk where the running sum crosses
//          u * total and scans inside it in a fixed order.
// Only the per-logit exponentials are single precision (random ~1e-6 relative
// errors that average out in the sums); normalisers, ratios and running sums
// carry ~1e-12 relative error, so the drawn token agrees with an exact
// evaluation except when u * total falls within ~1e-9 of a token boundary.
#include "common.cuh"

namespace magicdec {

constexpr int kAccChunk = 16384;      // logits per stats / sample CTA
constexpr int kAccThreads = 256;
constexpr int kAccPer = kAccChunk / kAccThreads;   // 64 logits per thread

// ------------------------------------------------------------ double-float
struct dflt {
    float hi, lo;
};

__device__ __forceinline__ dflt quick_two_sum(float a, float b) {
    const float s = a + b;
    return {s, b - (s - a)};
}

__device__ __forceinline__ dflt two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}

__device__ __forceinline__ dflt df_add_f(dflt a, float b) {
    dflt s = two_sum(a.hi, b);
    s.lo += a.lo;
    return quick_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ dflt df_sub(dflt a, dflt b) {
    dflt s = two_sum(a.hi, -b.hi);
    s.lo += a.lo - b.lo;
    return quick_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ dflt df_add(dflt a, dflt b) {
    dflt s = two_sum(a.hi, b.hi);
    s.lo += a.lo + b.lo;
    return quick_two_sum(s.hi, s.lo);
}

// float x double-float -> double-float
__device__ __forceinline__ dflt df_mul_f(float a, dflt b) {
    const float p = a * b.hi;
    const float e = fmaf(a, b.hi, -p) + a * b.lo;
    return quick_two_sum(p, e);
}

__device__ __forceinline__ dflt df_from_double(double x) {
    const float hi = (float)x;
    return {hi, (float)(x - (double)hi)};
}

__device__ __forceinline__ double df_to_double(dflt a) { return (double)a.hi + (double)a.lo; }

// ------------------------------------------------------------------- stats
struct RowStat {
    double s;          // sum over the chunk of exp(x - m)
    float m;           // chunk max
    float top1, top2;
    int arg;
};

struct JobInfo {
    double st, sd;     // target / draft normalisers relative to mt / md
    float mt, md;
    int kind;          // 0 = nothing to sample, 1 = residual at row acc, 2 = bonus from target row gamma
    int acc;
    int amb;
    int pad;
};

struct AcceptParams {
    const float *target;      // [B, gamma+1, V]
    const float *draft;       // [B, gamma, V]
    const int32_t *draft_tok;
    const float *u_acc;
    const float *u_res;
    int32_t *n_acc;
    int32_t *out_tok;
    int32_t *n_amb;
    RowStat *stats;           // [B, rows_per_b, n_chunks]
    JobInfo *job;             // [B]
    double *chunk_sum;        // [B, n_chunks]
    int *counters;            // [B], zero between calls
    int *err;
    int B, gamma, V, n_chunks, rows_per_b, greedy;
};

// Row r of sequence b: r <= gamma -> target row r; else draft row r-gamma-1.
__device__ __forceinline__ const float *row_ptr(const AcceptParams &p, int b, int r) {
    if (r <= p.gamma) return p.target + ((long long)b * (p.gamma + 1) + r) * p.V;
    return p.draft + ((long long)b * p.gamma + (r - p.gamma - 1)) * p.V;
}

__device__ __forceinline__ void top_merge(float &t1, float &t2, int &arg, float u1, float u2, int uarg) {
    float lose;
    if (u1 > t1 || (u1 == t1 && uarg < arg)) {
        lose = t1;
        t1 = u1;
        arg = uarg;
    } else {
        lose = u1;
    }
    t2 = fmaxf(fmaxf(t2, u2), lose);
}

__global__ void __launch_bounds__(kAccThreads) accept_stats_kernel(const AcceptParams p) {
    __shared__ float red_f[kAccThreads / 32][3];
    __shared__ int red_i[kAccThreads / 32];
    __shared__ double red_d[kAccThreads / 32];
    __shared__ float chunk_max;
    const int chunk = blockIdx.x, row = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const int b = row / p.rows_per_b, r = row % p.rows_per_b;
    const float *x = row_ptr(p, b, r);
    const int t0 = chunk * kAccChunk, t1 = min(t0 + kAccChunk, p.V);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float v[kAccPer];
    const bool vec = ((p.V & 3) == 0) && (t1 - t0 == kAccChunk);
    if (vec) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x + t0);
#pragma unroll
        for (int k = 0; k < kAccPer / 4; ++k) {
            float4 q;
            asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(q.x), "=f"(q.y), "=f"(q.z), "=f"(q.w)
                         : "l"(x4 + k * kAccThreads + tid));
            v[4 * k] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kAccPer; ++k) {
            const int t = t0 + k * kAccThreads + tid;
            v[k] = t < t1 ? __ldg(x + t) : -INFINITY;
        }
    }
    // index of v[k]: vec -> t0 + 4*(k/4*256 + tid) + k%4; else t0 + k*256 + tid (both increasing in k)
    float mx = -INFINITY, top1 = -INFINITY, top2 = -INFINITY;
    int arg = 0x7fffffff;
#pragma unroll
    for (int k = 0; k < kAccPer; ++k) {
        const float e = v[k];
        mx = fmaxf(mx, e);
        if (e > top1) {
            top2 = top1;
            top1 = e;
            arg = vec ? t0 + 4 * ((k >> 2) * kAccThreads + tid) + (k & 3) : t0 + k * kAccThreads + tid;
        } else if (e > top2) {
            top2 = e;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u1 = __shfl_xor_sync(0xffffffffu, top1, o);
        const float u2 = __shfl_xor_sync(0xffffffffu, top2, o);
        const int ua = __shfl_xor_sync(0xffffffffu, arg, o);
        top_merge(top1, top2, arg, u1, u2, ua);
    }
    mx = warp_max(mx);
    if (lane == 0) {
        red_f[warp][0] = mx;
        red_f[warp][1] = top1;
        red_f[warp][2] = top2;
        red_i[warp] = arg;
    }
    __syncthreads();
    if (tid == 0) {
        float m = red_f[0][0], a1 = red_f[0][1], a2 = red_f[0][2];
        int aa = red_i[0];
        for (int w = 1; w < kAccThreads / 32; ++w) {
            m = fmaxf(m, red_f[w][0]);
            top_merge(a1, a2, aa, red_f[w][1], red_f[w][2], red_i[w]);
        }
        chunk_max = m;
        red_f[0][1] = a1;
        red_f[0][2] = a2;
        red_i[0] = aa;
    }
    __syncthreads();
    const float m = chunk_max;
    dflt acc = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kAccPer; ++k) acc = df_add_f(acc, fast_exp2((v[k] - m) * kLog2e));
    double s = df_to_double(acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red_d[warp] = s;
    __syncthreads();
    if (tid == 0) {
        double tot = 0.0;
        for (int w = 0; w < kAccThreads / 32; ++w) tot += red_d[w];
        RowStat st;
        st.s = tot;
        st.m = m;
        st.top1 = red_f[0][1];
        st.top2 = red_f[0][2];
        st.arg = red_i[0];
        p.stats[((long long)b * p.rows_per_b + r) * p.n_chunks + chunk] = st;
    }
}

// Whole-row statistics, merged in fp64: max m and S = sum exp(x - m).
struct RowAll {
    double s;
    float m, top1, top2;
    int arg;
};

__device__ RowAll row_stat(const AcceptParams &p, int b, int r) {
    const RowStat *src = p.stats + ((long long)b * p.rows_per_b + r) * p.n_chunks;
    RowAll a{0.0, -INFINITY, -INFINITY, -INFINITY, 0x7fffffff};
    for (int c = 0; c < p.n_chunks; ++c) a.m = fmaxf(a.m, src[c].m);
    for (int c = 0; c < p.n_chunks; ++c) {
        const RowStat st = src[c];
        if (st.m != -INFINITY) a.s += st.s * exp((double)st.m - (double)a.m);
        top_merge(a.top1, a.top2, a.arg, st.top1, st.top2, st.arg);
    }
    return a;
}

// One thread per sequence (the chain is sequential; each step touches a few
// chunk records and two logits).
__global__ void accept_chain_kernel(const AcceptParams p) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    const int gamma = p.gamma, V = p.V;
    int32_t *out = p.out_tok + (long long)b * (gamma + 1);
    JobInfo job{};
    int amb = 0, acc = gamma, emit = -1;
    for (int i = 0; i < gamma; ++i) {
        const RowAll ts = row_stat(p, b, i);
        const int x = __ldg(p.draft_tok + (long long)b * gamma + i);
        bool ok;
        if (p.greedy) {
            if ((double)ts.top1 - (double)ts.top2 < 1e-4) ++amb;
            ok = (x == ts.arg);
            if (!ok) emit = ts.arg;
        } else {
            const RowAll ds = row_stat(p, b, gamma + 1 + i);
            if (x < 0 || x >= V) {
                ok = false;
            } else {
                const double tx = __ldg(row_ptr(p, b, i) + x);
                const double dx = __ldg(row_ptr(p, b, gamma + 1 + i) + x);
                const double px = exp(tx - (double)ts.m) / ts.s;
                const double qx = exp(dx - (double)ds.m) / ds.s;
                if (qx > 0.0) {
                    const double ratio = px / qx;
                    const double u = __ldg(p.u_acc + (long long)b * gamma + i);
                    ok = u < ratio;
                    if (fabs(u - ratio) < 1e-4) ++amb;
                } else {
                    ok = px > 0.0;
                }
            }
            if (!ok) {
                job.kind = 1;
                job.mt = ts.m; job.st = ts.s;
                job.md = ds.m; job.sd = ds.s;
            }
        }
        if (!ok) { acc = i; break; }
        out[i] = x;
    }
    if (acc == gamma) {
        const RowAll ts = row_stat(p, b, gamma);
        if (p.greedy) {
            if ((double)ts.top1 - (double)ts.top2 < 1e-4) ++amb;
            emit = ts.arg;
        } else {
            job.kind = 2;
            job.mt = ts.m; job.st = ts.s;
        }
    }
    for (int i = acc + 1; i <= gamma; ++i) out[i] = -1;
    p.n_acc[b] = acc;
    if (p.greedy) {
        out[acc] = emit;
        if (p.n_amb) p.n_amb[b] = amb;
    }
    job.acc = acc;
    job.amb = amb;
    p.job[b] = job;
}

// Resample weight of logit index t in double-float.
struct WeightCtx {
    const float *tr, *dr;
    float mt, md;
    dflt inv_st, inv_sd;
    int kind;
    bool use_p;
};

__device__ __forceinline__ dflt weight_at(const WeightCtx &w, int t) {
    const dflt pt = df_mul_f(fast_exp2((__ldg(w.tr + t) - w.mt) * kLog2e), w.inv_st);
    if (w.kind == 2 || w.use_p) return pt;
    const dflt qt = df_mul_f(fast_exp2((__ldg(w.dr + t) - w.md) * kLog2e), w.inv_sd);
    const dflt d = df_sub(pt, qt);
    return d.hi > 0.f ? d : dflt{0.f, 0.f};
}

__device__ double block_sum_d(double v, double *scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    double t = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += scratch[w];
    return t;
}

// Sum of weights over [t0, t1) (thread-strided double-float, then fp64 tree).
__device__ double chunk_weight_sum(const WeightCtx &w, int t0, int t1, double *scratch) {
    dflt acc = {0.f, 0.f};
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) acc = df_add(acc, weight_at(w, t));
    return block_sum_d(df_to_double(acc), scratch);
}

__global__ void __launch_bounds__(kAccThreads) accept_sample_kernel(const AcceptParams p) {
    __shared__ double scratch[kAccThreads / 32];
    __shared__ double seg[kAccThreads];
    __shared__ int is_last;
    const int chunk = blockIdx.x, b = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const JobInfo job = p.job[b];
    if (job.kind == 0) return;
    WeightCtx w;
    w.kind = job.kind;
    w.use_p = false;
    w.tr = row_ptr(p, b, job.kind == 2 ? p.gamma : job.acc);
    w.dr = job.kind == 1 ? row_ptr(p, b, p.gamma + 1 + job.acc) : nullptr;
    w.mt = job.mt;
    w.md = job.md;
    w.inv_st = df_from_double(1.0 / job.st);
    w.inv_sd = df_from_double(job.kind == 1 ? 1.0 / job.sd : 0.0);
    const int t0 = chunk * kAccChunk, t1 = min(t0 + kAccChunk, p.V);
    const double csum = chunk_weight_sum(w, t0, t1, scratch);
    if (threadIdx.x == 0) {
        p.chunk_sum[(long long)b * p.n_chunks + chunk] = csum;
        __threadfence();
        const int old = atomicAdd(p.counters + b, 1);
        is_last = (old == p.n_chunks - 1);
        if (is_last) {
            __threadfence();
            p.counters[b] = 0;
        }
    }
    __syncthreads();
    if (!is_last) return;

    // Last CTA of this sequence: find the token.
    __threadfence();
    const double u = __ldg(p.u_res + b);
    const double *cs = p.chunk_sum + (long long)b * p.n_chunks;
    double W = 0.0;
    for (int c = 0; c < p.n_chunks; ++c) W += __ldcg(cs + c);
    bool use_p = false;
    if (!(W > 0.0)) {
        // Residual empty (p == q up to rounding): draw from p instead; the
        // chunk sums of p are recomputed here into seg[] (n_chunks <= 256).
        use_p = true;
        w.use_p = true;
        W = 0.0;
        for (int c = 0; c < p.n_chunks; ++c) {
            const double v = chunk_weight_sum(w, c * kAccChunk, min((c + 1) * kAccChunk, p.V), scratch);
            if (threadIdx.x == 0) seg[c] = v;
            W += v;
        }
        __syncthreads();
    }
    const double target = u * W, tol = 1e-7 * W;
    double before = 0.0;
    int cstar = -1;
    for (int c = 0; c < p.n_chunks; ++c) {
        const double v = use_p ? seg[c] : __ldcg(cs + c);
        if (before + v > target) { cstar = c; break; }
        before += v;
    }
    int amb = job.amb;
    if (cstar < 0) {
        // rounding pushed target past the total: the last chunk with weight
        before = 0.0;
        for (int c = 0; c < p.n_chunks; ++c) {
            const double v = use_p ? seg[c] : __ldcg(cs + c);
            if (v > 0.0) cstar = c;
        }
        if (cstar < 0) cstar = p.n_chunks - 1;
        for (int c = 0; c < cstar; ++c) before += use_p ? seg[c] : __ldcg(cs + c);
        ++amb;
    }
    __syncthreads();   // every thread has read seg[] for the chunk search
    // Scan inside chunk cstar: each thread owns a contiguous run of logits.
    const int c0 = cstar * kAccChunk, c1 = min(c0 + kAccChunk, p.V);
    const int per = (c1 - c0 + kAccThreads - 1) / kAccThreads;
    const int my0 = c0 + threadIdx.x * per, my1 = min(my0 + per, c1);
    dflt mine = {0.f, 0.f};
    for (int t = my0; t < my1; ++t) mine = df_add(mine, weight_at(w, t));
    seg[threadIdx.x] = df_to_double(mine);
    __syncthreads();
    if (threadIdx.x == 0) {
        double run = before;
        int owner = -1;
        for (int i = 0; i < kAccThreads; ++i) {
            if (run + seg[i] > target) { owner = i; break; }
            run += seg[i];
        }
        int token = -1;
        if (owner >= 0) {
            const int s0 = c0 + owner * per, s1 = min(s0 + per, c1);
            double prev = run;
            for (int t = s0; t < s1; ++t) {
                const double nxt = prev + df_to_double(weight_at(w, t));
                if (nxt > target) {
                    token = t;
                    if ((t > 0 && target - prev < tol) || (t < p.V - 1 && nxt - target < tol)) ++amb;
                    break;
                }
                prev = nxt;
            }
        }
        if (token < 0) {
            // rounding: the last logit with positive weight in the chunk
            for (int t = c1 - 1; t >= c0; --t)
                if (weight_at(w, t).hi > 0.f) { token = t; break; }
            if (token < 0) token = c1 - 1;
            ++amb;
        }
        p.out_tok[(long long)b * (p.gamma + 1) + job.acc] = token;
        if (p.n_amb) p.n_amb[b] = amb;
    }
}

// ------------------------------------------------------------------- host side
static size_t align256a(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout: [counters: kAcceptMaxBatch int32, always left zero]
//                   [row stats][per-sequence job][per-chunk weight sums]
size_t accept_workspace_bytes(int B, int gamma, int V) {
    const int n_chunks = (V + kAccChunk - 1) / kAccChunk;
    const int rows = 2 * gamma + 1;
    return (size_t)kAcceptMaxBatch * 4 + align256a((size_t)B * rows * n_chunks * sizeof(RowStat)) +
           align256a((size_t)B * sizeof(JobInfo)) + align256a((size_t)B * n_chunks * sizeof(double));
}

magicdec_status launch_spec_accept(int B, int gamma, int V, const float *target, const float *draft,
                                   const int32_t *draft_tok, const float *u_acc, const float *u_res, int greedy,
                                   int32_t *n_acc, int32_t *out_tok, int32_t *n_amb, void *ws, cudaStream_t st) {
    AcceptParams prm{};
    prm.target = target;
    prm.draft = draft;
    prm.draft_tok = draft_tok;
    prm.u_acc = u_acc;
    prm.u_res = u_res;
    prm.n_acc = n_acc;
    prm.out_tok = out_tok;
    prm.n_amb = n_amb;
    prm.B = B;
    prm.gamma = gamma;
    prm.V = V;
    prm.greedy = greedy ? 1 : 0;
    prm.n_chunks = (V + kAccChunk - 1) / kAccChunk;
    prm.rows_per_b = greedy ? gamma + 1 : 2 * gamma + 1;
    prm.err = magicdec_host::device_error_word();
    const int rows_alloc = 2 * gamma + 1;
    uint8_t *w = static_cast<uint8_t *>(ws);
    prm.counters = reinterpret_cast<int *>(w);
    w += (size_t)kAcceptMaxBatch * 4;
    prm.stats = reinterpret_cast<RowStat *>(w);
    w += align256a((size_t)B * rows_alloc * prm.n_chunks * sizeof(RowStat));
    prm.job = reinterpret_cast<JobInfo *>(w);
    w += align256a((size_t)B * sizeof(JobInfo));
    prm.chunk_sum = reinterpret_cast<double *>(w);

    magicdec_status s = magicdec_host::launch_pdl(accept_stats_kernel, dim3(prm.n_chunks, B * prm.rows_per_b),
                                                  dim3(kAccThreads), 0, st, prm);
    if (s != MAGICDEC_OK) return s;
    s = magicdec_host::launch_pdl(accept_chain_kernel, dim3((B + 127) / 128), dim3(128), 0, st, prm);
    if (s != MAGICDEC_OK || greedy) return s;
    return magicdec_host::launch_pdl(accept_sample_kernel, dim3(prm.n_chunks, B), dim3(kAccThreads), 0, st, prm);
}

}  // namespace magicdec
