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

constexpr int kStatChunk = 1024;      // logits per statistics record (one warp)
constexpr int kAccChunk = 4096;       // logits per sample CTA
constexpr int kAccThreads = 256;
constexpr int kAccPer = kStatChunk / 32;  // 32 logits per lane of a statistics warp, held in registers

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

// Warp sum of double-float values in a fixed butterfly order (fp32 pipe only).
__device__ __forceinline__ dflt warp_sum_df(dflt a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        dflt b;
        b.hi = __shfl_xor_sync(0xffffffffu, a.hi, o);
        b.lo = __shfl_xor_sync(0xffffffffu, a.lo, o);
        a = df_add(a, b);
    }
    return a;
}

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
    RowStat *stats;           // [B, rows_per_b, n_stat_chunks]
    JobInfo *job;             // [B]
    double *chunk_sum;        // [B, n_chunks]
    int *counters;            // [B], zero between calls
    int *err;
    int B, gamma, V, n_chunks, n_stat_chunks, rows_per_b, greedy;
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

// One record per warp and 1024-logit slice: lane l holds logits
// t0 + k*128 + 4l .. +3 (float4 path) or t0 + k*32 + l (scalar path), so each
// load instruction of the warp is coalesced and no block-level reduction is
// needed.  Sampling mode records the slice's max m and S = sum exp(x - m):
// each lane sums its 32 exponentials pairwise in fp32 (error ~1e-7 relative,
// the order of the exponential's own), lanes merge in fp64.  Greedy mode
// records only the top two logits and the argmax (smallest index on ties).
template <bool GREEDY>
__global__ void __launch_bounds__(kAccThreads) accept_stats_kernel(const AcceptParams p) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * (kAccThreads / 32) + warp;     // (row, record)
    const long long n_work = (long long)p.B * p.rows_per_b * p.n_stat_chunks;
    if (gw >= n_work) return;
    const long long row = gw / p.n_stat_chunks;
    const int rec = (int)(gw - row * p.n_stat_chunks);
    const int b = (int)(row / p.rows_per_b), r = (int)(row % p.rows_per_b);
    const float *x = row_ptr(p, b, r);
    const int t0 = rec * kStatChunk, t1 = min(t0 + kStatChunk, p.V);

    float v[kAccPer];
    const bool vec = ((p.V & 3) == 0);
    // index of v[k2]: t0 + (k2 >> 2) * 128 + 4 * lane + (k2 & 3) (float4 path),
    //                 t0 + k2 * 32 + lane (scalar path); increasing in k2
    if (vec) {
#pragma unroll
        for (int k2 = 0; k2 < kAccPer / 4; ++k2) {
            const int t = t0 + k2 * 128 + 4 * lane;
            float4 q = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (t < t1)
                asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                             : "=f"(q.x), "=f"(q.y), "=f"(q.z), "=f"(q.w)
                             : "l"(x + t));
            v[4 * k2] = q.x; v[4 * k2 + 1] = q.y; v[4 * k2 + 2] = q.z; v[4 * k2 + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int k2 = 0; k2 < kAccPer; ++k2) {
            const int t = t0 + k2 * 32 + lane;
            v[k2] = t < t1 ? __ldg(x + t) : -INFINITY;
        }
    }
    RowStat st;
    if (GREEDY) {
        float top1 = -INFINITY, top2 = -INFINITY;
        int arg = 0x7fffffff;
#pragma unroll
        for (int k2 = 0; k2 < kAccPer; ++k2) {
            const float e = v[k2];
            const int idx = vec ? t0 + (k2 >> 2) * 128 + 4 * lane + (k2 & 3) : t0 + k2 * 32 + lane;
            if (e > top1) {     // strict: the smallest index keeps a tie
                top2 = top1;
                top1 = e;
                arg = idx;
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
        st.s = 0.0;
        st.m = top1;
        st.top1 = top1;
        st.top2 = top2;
        st.arg = arg;
    } else {
        float mx = -INFINITY;
#pragma unroll
        for (int k2 = 0; k2 < kAccPer; ++k2) mx = fmaxf(mx, v[k2]);
        const float m = warp_max(mx);
        const float mb = m * kLog2e;
        float e[kAccPer];
#pragma unroll
        for (int k2 = 0; k2 < kAccPer; ++k2) e[k2] = fast_exp2(fmaf(v[k2], kLog2e, -mb));
#pragma unroll
        for (int w = kAccPer / 2; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) e[i] += e[i + w];
        double sum = (double)e[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        st.s = sum;
        st.m = m;
        st.top1 = m;
        st.top2 = m;
        st.arg = 0;
    }
    if (lane == 0) p.stats[row * p.n_stat_chunks + rec] = st;
}

// Whole-row statistics, merged in fp64: max m and S = sum exp(x - m).
struct RowAll {
    double s;
    float m, top1, top2;
    int arg;
};

constexpr int kMaxRows = 2 * 32 + 1;     // rows per sequence (gamma <= 32)
constexpr int kChainThreads = 256;

// One CTA per sequence.  Warp r merges row r's chunk records (lane c takes
// chunk c: one fp64 exponential per lane, fixed-order butterfly sum); warp 0
// then evaluates p(x)/q(x) for the gamma draft tokens (one position per
// lane), and thread 0 runs the sequential accept chain on those numbers.
__global__ void __launch_bounds__(kChainThreads) accept_chain_kernel(const AcceptParams p) {
    __shared__ RowAll rs[kMaxRows];
    __shared__ double ratio[32];
    __shared__ int okq0[32];
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    const int gamma = p.gamma, V = p.V;
    for (int r = warp; r < p.rows_per_b; r += kChainThreads / 32) {
        const RowStat *src = p.stats + ((long long)b * p.rows_per_b + r) * p.n_stat_chunks;
        float m = -INFINITY, t1 = -INFINITY, t2 = -INFINITY;
        int arg = 0x7fffffff;
        for (int c = lane; c < p.n_stat_chunks; c += 32) {
            const RowStat st = src[c];
            m = fmaxf(m, st.m);
            top_merge(t1, t2, arg, st.top1, st.top2, st.arg);
        }
        m = warp_max(m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float u1 = __shfl_xor_sync(0xffffffffu, t1, o);
            const float u2 = __shfl_xor_sync(0xffffffffu, t2, o);
            const int ua = __shfl_xor_sync(0xffffffffu, arg, o);
            top_merge(t1, t2, arg, u1, u2, ua);
        }
        double sum = 0.0;
        for (int c = lane; c < p.n_stat_chunks; c += 32) {
            const RowStat st = src[c];
            if (st.m != -INFINITY) sum += st.s * exp((double)st.m - (double)m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) rs[r] = RowAll{sum, m, t1, t2, arg};
    }
    __syncthreads();
    if (warp != 0) return;
    if (!p.greedy) {
        // ratio_i = p_i(x_i) / q_i(x_i); okq0: 1 = accept (q = 0 < p), 2 = reject
        for (int i = lane; i < gamma; i += 32) {
            const int x = __ldg(p.draft_tok + (long long)b * gamma + i);
            double rt = -1.0;
            int oq = 0;
            if (x >= 0 && x < V) {
                const RowAll ts = rs[i], ds = rs[gamma + 1 + i];
                const double px = exp((double)__ldg(row_ptr(p, b, i) + x) - (double)ts.m) / ts.s;
                const double qx = exp((double)__ldg(row_ptr(p, b, gamma + 1 + i) + x) - (double)ds.m) / ds.s;
                if (qx > 0.0) rt = px / qx;
                else oq = px > 0.0 ? 1 : 2;
            } else {
                oq = 2;
            }
            ratio[i] = rt;
            okq0[i] = oq;
        }
        __syncwarp();
    }
    if (lane != 0) return;
    int32_t *out = p.out_tok + (long long)b * (gamma + 1);
    JobInfo job{};
    int amb = 0, acc = gamma, emit = -1;
    for (int i = 0; i < gamma; ++i) {
        const int x = __ldg(p.draft_tok + (long long)b * gamma + i);
        bool ok;
        if (p.greedy) {
            const RowAll ts = rs[i];
            if ((double)ts.top1 - (double)ts.top2 < 1e-4) ++amb;
            ok = (x == ts.arg);
            if (!ok) emit = ts.arg;
        } else {
            const int oq = okq0[i];
            if (oq) {
                ok = oq == 1;
            } else {
                const double rt = ratio[i];
                const double u = __ldg(p.u_acc + (long long)b * gamma + i);
                ok = u < rt;
                if (fabs(u - rt) < 1e-4) ++amb;
            }
            if (!ok) {
                const RowAll ts = rs[i], ds = rs[gamma + 1 + i];
                job.kind = 1;
                job.mt = ts.m; job.st = ts.s;
                job.md = ds.m; job.sd = ds.s;
            }
        }
        if (!ok) { acc = i; break; }
        out[i] = x;
    }
    if (acc == gamma) {
        const RowAll ts = rs[gamma];
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

// Block sum of double-float values in a fixed order; returned (as a double) to every thread.
__device__ double block_sum_df(dflt v, dflt *scratch) {
    v = warp_sum_df(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    dflt t = scratch[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = df_add(t, scratch[w]);
    return df_to_double(t);
}

// Resample weights of four logits (target xt, draft xd) summed in double-float.
__device__ __forceinline__ dflt weight4_vals(const WeightCtx &w, const float4 xt, const float4 xd, bool resid) {
    const float tv[4] = {xt.x, xt.y, xt.z, xt.w};
    const float dv[4] = {xd.x, xd.y, xd.z, xd.w};
    dflt acc = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const dflt pt = df_mul_f(fast_exp2((tv[j] - w.mt) * kLog2e), w.inv_st);
        if (!resid) {
            acc = df_add(acc, pt);
        } else {
            const dflt qt = df_mul_f(fast_exp2((dv[j] - w.md) * kLog2e), w.inv_sd);
            const dflt d = df_sub(pt, qt);
            if (d.hi > 0.f) acc = df_add(acc, d);
        }
    }
    return acc;
}

// Sum of weights over [t0, t1) (thread-strided double-float, then a fixed tree).
// A full, aligned chunk issues all its loads before any arithmetic.
__device__ double chunk_weight_sum(const WeightCtx &w, int t0, int t1, bool vec4, dflt *scratch) {
    constexpr int NV = kAccChunk / (4 * kAccThreads);     // float4 per thread in a full chunk
    dflt acc = {0.f, 0.f};
    const bool resid = !(w.kind == 2 || w.use_p);
    if (vec4 && t1 - t0 == kAccChunk && (t0 & 3) == 0 && blockDim.x == kAccThreads) {
        float4 xt[NV], xd[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int t = t0 + 4 * (int)threadIdx.x + i * 4 * kAccThreads;
            xt[i] = __ldg(reinterpret_cast<const float4 *>(w.tr + t));
            xd[i] = resid ? __ldg(reinterpret_cast<const float4 *>(w.dr + t)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) acc = df_add(acc, weight4_vals(w, xt[i], xd[i], resid));
    } else if (vec4 && ((t1 - t0) & 3) == 0 && (t0 & 3) == 0) {
        for (int t = t0 + 4 * threadIdx.x; t < t1; t += 4 * blockDim.x) {
            const float4 xt = __ldg(reinterpret_cast<const float4 *>(w.tr + t));
            const float4 xd = resid ? __ldg(reinterpret_cast<const float4 *>(w.dr + t)) : make_float4(0.f, 0.f, 0.f, 0.f);
            acc = df_add(acc, weight4_vals(w, xt, xd, resid));
        }
    } else {
        for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) acc = df_add(acc, weight_at(w, t));
    }
    return block_sum_df(acc, scratch);
}

// Inclusive block scan of one double per thread (fixed order).
__device__ double block_scan_d(double v, double *buf) {
    const int tid = threadIdx.x;
    buf[tid] = v;
    __syncthreads();
    for (int off = 1; off < (int)blockDim.x; off <<= 1) {
        const double add = tid >= off ? buf[tid - off] : 0.0;
        __syncthreads();
        buf[tid] += add;
        __syncthreads();
    }
    return buf[tid];
}

__global__ void __launch_bounds__(kAccThreads) accept_sample_kernel(const AcceptParams p) {
    __shared__ dflt scratch[kAccThreads / 32];
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
    const bool vec4 = (p.V & 3) == 0;
    const double csum = chunk_weight_sum(w, t0, t1, vec4, scratch);
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
        // chunk sums of p are recomputed here into seg[] (n_chunks <= 256 is
        // checked at the entry point).
        use_p = true;
        w.use_p = true;
        W = 0.0;
        for (int c = 0; c < p.n_chunks; ++c) {
            const double v = chunk_weight_sum(w, c * kAccChunk, min((c + 1) * kAccChunk, p.V), vec4, scratch);
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
    // Scan inside chunk cstar: each thread owns a contiguous run of logits; an
    // fp64 block scan of the run sums tells every thread where its run starts,
    // and the one run containing the crossing walks its logits.
    __shared__ int found_token, found_amb;
    if (threadIdx.x == 0) { found_token = -1; found_amb = 0; }
    const int c0 = cstar * kAccChunk, c1 = min(c0 + kAccChunk, p.V);
    const int per = (c1 - c0 + kAccThreads - 1) / kAccThreads;
    const int my0 = c0 + threadIdx.x * per, my1 = min(my0 + per, c1);
    dflt mine = {0.f, 0.f};
    for (int t = my0; t < my1; ++t) mine = df_add(mine, weight_at(w, t));
    const double my_sum = df_to_double(mine);
    const double incl = block_scan_d(my_sum, seg);
    const double start = before + (incl - my_sum);
    if (my0 < my1 && start <= target && target < before + incl) {
        double prev = start;
        for (int t = my0; t < my1; ++t) {
            const double nxt = prev + df_to_double(weight_at(w, t));
            if (nxt > target) {
                found_token = t;
                found_amb = ((t > 0 && target - prev < tol) || (t < p.V - 1 && nxt - target < tol)) ? 1 : 0;
                break;
            }
            prev = nxt;
        }
        if (found_token < 0) {   // rounding inside the run: its last positive weight
            for (int t = my1 - 1; t >= my0; --t)
                if (weight_at(w, t).hi > 0.f) { found_token = t; break; }
            found_amb = 1;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int token = found_token;
        amb += found_amb;
        if (token < 0) {
            // rounding pushed the target past the chunk: its last positive weight
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
    const int n_stat = (V + kStatChunk - 1) / kStatChunk;
    const int rows = 2 * gamma + 1;
    return (size_t)kAcceptMaxBatch * 4 + align256a((size_t)B * rows * n_stat * sizeof(RowStat)) +
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
    prm.n_stat_chunks = (V + kStatChunk - 1) / kStatChunk;
    prm.rows_per_b = greedy ? gamma + 1 : 2 * gamma + 1;
    if (2 * gamma + 1 > kMaxRows) return MAGICDEC_ERR_UNSUPPORTED;
    prm.err = magicdec_host::device_error_word();
    const int rows_alloc = 2 * gamma + 1;
    uint8_t *w = static_cast<uint8_t *>(ws);
    prm.counters = reinterpret_cast<int *>(w);
    w += (size_t)kAcceptMaxBatch * 4;
    prm.stats = reinterpret_cast<RowStat *>(w);
    w += align256a((size_t)B * rows_alloc * prm.n_stat_chunks * sizeof(RowStat));
    prm.job = reinterpret_cast<JobInfo *>(w);
    w += align256a((size_t)B * sizeof(JobInfo));
    prm.chunk_sum = reinterpret_cast<double *>(w);

    const long long n_work = (long long)B * prm.rows_per_b * prm.n_stat_chunks;
    magicdec_status s = magicdec_host::launch_pdl(greedy ? accept_stats_kernel<true> : accept_stats_kernel<false>,
                                                  dim3((unsigned)((n_work + kAccThreads / 32 - 1) / (kAccThreads / 32))),
                                                  dim3(kAccThreads), 0, st, prm);
    if (s != MAGICDEC_OK) return s;
    s = magicdec_host::launch_pdl(accept_chain_kernel, dim3(B), dim3(kChainThreads), 0, st, prm);
    if (s != MAGICDEC_OK || greedy) return s;
    return magicdec_host::launch_pdl(accept_sample_kernel, dim3(prm.n_chunks, B), dim3(kAccThreads), 0, st, prm);
}

}  // namespace magicdec
