// accept.cu -- speculative-sampling accept / resample (Leviathan et al., the
// rule behind Eq. 1 of the MagicDec paper, section 3.1) and greedy
// verification (paper section 5.1), sm_103a.
//
// The step streams the target logits [B, gamma+1, V] and draft logits
// [B, gamma, V] once (fp32, HBM-bound) and then touches one row pair per
// sequence again for the resample.  Four launches (greedy mode: the first
// two):
//   stats  one CTA per (row, 4096 logits): for each of its four 1024-logit
//          warp slices the max and sum of exp(x - max), merged into one
//          record (double-float across lanes and warps); greedy
//          mode keeps top-1 (smallest index among equals), top-2 and argmax;
//   chain  one CTA per sequence: a warp per row merges the row's records in
//          fp64, warp 0 evaluates p(x)/q(x) for each draft token in fp64 and
//          its thread 0 runs the sequential accept chain (or the greedy
//          argmax chain) and records the row(s) to resample from;
//   chunk  one CTA per (sequence, 4096-logit chunk) of the sampled row(s):
//          the chunk's sum of resample weights max(0, p - q), or p for the
//          bonus token, in reverse sequence order (the rows read last by the
//          statistics pass are still in L2);
//   draw   one CTA per sequence: finds the chunk where the running sum
//          crosses u * total (shuffle scan + ballot) and walks it with
//          double-float weights; the chunk sums, scans and comparisons of the
//          draw are double-float on the FP32 pipes (fp64 throughput is scarce).
// Only the per-logit exponentials are single precision (random ~1e-6 relative
// errors that average out in the sums); normalisers, ratios and running sums
// carry ~1e-12 relative error, so the drawn token agrees with an exact
// evaluation except when u * total falls within ~1e-9 of a token boundary.
#include "common.cuh"
#include "dfloat.cuh"

namespace magicdec {

constexpr int kStatChunk = 1024;      // logits per statistics record (one warp)
constexpr int kAccThreads = 128;     // statistics CTA: 4 warps, one record per 4 slices
constexpr int kAccPer = kStatChunk / 32;  // 32 logits per lane of a statistics warp, held in registers

// ------------------------------------------------------------------- stats
struct RowStat {
    dflt s;            // sum over the chunk of exp(x - m), double-float
    float m;           // chunk max
    float top1, top2;
    int arg;
};

struct JobInfo {
    // 1/S_t, 1/S_d as double-float: the target / draft normalisers relative to mt / md
    float inv_st_hi, inv_st_lo, inv_sd_hi, inv_sd_lo;
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
    RowStat *stats;           // [B, rows_per_b, n_stat_chunks]: one record per 4 slices of 1024 logits
    JobInfo *job;             // [B]
    int *err;
    dflt *chunk_sum;          // [B, n_chunks] weight sums of the sampled row(s), double-float
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

// One record per CTA: the CTA of (row, blockIdx.y) covers the row's 1024-logit
// slices 4*blockIdx.y .. +3, one per warp.  Lane l of a warp holds logits
// t0 + k*128 + 4l .. +3 (float4 path) or t0 + k*32 + l (scalar path), so each
// load instruction is coalesced.  Sampling mode records the CTA's max m and
// S = sum exp(x - m): the warps agree on m through shared memory, each lane
// sums its 32 exponentials pairwise in fp32 (error ~1e-7 relative, the order
// of the exponential's own), lanes and warps merge in double-float, in
// a fixed order.
// Greedy mode records only the top two logits and the argmax (smallest index
// on ties).
template <bool GREEDY>
__global__ void __launch_bounds__(kAccThreads) accept_stats_kernel(const AcceptParams p) {
    constexpr int NW = kAccThreads / 32;
    __shared__ float s_max[NW], s_t1[NW], s_t2[NW];
    __shared__ int s_arg[NW];
    __shared__ dflt s_sum[NW];
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = blockIdx.x;
    const int rec = blockIdx.y;
    const int slice = rec * NW + warp;
    const int b = (int)(row / p.rows_per_b), r = (int)(row % p.rows_per_b);
    const float *x = row_ptr(p, b, r);
    const int t0 = slice * kStatChunk, t1 = min(t0 + kStatChunk, p.V);   // empty past the row's end

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
            v[k2] = t < t1 ? ld_dep_f(x + t) : -INFINITY;
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
        if (lane == 0) {
            s_t1[warp] = top1;
            s_t2[warp] = top2;
            s_arg[warp] = arg;
        }
        __syncthreads();
        if (threadIdx.x != 0) return;
        for (int w2 = 1; w2 < NW; ++w2) top_merge(top1, top2, arg, s_t1[w2], s_t2[w2], s_arg[w2]);
        st.s = dflt{0.f, 0.f};
        st.m = top1;
        st.top1 = top1;
        st.top2 = top2;
        st.arg = arg;
    } else {
        float mx = -INFINITY;
#pragma unroll
        for (int k2 = 0; k2 < kAccPer; ++k2) mx = fmaxf(mx, v[k2]);
        mx = warp_max(mx);
        if (lane == 0) s_max[warp] = mx;
        __syncthreads();
        float m = s_max[0];
#pragma unroll
        for (int w2 = 1; w2 < NW; ++w2) m = fmaxf(m, s_max[w2]);
        dflt sum = {0.f, 0.f};
        if (m != -INFINITY) {
            const float mb = m * kLog2e;
            float e[kAccPer];
#pragma unroll
            for (int k2 = 0; k2 < kAccPer; ++k2) e[k2] = fast_exp2(fmaf(v[k2], kLog2e, -mb));
#pragma unroll
            for (int w = kAccPer / 2; w > 0; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) e[i] += e[i + w];
            // lanes and warps merge in double-float on the FP32 pipes (fp64
            // throughput is scarce on this GPU)
            sum = warp_sum_df(dflt{e[0], 0.f});
        }
        if (lane == 0) s_sum[warp] = sum;
        __syncthreads();
        if (threadIdx.x != 0) return;
        dflt S = s_sum[0];
        for (int w2 = 1; w2 < NW; ++w2) S = df_add(S, s_sum[w2]);
        st.s = S;
        st.m = m;
        st.top1 = m;
        st.top2 = m;
        st.arg = 0;
    }
    p.stats[row * p.n_stat_chunks + rec] = st;
}

// Whole-row statistics: max m and S = sum exp(x - m) (double-float).
struct RowAll {
    dflt s;
    float m, top1, top2;
    int arg;
};

constexpr int kMaxRows = 2 * 32 + 1;     // rows per sequence (gamma <= 32)
constexpr int kChainThreads = 256;

// One CTA per sequence.  Warp r merges row r's chunk records (lane c takes
// chunk c: one double-float exponential per lane, fixed-order butterfly sum);
// warp 0 then evaluates p(x)/q(x) for the gamma draft tokens (one position
// per lane), and thread 0 runs the sequential accept chain on those numbers.
// All of it is double-float on the FP32 pipes, but for ratios whose
// exponentials could underflow (logits more than 80 below their row's
// maximum), which take the fp64 path.
__global__ void __launch_bounds__(kChainThreads) accept_chain_kernel(const AcceptParams p) {
    __shared__ RowAll rs[kMaxRows];
    __shared__ dflt ratio[32];
    __shared__ int okq0[32];
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    const int gamma = p.gamma, V = p.V;
    // the draft tokens' target and draft logits, loaded before the record merge
    // so that their latency overlaps it (warp 0, one position per lane)
    float xt = 0.f, xd = 0.f;
    int xtok = -1;
    if (!p.greedy && warp == 0 && lane < gamma) {
        xtok = ld_dep(p.draft_tok + (long long)b * gamma + lane);
        if (xtok >= 0 && xtok < V) {
            xt = ld_dep_f(row_ptr(p, b, lane) + xtok);
            xd = ld_dep_f(row_ptr(p, b, gamma + 1 + lane) + xtok);
        }
    }
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
        // S = sum of s_c exp(m_c - m), in double-float on the FP32 pipes
        dflt sum = {0.f, 0.f};
        for (int c = lane; c < p.n_stat_chunks; c += 32) {
            const RowStat st = src[c];
            if (st.m != -INFINITY) sum = df_add(sum, df_mul(st.s, df_exp_diff(st.m, m)));
        }
        sum = warp_sum_df(sum);
        if (lane == 0) rs[r] = RowAll{sum, m, t1, t2, arg};
    }
    __syncthreads();
    if (warp != 0) return;
    if (!p.greedy) {
        // ratio_i = p_i(x_i) / q_i(x_i); okq0: 1 = accept (q = 0 < p), 2 = reject
        if (lane < gamma) {               // gamma <= 32: position i = lane, logits prefetched
            const int i = lane;
            dflt rt = {-1.f, 0.f};
            int oq = 0;
            if (xtok >= 0 && xtok < V) {
                const RowAll ts = rs[i], ds = rs[gamma + 1 + i];
                if (xt - ts.m > -80.f && xd - ds.m > -80.f) {
                    // p / q = exp(xt - mt) S_d / (exp(xd - md) S_t)
                    rt = df_div(df_mul(df_exp_diff(xt, ts.m), ds.s), df_mul(df_exp_diff(xd, ds.m), ts.s));
                } else {
                    // an exponential may underflow: q = 0 < p accepts, p = q = 0 rejects
                    const double dp = (double)xt - (double)ts.m, dq = (double)xd - (double)ds.m;
                    const double px = exp(dp) / df_to_double(ts.s), qx = exp(dq) / df_to_double(ds.s);
                    if (qx > 0.0) rt = df_from_double(px / qx);
                    else oq = px > 0.0 ? 1 : 2;
                }
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
        const int x = ld_dep(p.draft_tok + (long long)b * gamma + i);
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
                const dflt rt = ratio[i];
                const float u = ld_dep_f(p.u_acc + (long long)b * gamma + i);
                ok = df_lt(dflt{u, 0.f}, rt);
                if (fabsf(df_sub(rt, dflt{u, 0.f}).hi) < 1e-4f) ++amb;
            }
            if (!ok) {
                const RowAll ts = rs[i], ds = rs[gamma + 1 + i];
                job.kind = 1;
                job.mt = ts.m;
                job.md = ds.m;
                const dflt it = df_div(dflt{1.f, 0.f}, ts.s), id = df_div(dflt{1.f, 0.f}, ds.s);
                job.inv_st_hi = it.hi;
                job.inv_st_lo = it.lo;
                job.inv_sd_hi = id.hi;
                job.inv_sd_lo = id.lo;
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
            job.mt = ts.m;
            const dflt it = df_div(dflt{1.f, 0.f}, ts.s);
            job.inv_st_hi = it.hi;
            job.inv_st_lo = it.lo;
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

// Weight of one logit pair as an unnormalised double-float pair hi + lo.
// p = e_t * (1/S_t) and q = e_d * (1/S_d) are split exactly into hi + lo (one
// FMA each), p - q is one two-sum of the high parts plus the low parts, and a
// pair whose value is not positive weighs 0.  Every term is within ~1e-14 of
// the exact product difference of the fp32 exponentials.
__device__ __forceinline__ dflt weight_of(const WeightCtx &w, float xt, float xd, bool resid) {
    const float et = fast_exp2((xt - w.mt) * kLog2e);
    const float ph = et * w.inv_st.hi;
    const float pl = fmaf(et, w.inv_st.hi, -ph) + et * w.inv_st.lo;
    if (!resid) return dflt{ph, pl};
    const float ed = fast_exp2((xd - w.md) * kLog2e);
    const float qh = ed * w.inv_sd.hi;
    const float ql = fmaf(ed, w.inv_sd.hi, -qh) + ed * w.inv_sd.lo;
    const float sh = ph - qh;
    const float bb = sh - ph;
    const float lo = ((ph - (sh - bb)) + (-qh - bb)) + (pl - ql);
    return sh + lo > 0.f ? dflt{sh, lo} : dflt{0.f, 0.f};
}

// A weight that is not positive is returned as exactly {0, 0}.
__device__ __forceinline__ bool weight_positive(dflt d) { return d.hi != 0.f || d.lo != 0.f; }

__device__ __forceinline__ dflt weight_at(const WeightCtx &w, int t) {
    const bool resid = !(w.kind == 2 || w.use_p);
    return weight_of(w, ld_dep_f(w.tr + t), resid ? ld_dep_f(w.dr + t) : 0.f, resid);
}

// Running sum of non-negative unnormalised pairs: a two-sum of the high parts,
// the low parts and rounding errors gathered in lo (renormalised by the caller).
__device__ __forceinline__ void acc_add(dflt &acc, dflt d) {
    const float sh = acc.hi + d.hi;
    const float bb = sh - acc.hi;
    acc.lo += ((acc.hi - (sh - bb)) + (d.hi - bb)) + d.lo;
    acc.hi = sh;
}

__device__ __forceinline__ dflt acc_done(dflt acc) { return quick_two_sum(acc.hi, acc.lo); }

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

// Resample weights of four logits (target xt, draft xd) added to acc.
__device__ __forceinline__ void weight4_acc(dflt &acc, const WeightCtx &w, const float4 xt, const float4 xd,
                                            bool resid) {
    acc_add(acc, weight_of(w, xt.x, xd.x, resid));
    acc_add(acc, weight_of(w, xt.y, xd.y, resid));
    acc_add(acc, weight_of(w, xt.z, xd.z, resid));
    acc_add(acc, weight_of(w, xt.w, xd.w, resid));
}

// Resample weight of one logit pair in fp32, for the chunk sums: each
// normaliser's double-float reciprocal enters through one FMA, so the result
// is the exact value rounded once or twice (unbiased, ~1e-7 relative: the
// order of the exponential's own error); the sums are accumulated in
// double-float.  The walk inside the chunk that holds the draw uses the
// double-float weights above.
__device__ __forceinline__ float weight_fast(const WeightCtx &w, float xt, float xd, bool resid) {
    const float et = fast_exp2((xt - w.mt) * kLog2e);
    const float pw = fmaf(et, w.inv_st.lo, et * w.inv_st.hi);
    if (!resid) return pw;
    const float ed = fast_exp2((xd - w.md) * kLog2e);
    const float qw = fmaf(ed, w.inv_sd.lo, ed * w.inv_sd.hi);
    return fmaxf(pw - qw, 0.f);
}

__device__ __forceinline__ void weight4_fast_acc(dflt &acc, const WeightCtx &w, const float4 xt, const float4 xd,
                                                 bool resid) {
    acc_add(acc, dflt{weight_fast(w, xt.x, xd.x, resid), 0.f});
    acc_add(acc, dflt{weight_fast(w, xt.y, xd.y, resid), 0.f});
    acc_add(acc, dflt{weight_fast(w, xt.z, xd.z, resid), 0.f});
    acc_add(acc, dflt{weight_fast(w, xt.w, xd.w, resid), 0.f});
}

// Inclusive scan of one double-float per thread in thread order: shuffle
// scans in each warp, a scan of the warp totals by warp 0, two barriers.  The
// sums of the draw run on the FP32 pipes in double-float (~1e-14 relative)
// rather than in fp64, whose pipe is narrow on this GPU.
__device__ dflt block_scan_df(dflt v, dflt *wtot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    dflt x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const dflt y = df_shfl_up(x, o);
        if (lane >= o) x = df_add(x, y);
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        dflt t = lane < nw ? wtot[lane] : dflt{0.f, 0.f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const dflt y = df_shfl_up(t, o);
            if (lane >= o) t = df_add(t, y);
        }
        if (lane < nw) wtot[lane] = t;
    }
    __syncthreads();
    return warp ? df_add(x, wtot[warp - 1]) : x;
}

// Sum of the chunk sums in a fixed order, computed by one warp (every lane
// returns it): lane l adds its contiguous block, then a shuffle scan.
__device__ dflt warp_chunk_total(const dflt *csum, int n, int lane) {
    const int per = (n + 31) / 32;
    const int lo = min(n, lane * per), hi = min(n, lo + per);
    dflt part = {0.f, 0.f};
    for (int c = lo; c < hi; ++c) part = df_add(part, csum[c]);
    dflt incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const dflt y = df_shfl_up(incl, o);
        if (lane >= o) incl = df_add(incl, y);
    }
    return df_shfl(incl, 31);
}

constexpr int kSmpThreads = 1024;
constexpr int kSmpChunk = 4 * kSmpThreads;   // logits per chunk: one float4 of each row per thread
constexpr int kSmpBatch = 4;                 // chunks whose loads are in flight together
constexpr int kSmpMaxChunks = 256;

// Chunk sums of the weights of chunks c0 .. c0+kSmpBatch-1 into csum[].
// Thread t holds logits 4t .. 4t+3 of each chunk; a chunk's per-thread sums
// are reduced in a fixed order (warps by shuffles, then warp 0's lanes).
__device__ __forceinline__ void batch_chunk_sums(const WeightCtx &w, bool resid, int V, bool vec4, int c0,
                                                 int n_chunks, dflt (*wred)[32], dflt *csum) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float4 xt[kSmpBatch], xd[kSmpBatch];
    const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
    for (int u = 0; u < kSmpBatch; ++u) {
        const int t = (c0 + u) * kSmpChunk + 4 * tid;
        xt[u] = none;
        xd[u] = none;
        if (c0 + u < n_chunks && t < V) {
            if (vec4) {
                xt[u] = ld_dep_f4(reinterpret_cast<const float4 *>(w.tr + t));
                if (resid) xd[u] = ld_dep_f4(reinterpret_cast<const float4 *>(w.dr + t));
            } else {
                float a[4], d[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a[e] = t + e < V ? ld_dep_f(w.tr + t + e) : -INFINITY;
                    d[e] = (resid && t + e < V) ? ld_dep_f(w.dr + t + e) : -INFINITY;
                }
                xt[u] = make_float4(a[0], a[1], a[2], a[3]);
                xd[u] = make_float4(d[0], d[1], d[2], d[3]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kSmpBatch; ++u) {
        dflt acc = {0.f, 0.f};
        weight4_acc(acc, w, xt[u], xd[u], resid);
        acc = warp_sum_df(acc_done(acc));
        if (lane == 0) wred[u][warp] = acc;
    }
    __syncthreads();
    if (warp < kSmpBatch) {
        dflt v = wred[warp][lane];
        v = warp_sum_df(v);
        if (lane == 0 && c0 + warp < n_chunks) csum[c0 + warp] = v;
    }
    __syncthreads();
}

constexpr int kChkThreads = 256;
constexpr int kChkPer = kSmpChunk / (4 * kChkThreads);   // float4 of each row per thread (4)

// Weight sum of chunk blockIdx.x of sequence B-1-blockIdx.y into
// chunk_sum[b][c] (kind 1: residual max(0, p - q); kind 2: p), with the fp32
// weights above.  Sequences go in reverse order: the statistics pass read the
// last sequences' rows last, so those are still in L2.  All loads of a thread
// are issued before any arithmetic; the block sum is reduced in a fixed order.
__global__ void __launch_bounds__(kChkThreads) accept_chunk_kernel(const AcceptParams p) {
    __shared__ dflt wred[kChkThreads / 32];
    const int c = blockIdx.x, b = p.B - 1 - (int)blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    w.inv_st = dflt{job.inv_st_hi, job.inv_st_lo};
    w.inv_sd = dflt{job.inv_sd_hi, job.inv_sd_lo};
    const bool resid = job.kind == 1;
    const int V = p.V, t0 = c * kSmpChunk;
    const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 xt[kChkPer], xd[kChkPer];
#pragma unroll
    for (int i = 0; i < kChkPer; ++i) {
        const int t = t0 + 4 * tid + i * 4 * kChkThreads;
        xt[i] = none;
        xd[i] = none;
        if (t < V) {
            if ((V & 3) == 0) {
                xt[i] = ld_dep_f4(reinterpret_cast<const float4 *>(w.tr + t));
                if (resid) xd[i] = ld_dep_f4(reinterpret_cast<const float4 *>(w.dr + t));
            } else {
                float a[4], d[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a[e] = t + e < V ? ld_dep_f(w.tr + t + e) : -INFINITY;
                    d[e] = (resid && t + e < V) ? ld_dep_f(w.dr + t + e) : -INFINITY;
                }
                xt[i] = make_float4(a[0], a[1], a[2], a[3]);
                xd[i] = make_float4(d[0], d[1], d[2], d[3]);
            }
        }
    }
    dflt acc = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kChkPer; ++i) weight4_fast_acc(acc, w, xt[i], xd[i], resid);
    acc = warp_sum_df(acc_done(acc));
    if (lane == 0) wred[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        // the 8 warp sums, combined by a fixed shuffle tree
        dflt t = lane < kChkThreads / 32 ? wred[lane] : dflt{0.f, 0.f};
#pragma unroll
        for (int o = (kChkThreads / 32) / 2; o > 0; o >>= 1) {
            dflt u;
            u.hi = __shfl_down_sync(0xffffffffu, t.hi, o);
            u.lo = __shfl_down_sync(0xffffffffu, t.lo, o);
            t = df_add(t, u);
        }
        if (lane == 0) p.chunk_sum[(long long)b * p.n_chunks + c] = t;
    }
}

// One CTA per sequence with something to draw (job kind 1: the residual
// norm(max(0, p - q)) at the rejected position; kind 2: the bonus token from
// the last target row).  From the chunk sums it finds the chunk where the
// cumulative weight passes u * total and walks it.  An empty residual (p == q
// up to rounding) is redrawn from p, whose chunk sums this CTA recomputes.
__global__ void __launch_bounds__(kSmpThreads, 1) accept_sample_kernel(const AcceptParams p) {
    __shared__ dflt csum[kSmpMaxChunks];
    __shared__ dflt wred[kSmpBatch][32];
    __shared__ dflt wtot[32];
    __shared__ dflt s_W, s_before;
    __shared__ int s_cstar, s_amb;
    __shared__ int found_token, found_amb;
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    w.inv_st = dflt{job.inv_st_hi, job.inv_st_lo};
    w.inv_sd = dflt{job.inv_sd_hi, job.inv_sd_lo};
    const int V = p.V, n_chunks = p.n_chunks;
    const bool vec4 = (V & 3) == 0;
    bool resid = job.kind == 1;
    for (int c = tid; c < n_chunks; c += kSmpThreads) csum[c] = p.chunk_sum[(long long)b * n_chunks + c];
    __syncthreads();
    if (warp == 0) s_W = warp_chunk_total(csum, n_chunks, lane);
    __syncthreads();
    dflt W = s_W;
    if (!df_positive(W)) {
        // Residual empty (p == q up to rounding): draw from p instead.
        w.use_p = true;
        resid = false;
        for (int c = 0; c < n_chunks; c += kSmpBatch) batch_chunk_sums(w, resid, V, vec4, c, n_chunks, wred, csum);
        if (warp == 0) s_W = warp_chunk_total(csum, n_chunks, lane);
        __syncthreads();
        W = s_W;
    }
    const float u = ld_dep_f(p.u_res + b);
    const dflt target = df_mul_f(u, W);
    const float tol = 1e-7f * W.hi;
    int amb = job.amb;
    if (warp == 0) {
        // lane l sums its contiguous block of chunks; a shuffle scan over the
        // lanes and a ballot find the lane whose block holds the crossing
        const int per = (n_chunks + 31) / 32;
        const int lo = min(n_chunks, lane * per), hi = min(n_chunks, lo + per);
        dflt part = {0.f, 0.f};
        for (int c = lo; c < hi; ++c) part = df_add(part, csum[c]);
        dflt incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const dflt y = df_shfl_up(incl, o);
            if (lane >= o) incl = df_add(incl, y);
        }
        const dflt excl = df_sub(incl, part);
        const unsigned own = __ballot_sync(0xffffffffu, hi > lo && df_le(excl, target) && df_lt(target, incl));
        int cs = -1;
        if (own && lane == __ffs(own) - 1) {
            dflt before = excl;
            for (int c = lo; c < hi; ++c) {
                const dflt nb = df_add(before, csum[c]);
                if (df_lt(target, nb)) { cs = c; break; }
                before = nb;
            }
            if (cs >= 0) {
                s_cstar = cs;
                s_before = before;
                s_amb = 0;
            }
        }
        cs = __shfl_sync(0xffffffffu, cs, own ? __ffs(own) - 1 : 0);
        if (cs < 0 && lane == 0) {
            // rounding pushed the target past the total: the last chunk with weight
            int last = -1;
            for (int c = 0; c < n_chunks; ++c)
                if (df_positive(csum[c])) last = c;
            if (last < 0) last = n_chunks - 1;
            dflt bf = {0.f, 0.f};
            for (int c = 0; c < last; ++c) bf = df_add(bf, csum[c]);
            s_cstar = last;
            s_before = bf;
            s_amb = 1;
        }
    }
    if (tid == 0) { found_token = -1; found_amb = 0; }
    __syncthreads();
    const int cstar = s_cstar;
    const dflt before = s_before;
    amb += s_amb;
    if (tid == 0) { found_token = -1; found_amb = 0; }
    // Walk chunk cstar: thread t owns its logits 4t .. 4t+3; a double-float
    // block scan of the per-thread sums tells every thread where its run
    // starts, and the one run containing the crossing walks its four weights.
    const int cb = cstar * kSmpChunk, ce = min(cb + kSmpChunk, V);
    const int my0 = cb + 4 * tid;
    dflt wt[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        wt[e] = my0 + e < ce ? weight_of(w, ld_dep_f(w.tr + my0 + e), resid ? ld_dep_f(w.dr + my0 + e) : 0.f, resid)
                             : dflt{0.f, 0.f};
    dflt mine = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) acc_add(mine, wt[e]);
    const dflt my_sum = acc_done(mine);
    const dflt incl = block_scan_df(my_sum, wtot);
    const dflt start = df_add(before, df_sub(incl, my_sum));
    if (my0 < ce && df_le(start, target) && df_lt(target, df_add(before, incl))) {
        dflt prev = start;
        int tok = -1, last_pos = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (weight_positive(wt[e])) last_pos = e;
            const dflt nxt = df_add(prev, wt[e]);
            if (tok < 0 && df_lt(target, nxt)) {
                tok = e;
                const int t = my0 + e;
                found_amb = ((t > 0 && df_sub(target, prev).hi < tol) || (t < V - 1 && df_sub(nxt, target).hi < tol))
                                ? 1 : 0;
            }
            if (tok < 0) prev = nxt;
        }
        if (tok >= 0) {
            found_token = my0 + tok;
        } else if (last_pos >= 0) {   // rounding inside the run: its last positive weight
            found_token = my0 + last_pos;
            found_amb = 1;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int token = found_token;
        amb += found_amb;
        if (token < 0) {
            // rounding pushed the target past the chunk: its last positive weight
            for (int t = ce - 1; t >= cb; --t)
                if (weight_positive(weight_at(w, t))) { token = t; break; }
            if (token < 0) token = ce - 1;
            ++amb;
        }
        p.out_tok[(long long)b * (p.gamma + 1) + job.acc] = token;
        if (p.n_amb) p.n_amb[b] = amb;
    }
}

// ------------------------------------------------------------------- host side
static size_t align256a(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout: [row stats][per-sequence job][chunk sums]; no initial
// contents needed.
size_t accept_workspace_bytes(int B, int gamma, int V) {
    const int n_stat = ((V + kStatChunk - 1) / kStatChunk + kAccThreads / 32 - 1) / (kAccThreads / 32);
    const int n_chunks = (V + kSmpChunk - 1) / kSmpChunk;
    const int rows = 2 * gamma + 1;
    return align256a((size_t)B * rows * n_stat * sizeof(RowStat)) + align256a((size_t)B * sizeof(JobInfo)) +
           align256a((size_t)B * n_chunks * sizeof(dflt));
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
    prm.n_stat_chunks = ((V + kStatChunk - 1) / kStatChunk + kAccThreads / 32 - 1) / (kAccThreads / 32);
    prm.n_chunks = (V + kSmpChunk - 1) / kSmpChunk;
    prm.rows_per_b = greedy ? gamma + 1 : 2 * gamma + 1;
    if (2 * gamma + 1 > kMaxRows) return MAGICDEC_ERR_UNSUPPORTED;
    prm.err = magicdec_host::device_error_word();
    const int rows_alloc = 2 * gamma + 1;
    uint8_t *w = static_cast<uint8_t *>(ws);
    prm.stats = reinterpret_cast<RowStat *>(w);
    w += align256a((size_t)B * rows_alloc * prm.n_stat_chunks * sizeof(RowStat));
    prm.job = reinterpret_cast<JobInfo *>(w);
    w += align256a((size_t)B * sizeof(JobInfo));
    prm.chunk_sum = reinterpret_cast<dflt *>(w);

    magicdec_status s = magicdec_host::launch_pdl(greedy ? accept_stats_kernel<true> : accept_stats_kernel<false>,
                                                  dim3((unsigned)(B * prm.rows_per_b), (unsigned)prm.n_stat_chunks),
                                                  dim3(kAccThreads), 0, st, prm);
    if (s != MAGICDEC_OK) return s;
    s = magicdec_host::launch_pdl(accept_chain_kernel, dim3(B), dim3(kChainThreads), 0, st, prm);
    if (s != MAGICDEC_OK || greedy) return s;
    s = magicdec_host::launch_pdl(accept_chunk_kernel, dim3(prm.n_chunks, B), dim3(kChkThreads), 0, st, prm);
    if (s != MAGICDEC_OK) return s;
    return magicdec_host::launch_pdl(accept_sample_kernel, dim3(B), dim3(kSmpThreads), 0, st, prm);
}

}  // namespace magicdec
