// Accuracy check of df_exp_diff and df_div (long_context_self_gb300/csrc/dfloat.cuh):
// the double-float exp(a - b) and quotient of the accept kernels against the
// host's long-double arithmetic on the same inputs.  Prints the largest
// errors and exits non-zero when they exceed the bounds stated below.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_runtime.h>

#include "../long_context_self_gb300/csrc/dfloat.cuh"

using magicdec::dflt;

__global__ void div_kernel(const float *ah, const float *al, const float *bh, const float *bl, float *qh, float *ql,
                           int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const dflt q = magicdec::df_div(dflt{ah[i], al[i]}, dflt{bh[i], bl[i]});
        qh[i] = q.hi;
        ql[i] = q.lo;
    }
}

__global__ void exp_diff_kernel(const float *a, const float *b, float *hi, float *lo, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const dflt e = magicdec::df_exp_diff(a[i], b[i]);
        hi[i] = e.hi;
        lo[i] = e.lo;
    }
}

int main() {
    // b over several magnitudes and signs; a = b - delta with delta dense over
    // [0, 90] (the cut-off at 87 included) plus pseudo-random deltas.
    const float bs[] = {-30.f, -1.5f, 0.f, 0.37f, 1.f, 5.f, 12.25f, 40.f, 88.f, 1000.5f};
    std::vector<float> a, b;
    uint64_t st = 0x9e3779b97f4a7c15ull;
    for (float bv : bs) {
        for (int i = 0; i <= 9000; ++i) {
            b.push_back(bv);
            a.push_back(bv - 0.01f * (float)i);
        }
        for (int i = 0; i < 20000; ++i) {
            st = st * 6364136223846793005ull + 1442695040888963407ull;
            const float u = (float)((st >> 40) & 0xffffff) / 16777216.0f;
            b.push_back(bv);
            a.push_back(bv - 90.f * u * u);
        }
    }
    const int n = (int)a.size();
    float *da, *db, *dh, *dl;
    if (cudaMalloc(&da, n * 4) || cudaMalloc(&db, n * 4) || cudaMalloc(&dh, n * 4) || cudaMalloc(&dl, n * 4)) return 2;
    cudaMemcpy(da, a.data(), n * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(db, b.data(), n * 4, cudaMemcpyHostToDevice);
    exp_diff_kernel<<<(n + 255) / 256, 256>>>(da, db, dh, dl, n);
    if (cudaDeviceSynchronize() != cudaSuccess) return 2;
    std::vector<float> hi(n), lo(n);
    cudaMemcpy(hi.data(), dh, n * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(lo.data(), dl, n * 4, cudaMemcpyDeviceToHost);
    // Down to exp(-70) the low part is a normal float: 1e-11 relative.  Below it
    // the low part goes subnormal and the value is under 4e-31 of the row's
    // largest term (1): there, and past the cut-off at -87 (result 0), the
    // error must stay under an absolute 2e-38.
    long double max_rel = 0.0L, worst_d = 0.0L, max_abs_tail = 0.0L;
    int checked = 0, tail = 0;
    for (int i = 0; i < n; ++i) {
        const long double d = (long double)a[i] - (long double)b[i];
        const long double got = (long double)hi[i] + (long double)lo[i];
        const long double ref = expl(d);
        if (d < -70.0L) {
            const long double ab = fabsl(got - ref);
            if (ab > max_abs_tail) max_abs_tail = ab;
            ++tail;
            continue;
        }
        const long double rel = fabsl(got - ref) / ref;
        if (rel > max_rel) { max_rel = rel; worst_d = d; }
        ++checked;
    }
    printf("checked %d max_rel %.3Le at a-b %.6Lf; tail %d max_abs %.3Le\n", checked, max_rel, worst_d, tail,
           max_abs_tail);

    // df_div on normalised double-float pairs over magnitudes 2^-40 .. 2^40:
    // 1e-13 relative against long double.
    const int m = 200000;
    std::vector<float> ah(m), al(m), bh(m), bl(m), qh(m), ql(m);
    std::vector<long double> av(m), bv(m);
    for (int i = 0; i < m; ++i) {
        for (int w = 0; w < 2; ++w) {
            st = st * 6364136223846793005ull + 1442695040888963407ull;
            const double frac = 1.0 + (double)(st >> 11) / 9007199254740992.0;          // [1, 2), 53 bits
            st = st * 6364136223846793005ull + 1442695040888963407ull;
            const double x = frac * std::ldexp(1.0, (int)((st >> 33) % 80) - 40);
            const float h = (float)x, l = (float)(x - (double)h);
            (w ? bh : ah)[i] = h;
            (w ? bl : al)[i] = l;
            (w ? bv : av)[i] = (long double)h + (long double)l;
        }
    }
    float *dah, *dal, *dbh, *dbl, *dqh, *dql;
    if (cudaMalloc(&dah, m * 4) || cudaMalloc(&dal, m * 4) || cudaMalloc(&dbh, m * 4) || cudaMalloc(&dbl, m * 4) ||
        cudaMalloc(&dqh, m * 4) || cudaMalloc(&dql, m * 4))
        return 2;
    cudaMemcpy(dah, ah.data(), m * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dal, al.data(), m * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dbh, bh.data(), m * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dbl, bl.data(), m * 4, cudaMemcpyHostToDevice);
    div_kernel<<<(m + 255) / 256, 256>>>(dah, dal, dbh, dbl, dqh, dql, m);
    if (cudaDeviceSynchronize() != cudaSuccess) return 2;
    cudaMemcpy(qh.data(), dqh, m * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(ql.data(), dql, m * 4, cudaMemcpyDeviceToHost);
    long double max_rel_div = 0.0L;
    for (int i = 0; i < m; ++i) {
        const long double ref = av[i] / bv[i];
        const long double rel = fabsl(((long double)qh[i] + (long double)ql[i]) - ref) / fabsl(ref);
        if (rel > max_rel_div) max_rel_div = rel;
    }
    printf("div checked %d max_rel %.3Le\n", m, max_rel_div);
    return (max_rel < 1e-11L && max_abs_tail < 2e-38L && max_rel_div < 1e-13L) ? 0 : 1;
}
