// gla_value_prep: the value-side half of the bilinear gate G_t = alpha_t^T beta_t
// ("Gated Linear Attention Transformers with Hardware-Efficient Training",
// §4.1 Table 1, DFW row; the chunkwise form of its appendix on the general
// formulation, with D' = d_end / d_r and D^dagger = d_r / d_start).
//
// For chunk n and value column j, with B'_r[j] the in-chunk inclusive
// cumulative log beta (B'_{-1} = 0) and B'_C[j] its value at the chunk's end,
// the chunk pass needs
//   V^_r[j] = v_r[j] exp(B'_C[j] - B'_r[j])        (= V (.) D', every factor <= 1)
//   B'_C[j]                                          (the column decay gamma' = exp(B'_C))
// and then forms
//   O_r[j]  = exp(B'_r[j] - B'_C[j]) ( ((Q (.) Lambda) S_[n-1] Diag(gamma'))[r][j] + (P V^)[r][j] ),
//   S_[n]   = Diag(gamma) S_[n-1] Diag(gamma') + (K (.) Gamma)^T V^.
// One reference per chunk, at its end, serves the state and the intra
// product alike. In exact arithmetic this equals the recurrence; in floating
// point it stays exact to rounding while every partial sum of log beta inside
// the chunk is within e^kVGuard, so that exp(B'_r - B'_C) neither overflows
// nor V^ underflows. A head with any chunk beyond that is flagged, and the
// exact CUDA-core pass computes that head instead.
//
// One CTA covers 128 columns of one chunk of one (b,h); each thread walks
// its two columns from the chunk's last row back to its first, so the
// suffix sums need no second pass. Rows at or past T are neither read nor
// written (the chunk pass fills them with zeros on load).
#include <cuda_bf16.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int VT = kDvTile / 2;   // threads per CTA, two columns each
constexpr int RB = 16;            // rows loaded per batch

struct VArgs {
    const __nv_bfloat16* v;   // [BH][T][dv]
    const float* log_b;       // [BH][T][dv]
    __nv_bfloat16* vh;        // [BH][T][dv]   V (.) D'
    float* lbc;               // [BH][nchunks][dv]  B'_C
    int* flag;                // [BH], zeroed before the launch
    int T, dv, nchunks;
};

__global__ void __launch_bounds__(VT) gla_value_prep_kernel(VArgs a)
{
    const int j = blockIdx.x * kDvTile + 2 * threadIdx.x;
    const int c = blockIdx.y, bh = blockIdx.z;
    const int t0 = c * kChunk;
    const int nr = min(kChunk, a.T - t0);
    const size_t base = ((size_t)bh * a.T + t0) * a.dv + j;
    const float* lb = a.log_b + base;
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(a.v + base);
    __nv_bfloat162* vh = reinterpret_cast<__nv_bfloat162*>(a.vh + base);
    const size_t rs = a.dv / 2;   // row stride in column pairs
    float s0 = 0.f, s1 = 0.f;     // sum of log beta over the rows after the current one
    float m = 0.f;                // largest |partial sum| seen
    for (int r1 = nr; r1 > 0; r1 -= RB) {
        float2 x[RB];
        __nv_bfloat162 y[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const int r = r1 - 1 - i;
            if (r >= 0) {
                x[i] = make_float2(lb[(size_t)r * a.dv], lb[(size_t)r * a.dv + 1]);
                y[i] = v[r * rs];
            }
        }
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const int r = r1 - 1 - i;
            if (r >= 0) {
                const float2 f = __bfloat1622float2(y[i]);
                vh[r * rs] = __floats2bfloat162_rn(f.x * expf(s0), f.y * expf(s1));
                s0 += x[i].x;
                s1 += x[i].y;
                m = fmaxf(m, fmaxf(fabsf(s0), fabsf(s1)));
            }
        }
    }
    float* out = a.lbc + ((size_t)bh * a.nchunks + c) * a.dv + j;
    out[0] = s0;
    out[1] = s1;
    if (!(m <= kVGuard)) a.flag[bh] = 1;   // also catches NaN
}

}  // namespace

cudaError_t launch_value_prep(const gla_fwd_params& p, const Plan& pl, void* ws, cudaStream_t s)
{
    uint8_t* base = static_cast<uint8_t*>(ws);
    const int BH = p.B * p.H;
    VArgs a;
    a.v = static_cast<const __nv_bfloat16*>(p.v);
    a.log_b = p.log_b;
    a.vh = reinterpret_cast<__nv_bfloat16*>(base + pl.off_vh);
    a.lbc = reinterpret_cast<float*>(base + pl.off_lbc);
    a.flag = reinterpret_cast<int*>(base + pl.off_flag);
    a.T = p.T; a.dv = p.dv; a.nchunks = pl.nchunks;
    cudaError_t e = cudaMemsetAsync(a.flag, 0, (size_t)BH * sizeof(int), s);
    if (e != cudaSuccess) return e;
    gla_value_prep_kernel<<<dim3(p.dv / kDvTile, pl.nchunks, BH), VT, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gla
