// Kernels of the sequence exchange: one long sequence cut into P segments
// (one per device, or per call), each run from a zero state, then chained.
//
// Because the recurrence S_t = Diag(alpha_t) S_(t-1) + k_t^T v_t is linear in
// S and the gate only scales rows, a segment started from S_in leaves
//
//     S_out = Diag(Gamma) S_in + S*,   Gamma = prod over the segment of alpha_t,
//
// where S* is what the segment leaves from a zero start ("Gated Linear
// Attention Transformers with Hardware-Efficient Training", §2.2: the state
// S_[0] handed from one segment to the next; the FlashQLA talk, "core technical
// principles": a wrongly started segment is corrected by one matrix per rank,
// then a short serial recurrence over ranks). The pair (Gamma, S*) therefore
// describes a segment completely, and two neighbours compose as
//
//     (Gamma_2, S*_2) o (Gamma_1, S*_1) = (Gamma_2 Gamma_1, Diag(Gamma_2) S*_1 + S*_2).
//
// Gamma is carried as log Gamma (a per-key sum of log alpha), so that a long
// segment's decay stays representable where the product would underflow.
//
// gla_seg_logsum_*: log Gamma of a segment from the log gate. A CTA sums 32
// key columns over a 1024-token slice in fp64 (eight warps of 128 tokens, a
// fixed order), then one thread per key adds the slices in order: the result
// is the same on every run.
// gla_pair_scan_kernel: the serial recurrence over P pairs, one thread per
// state element. gla_pair_combine_kernel: one composition, in place.
#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kSliceTok = 1024;   // tokens per CTA of the partial sums
constexpr int kWarpTok = 128;     // tokens per warp
constexpr int NT = 256;

// part[slice][bh][col] = sum of log_g[bh][t][col] over the slice's tokens.
// width = dk (per-key gate) or 1 (per-token scalar gate).
__global__ void __launch_bounds__(NT) gla_seg_logsum_partial(const float* __restrict__ lg, int T, int width,
                                                            double* __restrict__ part, long long BH)
{
    __shared__ double red[NT / 32][32];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int col = blockIdx.x * 32 + lane;
    const long long bh = blockIdx.y;
    const int slice = blockIdx.z;
    const int t0 = slice * kSliceTok + warp * kWarpTok;
    const int t1 = min(T, t0 + kWarpTok);
    double acc = 0.0;
    if (col < width) {
        const float* p = lg + ((size_t)bh * T) * width + col;
        int t = t0;
        // eight loads in flight per lane
        for (; t + 8 <= t1; t += 8) {
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = __ldg(p + (size_t)(t + i) * width);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc += (double)x[i];
        }
        for (; t < t1; ++t) acc += (double)__ldg(p + (size_t)t * width);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && col < width) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) s += red[w][lane];
        part[((size_t)slice * BH + bh) * width + col] = s;
    }
}

// log_Gamma[bh][k] from the slices' partial sums (width = dk: column k; width = 1:
// the per-token sum, the same for every key). Per-head scalar gate (part = null):
// T log(lambda_h).
__global__ void __launch_bounds__(NT) gla_seg_logsum_final(const double* __restrict__ part, int nslice, int width,
                                                          const float* __restrict__ log_lambda, int H, int T,
                                                          int dk, long long BH, float* __restrict__ out)
{
    const long long i = (long long)blockIdx.x * NT + threadIdx.x;
    if (i >= BH * dk) return;
    const long long bh = i / dk;
    const int k = (int)(i % dk);
    double s = 0.0;
    if (part) {
        const int col = width == 1 ? 0 : k;
        for (int sl = 0; sl < nslice; ++sl) s += part[((size_t)sl * BH + bh) * width + col];
    } else if (log_lambda) {
        s = (double)T * (double)log_lambda[bh % H];
    }
    out[i] = (float)s;
}

// S_in[d] = the state entering segment d, S_T = the state after the last one:
//   S = S0 (or 0); for d = 0..P-1: S_in[d] = S, S = exp(log_Gamma[d]) (.) S + S*[d].
// S*[d] is read before S_in[d] is written, so S_in may be S_star itself.
__global__ void __launch_bounds__(NT) gla_pair_scan_kernel(int P, const float* log_G, const float* S_star,
                                                          const float* S0, float* S_in, float* S_T,
                                                          long long BH, int dk, int dv)
{
    const long long st = (long long)dk * dv;
    const long long n = BH * st;
    for (long long e = (long long)blockIdx.x * NT + threadIdx.x; e < n; e += (long long)gridDim.x * NT) {
        const long long bh = e / st;
        const int k = (int)((e % st) / dv);
        float S = S0 ? S0[e] : 0.f;
        for (int d = 0; d < P; ++d) {
            const float cur = S_star[(size_t)d * n + e];
            const float g = expf(log_G[((size_t)d * BH + bh) * dk + k]);
            if (S_in) S_in[(size_t)d * n + e] = S;
            S = fmaf(g, S, cur);
        }
        if (S_T) S_T[e] = S;
    }
}

// (log_G1, S1) <- (log_G2, S2) o (log_G1, S1) = (log_G2 + log_G1, exp(log_G2) (.) S1 + S2).
__global__ void __launch_bounds__(NT) gla_pair_combine_kernel(const float* log_G2, const float* S2, float* log_G1,
                                                             float* S1, long long BH, int dk, int dv)
{
    const long long st = (long long)dk * dv;
    const long long n = BH * st;
    for (long long e = (long long)blockIdx.x * NT + threadIdx.x; e < n; e += (long long)gridDim.x * NT) {
        const long long bh = e / st;
        const long long r = e % st;
        const int k = (int)(r / dv), j = (int)(r % dv);
        const float lg2 = log_G2[bh * dk + k];
        S1[e] = fmaf(expf(lg2), S1[e], S2[e]);
        if (j == 0) log_G1[bh * dk + k] += lg2;
    }
}

unsigned grid_for(long long n, int sms)
{
    long long b = (n + NT - 1) / NT;
    const long long cap = (long long)(sms > 0 ? sms : 148) * 8;
    if (b > cap) b = cap;
    return (unsigned)(b < 1 ? 1 : b);
}

}  // namespace

size_t seg_logsum_ws_bytes(const gla_fwd_params& p)
{
    if (p.T == 0 || (p.gate != GLA_GATE_PER_KEY && p.gate != GLA_GATE_TOKEN_SCALAR)) return 0;
    const int width = p.gate == GLA_GATE_PER_KEY ? p.dk : 1;
    const size_t nslice = ((size_t)p.T + kSliceTok - 1) / kSliceTok;
    return nslice * (size_t)p.B * p.H * width * sizeof(double);
}

cudaError_t launch_seg_logsum(const gla_fwd_params& p, float* log_Gamma, void* ws, cudaStream_t s)
{
    const long long BH = (long long)p.B * p.H;
    const size_t nout = (size_t)BH * p.dk * sizeof(float);
    if (p.T == 0 || p.gate == GLA_GATE_NONE) return cudaMemsetAsync(log_Gamma, 0, nout, s);
    const unsigned fin_blocks = (unsigned)((BH * p.dk + NT - 1) / NT);
    if (p.gate == GLA_GATE_HEAD_SCALAR) {
        gla_seg_logsum_final<<<fin_blocks, NT, 0, s>>>(nullptr, 0, 1, p.log_g, p.H, p.T, p.dk, BH, log_Gamma);
        return cudaGetLastError();
    }
    if (p.gate != GLA_GATE_PER_KEY && p.gate != GLA_GATE_TOKEN_SCALAR) return cudaErrorInvalidValue;
    const int width = p.gate == GLA_GATE_PER_KEY ? p.dk : 1;
    const int nslice = (p.T + kSliceTok - 1) / kSliceTok;
    if (BH > 65535 || nslice > 65535) return cudaErrorInvalidValue;
    double* part = static_cast<double*>(ws);
    dim3 grid((unsigned)((width + 31) / 32), (unsigned)BH, (unsigned)nslice);
    gla_seg_logsum_partial<<<grid, NT, 0, s>>>(p.log_g, p.T, width, part, BH);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    gla_seg_logsum_final<<<fin_blocks, NT, 0, s>>>(part, nslice, width, nullptr, p.H, p.T, p.dk, BH, log_Gamma);
    return cudaGetLastError();
}

cudaError_t launch_pair_scan(int P, const float* log_G, const float* S_star, const float* S0, float* S_in,
                             float* S_T, long long BH, int dk, int dv, int sms, cudaStream_t s)
{
    gla_pair_scan_kernel<<<grid_for(BH * dk * dv, sms), NT, 0, s>>>(P, log_G, S_star, S0, S_in, S_T, BH, dk, dv);
    return cudaGetLastError();
}

cudaError_t launch_pair_combine(const float* log_G2, const float* S2, float* log_G1, float* S1, long long BH,
                                int dk, int dv, int sms, cudaStream_t s)
{
    gla_pair_combine_kernel<<<grid_for(BH * dk * dv, sms), NT, 0, s>>>(log_G2, S2, log_G1, S1, BH, dk, dv);
    return cudaGetLastError();
}

}  // namespace gla
