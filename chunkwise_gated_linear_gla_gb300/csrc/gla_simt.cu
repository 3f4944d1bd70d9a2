// CUDA-core (fp32 FFMA) forward pass of chunkwise gated linear attention.
//
// This is the path for fp32 inputs (where the result must hold to ~1e-5) and
// for bf16 shapes the tensor-core path does not take. It follows the
// chunkwise form of "Gated Linear Attention Transformers with
// Hardware-Efficient Training", §4.2, with chunks of 16 rows (8 for keys
// wider than 256, whose state tiles take more shared memory):
//   Lambda_r = b_r / b_start, Gamma_r = b_end / b_r, gamma = b_end / b_start,
//   O_chunk = (Q (.) Lambda) S + (P (.) M) V,
//   S      <- (gamma^T 1) (.) S + (K (.) Gamma)^T V,
// where the intra-chunk scores P are evaluated pairwise in fp32 log space,
//   P_rs = sum_k Q_rk K_sk exp(logB_rk - logB_sk),  r >= s
// (same paper, §4.1 Eq. 4, the "intra-sub-chunk in full precision" part of
// §4.3). Every exponent is <= 0, so no factor exceeds 1 and no gate, however
// steep, overflows. Each CTA owns one (b,h) and 64 columns of dv (32 for
// keys wider than 256); columns of S are independent because the gate scales
// rows only.
//
// The bilinear gate G_t = alpha_t^T beta_t (Table 1's DFW row) adds a decay of
// the value columns: with B'_r the in-chunk cumulative log beta of column j,
//   O_chunk[r][j] = exp(B'_r[j]) ((Q (.) Lambda) S)[r][j]
//                   + sum_{s<=r} P_rs v_s[j] exp(B'_r[j] - B'_s[j]),
//   S[k][j] <- gamma[k] gamma'[j] S[k][j] + sum_r (K (.) Gamma)[r][k] v_r[j] exp(B'_end[j] - B'_r[j]),
// every exponent again <= 0.
#include <cuda_bf16.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int NT = 256;

struct SimtArgs {
    const void* q; const void* k; const void* v;
    const float* log_g; const float* log_b; const float* S0;
    void* O; float* ST;
    const int* only;   // null, or per-head flags: compute only the heads whose flag is set
    int B, H, T, dk, dv, gate;
};

template <typename T> __device__ __forceinline__ float ld_in(const T* p, size_t i);
template <> __device__ __forceinline__ float ld_in<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ void st_out(T* p, size_t i, float x);
template <> __device__ __forceinline__ void st_out<float>(float* p, size_t i, float x) { p[i] = x; }
template <> __device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16* p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// CS rows per chunk and DVT state columns per CTA: 16 and 64 for dk <= 256;
// for wider keys 8 and 32, so that the fp32 state tile and the chunk's key
// rows still fit in shared memory (dk up to kSimtMaxDk).
template <typename Tin, int CS, int DVT>
__global__ void __launch_bounds__(NT) gla_fwd_simt_kernel(SimtArgs a)
{
    extern __shared__ float smem[];
    const int dk = a.dk;
    float* S   = smem;                 // [dk][DVT]
    float* qr  = S + dk * DVT;         // [CS][dk] raw q
    float* kr  = qr + CS * dk;         // [CS][dk] raw k
    float* bc  = kr + CS * dk;         // [CS][dk] in-chunk cumulative log gate
    float* qt  = bc + CS * dk;         // [CS][dk] q (.) Lambda
    float* kt  = qt + CS * dk;         // [CS][dk] k (.) Gamma
    float* vv  = kt + CS * dk;         // [CS][DVT]
    float* A   = vv + CS * DVT;        // [CS][CS] masked intra scores
    float* gam = A + CS * CS;          // [dk] chunk decay gamma
    float* bcv = gam + dk;             // [CS][DVT] in-chunk cumulative log beta (bilinear gate)
    float* vg  = bcv + CS * DVT;       // [CS][DVT] v (.) Gamma' (bilinear gate)
    float* gv  = vg + CS * DVT;        // [DVT] chunk decay gamma' of the columns (bilinear gate)
    const bool bil = a.gate == GLA_GATE_BILINEAR;

    const int tid = threadIdx.x;
    const int bh = blockIdx.x;
    if (a.only && a.only[bh] == 0) return;
    const int h = bh % a.H;
    const int j0 = blockIdx.y * DVT;
    const int jn = min(DVT, a.dv - j0);
    const Tin* q = static_cast<const Tin*>(a.q) + (size_t)bh * a.T * dk;
    const Tin* k = static_cast<const Tin*>(a.k) + (size_t)bh * a.T * dk;
    const Tin* v = static_cast<const Tin*>(a.v) + (size_t)bh * a.T * a.dv;
    Tin* O = static_cast<Tin*>(a.O) + (size_t)bh * a.T * a.dv;
    const float* g = (a.gate == GLA_GATE_PER_KEY || bil) ? a.log_g + (size_t)bh * a.T * dk : nullptr;
    const float* lb = bil ? a.log_b + (size_t)bh * a.T * a.dv : nullptr;
    const float* gtok = (a.gate == GLA_GATE_TOKEN_SCALAR) ? a.log_g + (size_t)bh * a.T : nullptr;
    const float lam = (a.gate == GLA_GATE_HEAD_SCALAR) ? a.log_g[h] : 0.f;

    // S <- S0 tile (or 0)
    for (int i = tid; i < dk * DVT; i += NT) {
        int kk = i / DVT, j = i % DVT;
        float s = 0.f;
        if (a.S0 && j < jn) s = a.S0[((size_t)bh * dk + kk) * a.dv + j0 + j];
        S[i] = s;
    }

    const int nch = (a.T + CS - 1) / CS;
    for (int c = 0; c < nch; ++c) {
        const int t0 = c * CS;
        const int nr = min(CS, a.T - t0);
        __syncthreads();  // previous chunk done with every buffer
        for (int i = tid; i < CS * dk; i += NT) {
            int r = i / dk, kk = i % dk;
            bool ok = r < nr;
            qr[i] = ok ? ld_in<Tin>(q, (size_t)(t0 + r) * dk + kk) : 0.f;
            kr[i] = ok ? ld_in<Tin>(k, (size_t)(t0 + r) * dk + kk) : 0.f;
        }
        for (int i = tid; i < CS * DVT; i += NT) {
            int r = i / DVT, j = i % DVT;
            vv[i] = (r < nr && j < jn) ? ld_in<Tin>(v, (size_t)(t0 + r) * a.dv + j0 + j) : 0.f;
        }
        __syncthreads();
        // in-chunk cumulative log gate per key column; padded rows add 0
        for (int kk = tid; kk < dk; kk += NT) {
            float run = 0.f;
            for (int r = 0; r < CS; ++r) {
                float gl = 0.f;
                if (r < nr) {
                    if (g) gl = g[(size_t)(t0 + r) * dk + kk];
                    else if (gtok) gl = gtok[t0 + r];
                    else gl = lam;
                }
                run += gl;
                bc[r * dk + kk] = run;
            }
            const float last = run;
            gam[kk] = expf(last);
            for (int r = 0; r < CS; ++r) {
                const float b = bc[r * dk + kk];
                qt[r * dk + kk] = qr[r * dk + kk] * expf(b);
                kt[r * dk + kk] = kr[r * dk + kk] * expf(last - b);
            }
        }
        if (bil)   // in-chunk cumulative log beta per value column, gamma', and V (.) Gamma'
            for (int j = tid; j < DVT; j += NT) {
                float run = 0.f;
                for (int r = 0; r < CS; ++r) {
                    run += (r < nr && j < jn) ? lb[(size_t)(t0 + r) * a.dv + j0 + j] : 0.f;
                    bcv[r * DVT + j] = run;
                }
                gv[j] = expf(run);
                for (int r = 0; r < CS; ++r) vg[r * DVT + j] = vv[r * DVT + j] * expf(run - bcv[r * DVT + j]);
            }
        __syncthreads();
        // intra-chunk scores, pairwise in log space (r >= s)
        if constexpr (CS * (CS + 1) / 2 >= NT / 2) {
            // one thread per pair
            for (int p = tid; p < CS * (CS + 1) / 2; p += NT) {
                int r = 0;
                while ((r + 1) * (r + 2) / 2 <= p) ++r;
                const int s = p - r * (r + 1) / 2;
                float acc = 0.f;
                const float* qrow = qr + r * dk;
                const float* krow = kr + s * dk;
                const float* br = bc + r * dk;
                const float* bs = bc + s * dk;
                for (int kk = 0; kk < dk; ++kk) acc = fmaf(qrow[kk] * krow[kk], expf(br[kk] - bs[kk]), acc);
                A[r * CS + s] = acc;
            }
        } else {
            // few pairs and wide keys: one warp per pair, its lanes splitting the keys
            const int lane = tid & 31;
            for (int p = tid >> 5; p < CS * (CS + 1) / 2; p += NT / 32) {
                int r = 0;
                while ((r + 1) * (r + 2) / 2 <= p) ++r;
                const int s = p - r * (r + 1) / 2;
                float acc = 0.f;
                for (int kk = lane; kk < dk; kk += 32)
                    acc = fmaf(qr[r * dk + kk] * kr[s * dk + kk], expf(bc[r * dk + kk] - bc[s * dk + kk]), acc);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (lane == 0) A[r * CS + s] = acc;
            }
        }
        __syncthreads();
        // outputs: inter (Q (.) Lambda) S + intra (P (.) M) V
        for (int i = tid; i < CS * DVT; i += NT) {
            const int r = i / DVT, j = i % DVT;
            if (r >= nr || j >= jn) continue;
            float acc = 0.f;
            const float* qrow = qt + r * dk;
            for (int kk = 0; kk < dk; ++kk) acc = fmaf(qrow[kk], S[kk * DVT + j], acc);
            if (bil) {
                const float br = bcv[r * DVT + j];
                acc *= expf(br);
                for (int s = 0; s <= r; ++s)
                    acc = fmaf(A[r * CS + s], vv[s * DVT + j] * expf(br - bcv[s * DVT + j]), acc);
            } else {
                for (int s = 0; s <= r; ++s) acc = fmaf(A[r * CS + s], vv[s * DVT + j], acc);
            }
            st_out<Tin>(O, (size_t)(t0 + r) * a.dv + j0 + j, acc);
        }
        __syncthreads();
        // state: S <- (gamma^T 1) (.) S + (K (.) Gamma)^T V
        // (NT is a multiple of DVT, so a thread's column j is the same for every i)
        static_assert(NT % DVT == 0, "fixed state column per thread");
        const float* vs = bil ? vg : vv;
        const int jt = tid % DVT;
        float vcol[CS];
#pragma unroll
        for (int r = 0; r < CS; ++r) vcol[r] = vs[r * DVT + jt];
        const float gcol = bil ? gv[jt] : 1.f;
        for (int i = tid; i < dk * DVT; i += NT) {
            const int kk = i / DVT;
            float acc = gam[kk] * gcol * S[i];
#pragma unroll
            for (int r = 0; r < CS; ++r) acc = fmaf(kt[r * dk + kk], vcol[r], acc);
            S[i] = acc;
        }
    }
    __syncthreads();
    if (a.ST) {
        for (int i = tid; i < dk * DVT; i += NT) {
            int kk = i / DVT, j = i % DVT;
            if (j < jn) a.ST[((size_t)bh * dk + kk) * a.dv + j0 + j] = S[i];
        }
    }
}

size_t simt_smem_bytes(int dk, int CS, int DVT) {
    return sizeof(float) * ((size_t)dk * DVT + 5 * CS * dk + CS * DVT + CS * CS + dk + 2 * CS * DVT + DVT);
}

template <typename Tin, int CS, int DVT>
cudaError_t launch_cfg(const SimtArgs& a, const gla_fwd_params& p, cudaStream_t s)
{
    const size_t smem = simt_smem_bytes(p.dk, CS, DVT);
    dim3 grid(p.B * p.H, (p.dv + DVT - 1) / DVT);
    cudaError_t e = cudaFuncSetAttribute(gla_fwd_simt_kernel<Tin, CS, DVT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gla_fwd_simt_kernel<Tin, CS, DVT><<<grid, NT, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dtype(const SimtArgs& a, const gla_fwd_params& p, cudaStream_t s)
{
    if (p.dk <= kMaxDk) return launch_cfg<Tin, kSimtChunk, kSimtDvTile>(a, p, s);
    return launch_cfg<Tin, kSimtChunkWide, kSimtDvTileWide>(a, p, s);
}

}  // namespace

cudaError_t launch_simt(const gla_fwd_params& p, int* status, cudaStream_t s, const int* only)
{
    (void)status;
    SimtArgs a;
    a.only = only;
    a.q = p.q; a.k = p.k; a.v = p.v; a.log_g = p.log_g; a.log_b = p.log_b; a.S0 = p.S0; a.O = p.O; a.ST = p.ST;
    a.B = p.B; a.H = p.H; a.T = p.T; a.dk = p.dk; a.dv = p.dv; a.gate = p.gate;
    if (p.dk > kSimtMaxDk) return cudaErrorInvalidValue;
    return p.dtype == GLA_FP32 ? launch_dtype<float>(a, p, s) : launch_dtype<__nv_bfloat16>(a, p, s);
}

}  // namespace gla
