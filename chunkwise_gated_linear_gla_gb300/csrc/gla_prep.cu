// gla_chunk_prep: the per-chunk, dv-independent part of the chunkwise GLA
// forward pass ("Gated Linear Attention Transformers with Hardware-Efficient
// Training", §4.2-4.3). One CTA per (b, h, chunk of C = 64 rows):
//
//   Bc     in-chunk inclusive cumulative log gate (fp32, on chip only)
//   Qt     = Q (.) Lambda,  Lambda_r = exp(Bc_r)            -> workspace, bf16
//   Kt     = K (.) Gamma,   Gamma_r  = exp(Bc_end - Bc_r)   -> workspace, bf16
//   gamma  = exp(Bc_end)                                    -> workspace, fp32
//   A      = (P (.) M), P_rs = sum_k Q_rk K_sk exp(Bc_rk - Bc_sk), r >= s
//                                                            -> workspace, bf16
//
// The intra-chunk scores follow the secondary chunking of §4.3 with
// sub-chunks of c = 16 rows. For a query sub-chunk j and an earlier key
// sub-chunk u (j > u) the factors are referenced to the first row of j
// (f_j) and the last row of u (l_u):
//     P_ju = (Q_j (.) exp(Bc - f_j)) Diag(exp(f_j - l_u)) (K_u (.) exp(l_u - Bc))^T,
// where every exponent is <= 0, so nothing overflows however steep the gate
// (the paper's P_[i][j] with Lambda, Gamma and b_iC / b_(j+1)C). These run on
// the tensor cores (mma.sync, bf16 in, fp32 accumulate).
// A diagonal block (j = u) needs exp(Bc_r - Bc_s) for r >= s inside one
// sub-chunk; the same factors give it with a per-key scale exp(f_j - l_j) >= 1.
// While that scale stays below exp(kGuard) the product cannot overflow and is
// exact to rounding. A key column whose log gate falls by more than kGuard
// inside one sub-chunk is taken out of the MMA and added pairwise in fp32 log
// space instead (Eq. 4), which is the paper's full-precision intra-sub-chunk
// rule, applied only where it is needed.
#include <cuda_bf16.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int C = kChunk;
constexpr int SC = 16;                 // sub-chunk rows
constexpr int NSUB = C / SC;           // 4
constexpr int NPAIR = NSUB * (NSUB + 1) / 2;   // 10 lower (j >= u) blocks
constexpr int NTRI = SC * (SC + 1) / 2;        // 136 pairs r >= s in a block
constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr float kGuard = 60.f;

struct PrepArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const float* log_g;
    __nv_bfloat16* Qt;
    __nv_bfloat16* Kt;
    float* gam;
    __nv_bfloat16* A;
    int H, T, dk, nchunks, Tpad, gate;
};

__device__ __forceinline__ int pair_index(int j, int u) { return j * (j + 1) / 2 + u; }

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t x, float w0, float w1) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&x);
    float2 f = __bfloat1622float2(v);
    __nv_bfloat162 r = __floats2bfloat162_rn(f.x * w0, f.y * w1);
    return *reinterpret_cast<uint32_t*>(&r);
}

__global__ void __launch_bounds__(NT, 2) gla_chunk_prep_kernel(PrepArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int dk = a.dk;
    const int LD = dk + 8;  // bf16 row stride: 4-word skew keeps mma fragment loads conflict-free
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem);           // [C][LD]  Q (.) exp(Bc - f_j)
    __nv_bfloat16* Ks = Qs + C * LD;                                      // [C][LD]  K (.) exp(l_u - Bc)
    float* W = reinterpret_cast<float*>(Ks + C * LD);                     // [NPAIR][dk] exp(f_j - l_u)
    float* part = W + NPAIR * dk;                                         // [NWARP][NSUB][NTRI]
    int* steep_any = reinterpret_cast<int*>(part + NWARP * NSUB * NTRI);  // [NSUB]

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int c = blockIdx.x, bh = blockIdx.y, h = bh % a.H;
    const int t0 = c * C;
    const int nr = min(C, a.T - t0);
    const bool gated = a.gate != GLA_GATE_NONE;

    if (tid < NSUB) steep_any[tid] = 0;
    __syncthreads();

    // ---------------- phase 1: one thread per key column
    const int kk = tid;
    const bool active = kk < dk;
    float Bc[C];
    float f[NSUB], l[NSUB];
    bool steep[NSUB];
    if (active) {
        float run = 0.f;
        const float lam = (a.gate == GLA_GATE_HEAD_SCALAR) ? a.log_g[h] : 0.f;
        const float* g = (a.gate == GLA_GATE_PER_KEY) ? a.log_g + ((size_t)bh * a.T + t0) * dk + kk : nullptr;
#pragma unroll
        for (int r = 0; r < C; ++r) {
            float gl = 0.f;
            if (r < nr) gl = g ? __ldg(g + (size_t)r * dk) : lam;
            run += gl;
            Bc[r] = run;
        }
        const float gend = Bc[C - 1];
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
            f[j] = Bc[j * SC];
            l[j] = Bc[j * SC + SC - 1];
        }
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
#pragma unroll
            for (int u = 0; u <= j; ++u) {
                float w;
                if (u < j) {
                    w = __expf(f[j] - l[u]);
                } else {
                    steep[j] = (f[j] - l[j]) > kGuard;
                    w = steep[j] ? 0.f : __expf(f[j] - l[j]);
                }
                W[pair_index(j, u) * dk + kk] = w;
            }
            if (steep[j]) atomicOr(&steep_any[j], 1);
        }
        if (gated) a.gam[((size_t)bh * a.nchunks + c) * dk + kk] = __expf(gend);

        const __nv_bfloat16* qp = a.q + ((size_t)bh * a.T + t0) * dk + kk;
        const __nv_bfloat16* kp = a.k + ((size_t)bh * a.T + t0) * dk + kk;
        __nv_bfloat16* qo = a.Qt + ((size_t)bh * a.Tpad + t0) * dk + kk;
        __nv_bfloat16* ko = a.Kt + ((size_t)bh * a.Tpad + t0) * dk + kk;
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
            const float ef = __expf(f[j]);          // Lambda at the sub-chunk's first row
            const float eg = __expf(gend - l[j]);   // Gamma at the sub-chunk's last row
#pragma unroll
            for (int i = 0; i < SC; ++i) {
                const int r = j * SC + i;
                float qv = 0.f, kv = 0.f;
                if (r < nr) {
                    qv = __bfloat162float(qp[(size_t)r * dk]);
                    kv = __bfloat162float(kp[(size_t)r * dk]);
                }
                const float e1 = __expf(Bc[r] - f[j]);   // <= 1
                const float e2 = __expf(l[j] - Bc[r]);   // <= 1
                const float qs = qv * e1, ks = kv * e2;
                Qs[r * LD + kk] = __float2bfloat16_rn(qs);
                Ks[r * LD + kk] = __float2bfloat16_rn(ks);
                if (gated) {
                    qo[(size_t)r * dk] = __float2bfloat16_rn(qs * ef);
                    ko[(size_t)r * dk] = __float2bfloat16_rn(ks * eg);
                }
            }
        }
    }

    // exact log-space scores for steep key columns of diagonal blocks
#pragma unroll 1
    for (int j = 0; j < NSUB; ++j) {
        const bool mine = active && steep[j];
        float* pw = part + (warp * NSUB + j) * NTRI;
        if (__any_sync(0xffffffffu, mine)) {
            float qv[SC], kv[SC], bc[SC];
            const float* g = (a.gate == GLA_GATE_PER_KEY) ? a.log_g + ((size_t)bh * a.T + t0) * dk + kk : nullptr;
            const float lam = (a.gate == GLA_GATE_HEAD_SCALAR) ? a.log_g[h] : 0.f;
            float run = 0.f;
#pragma unroll
            for (int i = 0; i < SC; ++i) {
                const int r = j * SC + i;
                qv[i] = kv[i] = 0.f;
                float gl = 0.f;
                if (mine && r < nr) {
                    qv[i] = __bfloat162float(a.q[((size_t)bh * a.T + t0 + r) * dk + kk]);
                    kv[i] = __bfloat162float(a.k[((size_t)bh * a.T + t0 + r) * dk + kk]);
                    gl = g ? g[(size_t)r * dk] : lam;
                }
                // cumulative log gate inside the sub-chunk; only differences are used
                run += gl;
                bc[i] = run;
            }
#pragma unroll
            for (int r = 0; r < SC; ++r) {
#pragma unroll
                for (int s = 0; s <= r; ++s) {
                    float v = mine ? qv[r] * kv[s] * __expf(bc[r] - bc[s]) : 0.f;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) pw[r * (r + 1) / 2 + s] = v;
                }
            }
        } else {
            for (int p = lane; p < NTRI; p += 32) pw[p] = 0.f;
        }
    }
    __syncthreads();

    // ---------------- phase 2: lower blocks of A on the tensor cores
    __nv_bfloat16* Ao = a.A + ((size_t)bh * a.nchunks + c) * C * C;
    const int g8 = lane / 4, c4 = lane % 4;
    for (int blk = warp; blk < NPAIR; blk += NWARP) {
        int j = 0;
        while ((j + 1) * (j + 2) / 2 <= blk) ++j;
        const int u = blk - j * (j + 1) / 2;
        const float* w = W + blk * dk;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const __nv_bfloat16* qa = Qs + (j * SC + g8) * LD + 2 * c4;
        for (int k0 = 0; k0 < dk; k0 += 16) {
            const uint32_t a0 = *reinterpret_cast<const uint32_t*>(qa + k0);
            const uint32_t a1 = *reinterpret_cast<const uint32_t*>(qa + 8 * LD + k0);
            const uint32_t a2 = *reinterpret_cast<const uint32_t*>(qa + k0 + 8);
            const uint32_t a3 = *reinterpret_cast<const uint32_t*>(qa + 8 * LD + k0 + 8);
            const float2 w01 = *reinterpret_cast<const float2*>(w + k0 + 2 * c4);
            const float2 w89 = *reinterpret_cast<const float2*>(w + k0 + 2 * c4 + 8);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const __nv_bfloat16* kb = Ks + (u * SC + nt * 8 + g8) * LD + 2 * c4 + k0;
                uint32_t b0 = *reinterpret_cast<const uint32_t*>(kb);
                uint32_t b1 = *reinterpret_cast<const uint32_t*>(kb + 8);
                if (gated) {
                    b0 = scale_bf16x2(b0, w01.x, w01.y);
                    b1 = scale_bf16x2(b1, w89.x, w89.y);
                }
                mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
            }
        }
        const bool diag = (j == u);
        const bool corr = diag && steep_any[j];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int rl = g8 + hr * 8;               // row within the block
                const int sl = nt * 8 + 2 * c4;           // first of two columns
                float v0 = acc[nt][hr * 2 + 0], v1 = acc[nt][hr * 2 + 1];
                if (diag) {
                    if (corr) {
                        for (int wq = 0; wq < NWARP; ++wq) {
                            const float* pw = part + (wq * NSUB + j) * NTRI;
                            if (sl <= rl) v0 += pw[rl * (rl + 1) / 2 + sl];
                            if (sl + 1 <= rl) v1 += pw[rl * (rl + 1) / 2 + sl + 1];
                        }
                    }
                    if (sl > rl) v0 = 0.f;
                    if (sl + 1 > rl) v1 = 0.f;
                }
                __nv_bfloat162 o = __floats2bfloat162_rn(v0, v1);
                *reinterpret_cast<__nv_bfloat162*>(Ao + (j * SC + rl) * C + u * SC + sl) = o;
            }
        }
    }
    // upper blocks (j < u) are zero
    for (int idx = tid; idx < C * C / 2; idx += NT) {
        const int r = idx / (C / 2), s = (idx % (C / 2)) * 2;
        if (s / SC > r / SC) *reinterpret_cast<uint32_t*>(Ao + r * C + s) = 0u;
    }
}

size_t prep_smem_bytes(int dk) {
    return (size_t)2 * C * (dk + 8) * 2 + (size_t)NPAIR * dk * 4 + (size_t)NWARP * NSUB * NTRI * 4 + NSUB * 4;
}

}  // namespace

cudaError_t launch_prep(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s)
{
    (void)status;
    uint8_t* base = static_cast<uint8_t*>(ws);
    PrepArgs a;
    a.q = static_cast<const __nv_bfloat16*>(p.q);
    a.k = static_cast<const __nv_bfloat16*>(p.k);
    a.log_g = p.log_g;
    a.Qt = pl.raw_qk ? nullptr : reinterpret_cast<__nv_bfloat16*>(base + pl.off_qt);
    a.Kt = pl.raw_qk ? nullptr : reinterpret_cast<__nv_bfloat16*>(base + pl.off_kt);
    a.gam = reinterpret_cast<float*>(base + pl.off_gam);
    a.A = reinterpret_cast<__nv_bfloat16*>(base + pl.off_A);
    a.H = p.H; a.T = p.T; a.dk = p.dk; a.nchunks = pl.nchunks; a.Tpad = pl.Tpad; a.gate = p.gate;
    const size_t smem = prep_smem_bytes(p.dk);
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(pl.nchunks, p.B * p.H);
    gla_chunk_prep_kernel<<<grid, NT, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gla
