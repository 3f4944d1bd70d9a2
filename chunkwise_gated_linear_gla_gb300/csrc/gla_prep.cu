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
//
// Thread layout of the element-wise phase: thread t owns 8 consecutive key
// columns (one 16-byte vector of bf16) and RPT = dk/32 consecutive rows, so
// every warp reads and writes whole rows with 16-byte accesses. The
// cumulative gate is a two-level scan: a serial sum over the thread's rows,
// then the totals of the row groups above it.
#include <cuda_bf16.h>

#include "gla_internal.h"
#include "sm100.cuh"

namespace gla {
namespace {

constexpr int C = kChunk;
constexpr int SC = 16;                          // sub-chunk rows
constexpr int NSUB = C / SC;                    // 4
constexpr int NPAIR = NSUB * (NSUB + 1) / 2;    // 10 lower (j >= u) blocks
constexpr int NTRI = SC * (SC + 1) / 2;         // 136 pairs r >= s in a block
constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int ALD = C + 8;                      // bf16 row stride of the staged A tile
constexpr float kGuard = 60.f;

struct PrepArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const float* log_g;
    __nv_bfloat16* Qt;
    __nv_bfloat16* Kt;
    float* gam;
    __nv_bfloat16* A;
    int* status;
    int BH, H, T, nchunks, Tpad, gate;
};

constexpr uint64_t kCopyTimeoutNs = 2000000000ull;   // bounded wait for the q/k bulk copies
constexpr int ERR_PREP = 0x201;

template <int DK>
struct PL {
    static constexpr int NCG = DK / 8;          // column groups of 8
    static constexpr int NRG = NT / NCG;        // row groups
    static constexpr int RPT = C / NRG;         // rows per thread (dk / 32)
    static constexpr int QS_OFF = 0;                              // [C][DK] bf16, 16-byte chunks XOR-swizzled by row
    static constexpr int KS_OFF = QS_OFF + C * DK * 2;
    static constexpr int W_OFF = KS_OFF + C * DK * 2;             // [NPAIR][DK] fp32
    static constexpr int X_OFF = W_OFF + NPAIR * DK * 4;          // [2][NRG][DK] fp32 (totals, then first/last)
    static constexpr int CORR_OFF = X_OFF + 2 * NRG * DK * 4;     // [NSUB][NTRI] fp32
    static constexpr int STEEP_OFF = CORR_OFF + NSUB * NTRI * 4;  // [NSUB][DK] u8
    static constexpr int ANY_OFF = STEEP_OFF + NSUB * DK;         // [NSUB] int
    static constexpr int BAR_OFF = (ANY_OFF + 16 + 7) / 8 * 8;    // mbarrier of the q/k bulk copies
    static constexpr int SMEM = BAR_OFF + 16;
    static_assert(RPT >= 1 && SC % RPT == 0, "a thread's rows lie in one sub-chunk");
    static_assert(DK / 8 >= 8, "swizzle needs at least 8 chunks per row");
    static_assert(NCG % 8 == 0 || 32 % NCG == 0, "a warp owns whole rows");
    static_assert(C * ALD * 2 <= 2 * C * DK * 2, "A staging fits in the Q/K tiles");
};

// Element offset of (row, col) in a [C][DK] bf16 tile whose 16-byte chunks are
// XOR-swizzled by (row % 8): rows 8 apart share banks, so the mma fragment
// loads of 8 consecutive rows hit 8 different bank groups.
template <int DK>
__device__ __forceinline__ int swz(int row, int col) {
    return row * DK + ((((col >> 3) ^ (row & 7))) << 3) + (col & 7);
}

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

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}

// Resident CTAs per SM: the kernel is latency-bound, so smaller heads run three
// CTAs per SM (shared memory allows it; registers are bounded to fit).
template <int DK>
constexpr int prep_ctas_per_sm() { return DK <= 128 ? 3 : 2; }

template <int DK>
__global__ void __launch_bounds__(NT, prep_ctas_per_sm<DK>()) gla_chunk_prep_kernel(PrepArgs a)
{
    using L = PL<DK>;
    constexpr int RPT = L::RPT, NRG = L::NRG;
    extern __shared__ __align__(16) uint8_t smem[];
    // Qs/Ks first receive the raw q/k rows of the chunk (bulk copies), then are
    // overwritten in place, swizzled, with Q (.) exp(Bc - f_j) and K (.) exp(l_u - Bc).
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem + L::QS_OFF);
    __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem + L::KS_OFF);
    uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    float* W = reinterpret_cast<float*>(smem + L::W_OFF);                     // [NPAIR][DK] exp(f_j - l_u)
    float* X = reinterpret_cast<float*>(smem + L::X_OFF);
    float* corr = reinterpret_cast<float*>(smem + L::CORR_OFF);               // [NSUB][NTRI]
    uint8_t* steep = smem + L::STEEP_OFF;                                     // [NSUB][DK]
    int* steep_any = reinterpret_cast<int*>(smem + L::ANY_OFF);
    __nv_bfloat16* As = Qs;                                                   // [C][ALD], after the MMAs

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        sm100::mbar_init(cbar, 1);
        sm100::mbar_fence_init();
    }
    __syncthreads();
    // Persistent: work items (b*H+h, chunk) in order, strided by the grid. While
    // one item is computed, the next one's rows are prefetched into L2.
    const int total = a.BH * a.nchunks;
    for (int item = blockIdx.x, it = 0; item < total; item += gridDim.x, ++it) {
    const int c = item % a.nchunks, bh = item / a.nchunks, h = bh % a.H;
    const int t0 = c * C;
    const int nr = min(C, a.T - t0);
    const bool gated = a.gate != GLA_GATE_NONE;
    const int cg = tid % L::NCG, rg = tid / L::NCG;
    const int col0 = cg * 8, row0 = rg * RPT;
    const int j = row0 / SC;   // the sub-chunk this thread's rows lie in
    const float lam = (a.gate == GLA_GATE_HEAD_SCALAR) ? a.log_g[h] : 0.f;

    if (tid < NSUB) steep_any[tid] = 0;
    for (int i = tid; i < NSUB * DK; i += NT) steep[i] = 0;
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)nr * DK * 2;
        sm100::mbar_arrive_expect_tx(cbar, 2 * bytes);
        sm100::bulk_load(Qs, a.q + ((size_t)bh * a.T + t0) * DK, bytes, cbar);
        sm100::bulk_load(Ks, a.k + ((size_t)bh * a.T + t0) * DK, bytes, cbar);
        const int nx = item + gridDim.x;
        if (nx < total) {
            const int c2 = nx % a.nchunks, bh2 = nx / a.nchunks, nr2 = min(C, a.T - c2 * C);
            const size_t row = (size_t)bh2 * a.T + (size_t)c2 * C;
            sm100::prefetch_l2(a.q + row * DK, (uint32_t)nr2 * DK * 2);
            sm100::prefetch_l2(a.k + row * DK, (uint32_t)nr2 * DK * 2);
            if (a.gate == GLA_GATE_PER_KEY) sm100::prefetch_l2(a.log_g + row * DK, (uint32_t)nr2 * DK * 4);
        }
    }
    // rows past the end of the sequence are zero (the copies cover rows < nr only)
    for (int i = nr * DK / 8 + tid; i < C * DK / 8; i += NT) {
        reinterpret_cast<uint4*>(Qs)[i] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(Ks)[i] = make_uint4(0, 0, 0, 0);
    }

    // ---- 1. log gates of my rows and their running sum
    float Bc[RPT][8];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const bool ok = row0 + r < nr;
        if (a.gate == GLA_GATE_PER_KEY) {
            float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
            if (ok) {
                const float4* g = reinterpret_cast<const float4*>(a.log_g + ((size_t)bh * a.T + t0 + row0 + r) * DK + col0);
                x0 = __ldg(g);
                x1 = __ldg(g + 1);
            }
            Bc[r][0] = x0.x; Bc[r][1] = x0.y; Bc[r][2] = x0.z; Bc[r][3] = x0.w;
            Bc[r][4] = x1.x; Bc[r][5] = x1.y; Bc[r][6] = x1.z; Bc[r][7] = x1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) Bc[r][i] = ok ? lam : 0.f;
        }
    }
#pragma unroll
    for (int r = 1; r < RPT; ++r)
#pragma unroll
        for (int i = 0; i < 8; ++i) Bc[r][i] += Bc[r - 1][i];
#pragma unroll
    for (int i = 0; i < 8; ++i) X[rg * DK + col0 + i] = Bc[RPT - 1][i];
    __syncthreads();
    {
        float off[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int rr = 0; rr < rg; ++rr)
#pragma unroll
            for (int i = 0; i < 8; ++i) off[i] += X[rr * DK + col0 + i];
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) Bc[r][i] += off[i];
    }
    __syncthreads();   // totals read by everyone; the region now holds first/last rows
    float* first = X;
    float* last = X + NRG * DK;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        first[rg * DK + col0 + i] = Bc[0][i];
        last[rg * DK + col0 + i] = Bc[RPT - 1][i];
    }
    __syncthreads();

    // ---- 2. sub-chunk references, scaled operands, Q (.) Lambda and K (.) Gamma
    float f[8], l[8], ef[8], eg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[i] = first[(j * SC / RPT) * DK + col0 + i];
        l[i] = last[((j * SC + SC - 1) / RPT) * DK + col0 + i];
        const float gend = last[(NRG - 1) * DK + col0 + i];
        ef[i] = __expf(f[i]);
        eg[i] = __expf(gend - l[i]);
    }
    if (row0 == j * SC) {
        bool any = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool s = (f[i] - l[i]) > kGuard;
            steep[j * DK + col0 + i] = s ? 1 : 0;
            any |= s;
        }
        if (any) atomicOr(&steep_any[j], 1);
    }
    {
        const bool ok = sm100::mbar_wait(cbar, it & 1, kCopyTimeoutNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicExch(a.status, ERR_PREP);
            return;
        }
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int row = row0 + r;
        const uint4 qu = *reinterpret_cast<const uint4*>(Qs + row * DK + col0);
        const uint4 ku = *reinterpret_cast<const uint4*>(Ks + row * DK + col0);
        __syncwarp();   // the warp owns whole rows: all raw reads of this row precede the swizzled writes
        float qv[8], kv[8], qs[8], ks[8];
        unpack8(qu, qv);
        unpack8(ku, kv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            qs[i] = qv[i] * __expf(Bc[r][i] - f[i]);   // factor <= 1
            ks[i] = kv[i] * __expf(l[i] - Bc[r][i]);   // factor <= 1
        }
        *reinterpret_cast<uint4*>(Qs + swz<DK>(row, col0)) = pack8(qs);
        *reinterpret_cast<uint4*>(Ks + swz<DK>(row, col0)) = pack8(ks);
        if (gated) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                qs[i] *= ef[i];
                ks[i] *= eg[i];
            }
            *reinterpret_cast<uint4*>(a.Qt + ((size_t)bh * a.Tpad + t0 + row) * DK + col0) = pack8(qs);
            *reinterpret_cast<uint4*>(a.Kt + ((size_t)bh * a.Tpad + t0 + row) * DK + col0) = pack8(ks);
        }
    }
    for (int p = tid; p < NPAIR * DK; p += NT) {
        const int pr = p / DK, col = p % DK;
        int jj = 0;
        while ((jj + 1) * (jj + 2) / 2 <= pr) ++jj;
        const int uu = pr - jj * (jj + 1) / 2;
        const float fj = first[(jj * SC / RPT) * DK + col];
        const float lu = last[((uu * SC + SC - 1) / RPT) * DK + col];
        float w = __expf(fj - lu);
        if (jj == uu && (fj - lu) > kGuard) w = 0.f;
        W[p] = w;
    }
    if (gated)
        for (int col = tid; col < DK; col += NT)
            a.gam[((size_t)bh * a.nchunks + c) * DK + col] = __expf(last[(NRG - 1) * DK + col]);
    __syncthreads();

    // ---- 3. exact log-space scores for steep key columns of diagonal blocks
#pragma unroll 1
    for (int jj = 0; jj < NSUB; ++jj) {
        if (!steep_any[jj]) continue;   // block-uniform
        for (int p = tid; p < NTRI; p += NT) {
            int r = 0;
            while ((r + 1) * (r + 2) / 2 <= p) ++r;
            const int s = p - r * (r + 1) / 2;
            const int R = jj * SC + r, S = jj * SC + s;
            float acc = 0.f;
            if (R < nr) {
                for (int col = 0; col < DK; ++col) {
                    if (!steep[jj * DK + col]) continue;
                    float lg = 0.f;   // log(b_R / b_S) = sum of log gates over rows S+1..R
                    for (int i = S + 1; i <= R; ++i)
                        lg += (a.gate == GLA_GATE_PER_KEY) ? a.log_g[((size_t)bh * a.T + t0 + i) * DK + col] : lam;
                    const float qv = __bfloat162float(a.q[((size_t)bh * a.T + t0 + R) * DK + col]);
                    const float kv = __bfloat162float(a.k[((size_t)bh * a.T + t0 + S) * DK + col]);
                    acc += qv * kv * __expf(lg);
                }
            }
            corr[jj * NTRI + p] = acc;
        }
    }

    // ---- 4. lower blocks of A on the tensor cores
    const int g8 = lane / 4, c4 = lane % 4;
    float acc[2][2][4];
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        const int blk = warp + bi * NWARP;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[bi][nt][e] = 0.f;
        if (blk >= NPAIR) continue;
        int jb = 0;
        while ((jb + 1) * (jb + 2) / 2 <= blk) ++jb;
        const int ub = blk - jb * (jb + 1) / 2;
        const float* w = W + blk * DK;
        const int ra = jb * SC + g8;   // fragment rows ra and ra + 8 (same row % 8)
#pragma unroll 4
        for (int k0 = 0; k0 < DK; k0 += 16) {
            const uint32_t a0 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra, k0 + 2 * c4));
            const uint32_t a1 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra + 8, k0 + 2 * c4));
            const uint32_t a2 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra, k0 + 8 + 2 * c4));
            const uint32_t a3 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra + 8, k0 + 8 + 2 * c4));
            const float2 w01 = *reinterpret_cast<const float2*>(w + k0 + 2 * c4);
            const float2 w89 = *reinterpret_cast<const float2*>(w + k0 + 2 * c4 + 8);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int rb = ub * SC + nt * 8 + g8;
                uint32_t b0 = *reinterpret_cast<const uint32_t*>(Ks + swz<DK>(rb, k0 + 2 * c4));
                uint32_t b1 = *reinterpret_cast<const uint32_t*>(Ks + swz<DK>(rb, k0 + 8 + 2 * c4));
                if (gated) {
                    b0 = scale_bf16x2(b0, w01.x, w01.y);
                    b1 = scale_bf16x2(b1, w89.x, w89.y);
                }
                mma_bf16_16816(acc[bi][nt], a0, a1, a2, a3, b0, b1);
            }
        }
    }
    __syncthreads();   // every warp is done reading Qs/Ks; As reuses that space
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        const int blk = warp + bi * NWARP;
        if (blk >= NPAIR) continue;
        int jb = 0;
        while ((jb + 1) * (jb + 2) / 2 <= blk) ++jb;
        const int ub = blk - jb * (jb + 1) / 2;
        const bool diag = (jb == ub);
        const bool fix = diag && steep_any[jb];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int rl = g8 + hr * 8;
                const int sl = nt * 8 + 2 * c4;
                float v0 = acc[bi][nt][hr * 2 + 0], v1 = acc[bi][nt][hr * 2 + 1];
                if (diag) {
                    if (fix) {
                        if (sl <= rl) v0 += corr[jb * NTRI + rl * (rl + 1) / 2 + sl];
                        if (sl + 1 <= rl) v1 += corr[jb * NTRI + rl * (rl + 1) / 2 + sl + 1];
                    }
                    if (sl > rl) v0 = 0.f;
                    if (sl + 1 > rl) v1 = 0.f;
                }
                *reinterpret_cast<__nv_bfloat162*>(As + (jb * SC + rl) * ALD + ub * SC + sl) =
                    __floats2bfloat162_rn(v0, v1);
            }
    }
    // upper blocks (j < u) are zero
    for (int idx = tid; idx < C * C / 2; idx += NT) {
        const int r = idx / (C / 2), s = (idx % (C / 2)) * 2;
        if (s / SC > r / SC) *reinterpret_cast<uint32_t*>(As + r * ALD + s) = 0u;
    }
    __syncthreads();
    __nv_bfloat16* Ao = a.A + ((size_t)bh * a.nchunks + c) * C * C;
    for (int idx = tid; idx < C * C / 8; idx += NT) {
        const int r = idx / (C / 8), s = (idx % (C / 8)) * 8;
        *reinterpret_cast<uint4*>(Ao + r * C + s) = *reinterpret_cast<const uint4*>(As + r * ALD + s);
    }
    __syncthreads();   // shared tiles are refilled by the next item
    }
}

// Uniform gates (none, or one fixed decay lambda per head): the cumulative log
// gate of row r in a chunk is (r+1) log(lambda) for every key, so Lambda, Gamma
// and gamma are per-row scalars and the intra-chunk scores have the closed
// form P_rs = (q_r . k_s) lambda^(r-s), r >= s (the decay mask M_ij =
// lambda^(i-j) of "Lightning Attention-2", §3.2.1 Alg. 1). The scores are one
// plain q k^T product per 16-row block (mma.sync) scaled in the epilogue; no
// per-element exponentials and no steep-gate fallback are needed.
template <int DK>
constexpr int prep_uniform_ctas_per_sm() { return DK <= 128 ? 4 : 3; }

template <int DK>
__global__ void __launch_bounds__(NT, prep_uniform_ctas_per_sm<DK>()) gla_chunk_prep_uniform_kernel(PrepArgs a)
{
    using L = PL<DK>;
    constexpr int RPT = L::RPT;
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem);      // [C][DK], raw q, swizzled
    __nv_bfloat16* Ks = Qs + C * DK;                                   // [C][DK], raw k, swizzled
    uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + 2 * C * DK * 2);
    __nv_bfloat16* As = Qs;                                            // [C][ALD], after the MMAs

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        sm100::mbar_init(cbar, 1);
        sm100::mbar_fence_init();
    }
    __syncthreads();
    const int total = a.BH * a.nchunks;
    const bool gated = a.gate != GLA_GATE_NONE;
    for (int item = blockIdx.x, it = 0; item < total; item += gridDim.x, ++it) {
    const int c = item % a.nchunks, bh = item / a.nchunks, h = bh % a.H;
    const int t0 = c * C;
    const int nr = min(C, a.T - t0);
    const float lam = gated ? a.log_g[h] : 0.f;   // log(lambda_h) <= 0
    const int cg = tid % L::NCG, rg = tid / L::NCG;
    const int col0 = cg * 8, row0 = rg * RPT;

    if (tid == 0) {
        const uint32_t bytes = (uint32_t)nr * DK * 2;
        sm100::mbar_arrive_expect_tx(cbar, 2 * bytes);
        sm100::bulk_load(Qs, a.q + ((size_t)bh * a.T + t0) * DK, bytes, cbar);
        sm100::bulk_load(Ks, a.k + ((size_t)bh * a.T + t0) * DK, bytes, cbar);
        const int nx = item + gridDim.x;
        if (nx < total) {
            const int c2 = nx % a.nchunks, bh2 = nx / a.nchunks, nr2 = min(C, a.T - c2 * C);
            const size_t row = (size_t)bh2 * a.T + (size_t)c2 * C;
            sm100::prefetch_l2(a.q + row * DK, (uint32_t)nr2 * DK * 2);
            sm100::prefetch_l2(a.k + row * DK, (uint32_t)nr2 * DK * 2);
        }
    }
    for (int i = nr * DK / 8 + tid; i < C * DK / 8; i += NT) {
        reinterpret_cast<uint4*>(Qs)[i] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(Ks)[i] = make_uint4(0, 0, 0, 0);
    }
    if (gated && tid < DK) a.gam[((size_t)bh * a.nchunks + c) * DK + tid] = __expf(nr * lam);
    {
        const bool ok = sm100::mbar_wait(cbar, it & 1, kCopyTimeoutNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicExch(a.status, ERR_PREP);
            return;
        }
    }
    // swizzle in place for the fragment loads; Q (.) Lambda and K (.) Gamma with per-row factors
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int row = row0 + r;
        const uint4 qu = *reinterpret_cast<const uint4*>(Qs + row * DK + col0);
        const uint4 ku = *reinterpret_cast<const uint4*>(Ks + row * DK + col0);
        __syncwarp();   // the warp owns whole rows: all raw reads of this row precede the swizzled writes
        *reinterpret_cast<uint4*>(Qs + swz<DK>(row, col0)) = qu;
        *reinterpret_cast<uint4*>(Ks + swz<DK>(row, col0)) = ku;
        if (gated) {
            const bool valid = row < nr;
            const float lq = valid ? __expf((row + 1) * lam) : 0.f;       // b_row / b_start
            const float lk = valid ? __expf((nr - 1 - row) * lam) : 0.f;  // b_end / b_row
            float qv[8], kv[8];
            unpack8(qu, qv);
            unpack8(ku, kv);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                qv[i] *= lq;
                kv[i] *= lk;
            }
            *reinterpret_cast<uint4*>(a.Qt + ((size_t)bh * a.Tpad + t0 + row) * DK + col0) = pack8(qv);
            *reinterpret_cast<uint4*>(a.Kt + ((size_t)bh * a.Tpad + t0 + row) * DK + col0) = pack8(kv);
        }
    }
    __syncthreads();

    // lower blocks of q k^T on the tensor cores, scaled by lambda^(r-s) and masked
    const int g8 = lane / 4, c4 = lane % 4;
    float acc[2][2][4];
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        const int blk = warp + bi * NWARP;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[bi][nt][e] = 0.f;
        if (blk >= NPAIR) continue;
        int jb = 0;
        while ((jb + 1) * (jb + 2) / 2 <= blk) ++jb;
        const int ub = blk - jb * (jb + 1) / 2;
        const int ra = jb * SC + g8;
#pragma unroll 4
        for (int k0 = 0; k0 < DK; k0 += 16) {
            const uint32_t a0 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra, k0 + 2 * c4));
            const uint32_t a1 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra + 8, k0 + 2 * c4));
            const uint32_t a2 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra, k0 + 8 + 2 * c4));
            const uint32_t a3 = *reinterpret_cast<const uint32_t*>(Qs + swz<DK>(ra + 8, k0 + 8 + 2 * c4));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int rb = ub * SC + nt * 8 + g8;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(Ks + swz<DK>(rb, k0 + 2 * c4));
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(Ks + swz<DK>(rb, k0 + 8 + 2 * c4));
                mma_bf16_16816(acc[bi][nt], a0, a1, a2, a3, b0, b1);
            }
        }
    }
    __syncthreads();   // every warp is done reading Qs/Ks; As reuses that space
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        const int blk = warp + bi * NWARP;
        if (blk >= NPAIR) continue;
        int jb = 0;
        while ((jb + 1) * (jb + 2) / 2 <= blk) ++jb;
        const int ub = blk - jb * (jb + 1) / 2;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = jb * SC + g8 + hr * 8;
                const int s0 = ub * SC + nt * 8 + 2 * c4;
                float v0 = acc[bi][nt][hr * 2 + 0], v1 = acc[bi][nt][hr * 2 + 1];
                v0 = (s0 <= r) ? (gated ? v0 * __expf((r - s0) * lam) : v0) : 0.f;
                v1 = (s0 + 1 <= r) ? (gated ? v1 * __expf((r - s0 - 1) * lam) : v1) : 0.f;
                *reinterpret_cast<__nv_bfloat162*>(As + r * ALD + s0) = __floats2bfloat162_rn(v0, v1);
            }
    }
    for (int idx = tid; idx < C * C / 2; idx += NT) {
        const int r = idx / (C / 2), s2 = (idx % (C / 2)) * 2;
        if (s2 / SC > r / SC) *reinterpret_cast<uint32_t*>(As + r * ALD + s2) = 0u;
    }
    __syncthreads();
    __nv_bfloat16* Ao = a.A + ((size_t)bh * a.nchunks + c) * C * C;
    for (int idx = tid; idx < C * C / 8; idx += NT) {
        const int r = idx / (C / 8), s2 = (idx % (C / 8)) * 8;
        *reinterpret_cast<uint4*>(Ao + r * C + s2) = *reinterpret_cast<const uint4*>(As + r * ALD + s2);
    }
    __syncthreads();   // shared tiles are refilled by the next item
    }
}

template <int DK>
cudaError_t launch_prep_uniform_dk(const PrepArgs& a, int sms, cudaStream_t s)
{
    const int smem = 2 * C * DK * 2 + 16;
    const int total = a.BH * a.nchunks;
    const int resident = prep_uniform_ctas_per_sm<DK>() * sms;
    const dim3 grid(total < resident ? total : resident);
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_prep_uniform_kernel<DK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gla_chunk_prep_uniform_kernel<DK><<<grid, NT, smem, s>>>(a);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_prep_dk(const PrepArgs& a, int sms, cudaStream_t s)
{
    using L = PL<DK>;
    const int total = a.BH * a.nchunks;
    const int resident = prep_ctas_per_sm<DK>() * sms;
    const dim3 grid(total < resident ? total : resident);
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_prep_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    gla_chunk_prep_kernel<DK><<<grid, NT, L::SMEM, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s)
{
    uint8_t* base = static_cast<uint8_t*>(ws);
    PrepArgs a;
    a.q = static_cast<const __nv_bfloat16*>(p.q);
    a.k = static_cast<const __nv_bfloat16*>(p.k);
    a.log_g = p.log_g;
    a.Qt = pl.raw_qk ? nullptr : reinterpret_cast<__nv_bfloat16*>(base + pl.off_qt);
    a.Kt = pl.raw_qk ? nullptr : reinterpret_cast<__nv_bfloat16*>(base + pl.off_kt);
    a.gam = reinterpret_cast<float*>(base + pl.off_gam);
    a.A = reinterpret_cast<__nv_bfloat16*>(base + pl.off_A);
    a.status = status;
    a.BH = p.B * p.H; a.H = p.H; a.T = p.T; a.nchunks = pl.nchunks; a.Tpad = pl.Tpad; a.gate = p.gate;
    const int sms = pl.sms > 0 ? pl.sms : 148;
    if (p.gate != GLA_GATE_PER_KEY) {
        switch (p.dk) {
        case 64: return launch_prep_uniform_dk<64>(a, sms, s);
        case 128: return launch_prep_uniform_dk<128>(a, sms, s);
        case 256: return launch_prep_uniform_dk<256>(a, sms, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (p.dk) {
    case 64: return launch_prep_dk<64>(a, sms, s);
    case 128: return launch_prep_dk<128>(a, sms, s);
    case 256: return launch_prep_dk<256>(a, sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gla
