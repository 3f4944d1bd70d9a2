// Backward pass of chunkwise gated linear attention on CUDA cores (fp32 FFMA).
//
// For L with dL/dO = dO and dL/dS_T = dST (or 0) it returns dq, dk, dv, the
// gradient of log_g for the gate mode, and dS0. With b_t the inclusive
// cumulative gate and 16-row chunks [t0, t1) it uses the chunkwise form of
// "Gated Linear Attention Transformers with Hardware-Efficient Training"
// (§4.2, and the backward it describes for the chunk-level states in §3.3 and
// §4.3), with D_[n] the gradient of the state leaving chunk n through later
// chunks:
//   D_[n-1] = Diag(gamma_n) D_[n] + (Q_n (.) Lambda_n)^T dO_n,   D_[N] = dST,
//   dq_t = Lambda_t (.) (S_[n-1] do_t^T) + sum_{s<=t} e_ts (.) k_s (v_s . do_t),
//   dk_s = Gamma_s (.) (D_[n] v_s^T)     + sum_{t>=s} e_ts (.) q_t (v_s . do_t),
//   dv_s = (k_s (.) Gamma_s) D_[n]       + sum_{t>=s} P_ts do_t,
// with e_ts = b_t / b_s over keys (<= 1, taken as exp of a log difference),
// P_ts = sum_k q_tk k_sk e_tsk the causal intra-chunk scores, and dS0 =
// D_[0]. The gate gradient uses the parallel form O = ((Q (.) B)(K / B)^T (.)
// M) V (+ (Q (.) B) S0) and S_T = Diag(b_T)(S0 + sum_s (k_s / b_s)^T v_s):
//   dlog b_t = q_t (.) dq_t - k_t (.) dk_t  (+ rowsum(dST (.) S_T) at t = T-1),
//   dlog alpha_t = sum_{t' >= t} dlog b_t'.
// The bilinear gate (Table 1's DFW row, S_t = Diag(alpha_t) S_{t-1} Diag(beta_t) +
// k_t^T v_t) adds the same structure on the value columns: with b'_t the cumulative
// beta, Lambda' = b'_t / b'_start, Gamma' = b'_end / b'_t and gamma' = b'_end / b'_start,
//   D_[n-1] = Diag(gamma) D_[n] Diag(gamma') + (Q (.) Lambda)^T (dO (.) Lambda'),
// the inter products take dO (.) Lambda' and V (.) Gamma', the pair dots v_s . do_t
// and the dv intra term carry exp(B'_t - B'_s) per column, and
//   dlog beta_t = sum_{t' >= t} (o_t' (.) do_t' - v_t' (.) dv_t')  (+ colsum(dST (.) S_T) at T-1)
// with o recomputed in the reverse sweep (CUDA-core path only).
//
// Kernels: gla_bwd_states (forward sweep, writes the state after every
// chunk), gla_bwd_chunks (reverse sweep per (b,h, 64 dv columns): partial dq
// and dk over the tile's columns, dv, dS0), gla_bwd_finish (sums the partials
// in a fixed order, dlog b), gla_bwd_revsum (reverse cumulative sum over
// tokens), gla_bwd_token_gate / gla_bwd_head_gate (per-token or per-head gate
// gradients). Every reduction has a fixed order, so results are bitwise
// reproducible.
#include <cstring>

#include <cuda_bf16.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int CS = kSimtChunk;     // 16 rows per chunk
constexpr int DVT = kSimtDvTile;   // 64 dv columns per CTA
constexpr int NT = 256;

struct BwdArgs {
    const void* q; const void* k; const void* v; const void* dO;
    const float* log_g; const float* S0; const float* dST;
    float* gq; float* gk; float* gv; float* glog; float* gS0;
    float* Sst;    // [BH][nch][dk][dv] state after each chunk
    float* Pq;     // [nplanes][BH][T][dk] dq partials: one per dv tile (+ the intra plane on the bf16 path)
    float* Pk;     // [nplanes][BH][T][dk] dk partials, likewise
    float* Ag;     // [BH][nch][CS][CS] intra-chunk scores (bf16 path)
    float* bnd;    // [ndvt][BH][dk] rowsum(dST (.) S_T) partial per dv tile
    float* dla;    // [BH][T][dk] dlog b, then dlog alpha (per key)
    // bilinear gate: log beta, its gradient, and the per-token terms o (.) do - v (.) dv
    // (plus colsum(dST (.) S_T) at the last token) whose reverse cumulative sum it is
    const float* log_b; float* glb; float* dlbe;   // [BH][T][dv] each
    float* hpart;  // [H][HG_SPLIT] partial sums of the per-head gate gradient
    int B, H, T, dk, dv, gate, nch, ndvt, nplanes;
};

template <typename T> __device__ __forceinline__ float ld_in(const T* p, size_t i);
template <> __device__ __forceinline__ float ld_in<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

// L2 prefetch hints for the n bytes at p, one per 128-byte step, spread over nth threads;
// only addresses inside the range are named, so no alignment is required.
__device__ __forceinline__ void pf_range(const void* p, size_t n, int tid, int nth) {
    const char* c = static_cast<const char*>(p);
    for (size_t off = (size_t)tid * 128; off < n; off += (size_t)nth * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

// The inputs of chunk c (rows t0 .. t0 + CS, clipped to T) of head bh into L2: q and k rows,
// the gate rows, and this tile's v and dO columns.
__device__ __forceinline__ void pf_chunk_inputs(const struct BwdArgs& a, int bh, int c, int j0, int jn, size_t esz,
                                                bool with_q, bool with_do, int tid);

// log alpha_t for key kk of head bh (0 without a gate)
__device__ __forceinline__ float log_alpha(const BwdArgs& a, int bh, int t, int kk) {
    switch (a.gate) {
    case GLA_GATE_HEAD_SCALAR: return a.log_g[bh % a.H];
    case GLA_GATE_TOKEN_SCALAR: return a.log_g[(size_t)bh * a.T + t];
    case GLA_GATE_PER_KEY:
    case GLA_GATE_BILINEAR: return a.log_g[((size_t)bh * a.T + t) * a.dk + kk];
    }
    return 0.f;
}

// Float (x, j) of a [rows][DVT] tile in shared memory. The 16-byte groups of a row are
// XOR-swizzled by x mod 8, so that a warp reading one row per lane and a warp reading
// float4 column groups of consecutive rows both spread over all banks.
__device__ __forceinline__ int swz(int x, int j) { return x * DVT + (j ^ ((x & 7) << 2)); }

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void fma4(float4& acc, float s, float4 w) {
    acc.x = fmaf(s, w.x, acc.x); acc.y = fmaf(s, w.y, acc.y);
    acc.z = fmaf(s, w.z, acc.z); acc.w = fmaf(s, w.w, acc.w);
}
__device__ __forceinline__ float dot4(float4 u, float4 w, float acc) {
    return fmaf(u.x, w.x, fmaf(u.y, w.y, fmaf(u.z, w.z, fmaf(u.w, w.w, acc))));
}

__device__ __forceinline__ void pf_chunk_inputs(const BwdArgs& a, int bh, int c, int j0, int jn, size_t esz,
                                                bool with_q, bool with_do, int tid) {
    const int t0 = c * CS, nr = min(CS, a.T - t0);
    if (nr <= 0) return;
    const size_t row = (size_t)bh * a.T + t0;
    if (with_q) pf_range(static_cast<const char*>(a.q) + row * a.dk * esz, (size_t)nr * a.dk * esz, tid, NT);
    pf_range(static_cast<const char*>(a.k) + row * a.dk * esz, (size_t)nr * a.dk * esz, tid, NT);
    if (a.gate == GLA_GATE_PER_KEY || a.gate == GLA_GATE_BILINEAR)
        pf_range(a.log_g + row * a.dk, (size_t)nr * a.dk * 4, tid, NT);
    if (a.gate == GLA_GATE_TOKEN_SCALAR) pf_range(a.log_g + row, (size_t)nr * 4, tid, NT);
    if (tid < nr) {   // one row of this tile's v (and dO) columns per thread
        const size_t off = (row + tid) * a.dv + j0;
        pf_range(static_cast<const char*>(a.v) + off * esz, (size_t)jn * esz, 0, 1);
        if (with_do) pf_range(static_cast<const char*>(a.dO) + off * esz, (size_t)jn * esz, 0, 1);
    }
}

// ---------------------------------------------------------------- forward sweep: chunk states
template <typename Tin>
__global__ void __launch_bounds__(NT) gla_bwd_states_kernel(BwdArgs a)
{
    extern __shared__ __align__(16) float smem[];
    const int dk = a.dk, tid = threadIdx.x;
    float* S = smem;                 // [dk][DVT], swizzled
    float* kt = S + dk * DVT;        // [CS][dk] k (.) Gamma
    float* vv = kt + CS * dk;        // [CS][DVT]
    float* gam = vv + CS * DVT;      // [dk]
    float* gvb = gam + dk;           // [DVT] bilinear gate: the chunk's column decay gamma'
    const bool bil = a.gate == GLA_GATE_BILINEAR;
    const int bh = blockIdx.x, j0 = blockIdx.y * DVT, jn = min(DVT, a.dv - j0);
    const Tin* k = static_cast<const Tin*>(a.k) + (size_t)bh * a.T * dk;
    const Tin* v = static_cast<const Tin*>(a.v) + (size_t)bh * a.T * a.dv;
    for (int i = tid; i < dk * DVT; i += NT) {
        const int x = i / DVT, j = i % DVT;
        S[swz(x, j)] = (a.S0 && j < jn) ? a.S0[((size_t)bh * dk + x) * a.dv + j0 + j] : 0.f;
    }
    for (int c = 0; c < a.nch; ++c) {
        const int t0 = c * CS, nr = min(CS, a.T - t0);
        __syncthreads();
        if (c + 1 < a.nch) pf_chunk_inputs(a, bh, c + 1, j0, jn, sizeof(Tin), false, false, tid);
        for (int i = tid; i < CS * DVT; i += NT) {
            const int r = i / DVT, j = i % DVT;
            vv[i] = (r < nr && j < jn) ? ld_in<Tin>(v, (size_t)(t0 + r) * a.dv + j0 + j) : 0.f;
        }
        for (int x = tid; x < dk; x += NT) {
            float lg[CS], kv[CS], bcr[CS], run = 0.f;
#pragma unroll
            for (int r = 0; r < CS; ++r) {   // every load first, then the arithmetic
                lg[r] = r < nr ? log_alpha(a, bh, t0 + r, x) : 0.f;
                kv[r] = r < nr ? ld_in<Tin>(k, (size_t)(t0 + r) * dk + x) : 0.f;
            }
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                run += lg[r];
                bcr[r] = run;
            }
            gam[x] = expf(run);
#pragma unroll
            for (int r = 0; r < CS; ++r) kt[r * dk + x] = kv[r] * expf(run - bcr[r]);
        }
        if (bil) {
            // the column side: B'_r the in-chunk cumulative log beta, gamma' = exp(B'_end), and
            // V (.) Gamma' with Gamma'_r = exp(B'_end - B'_r) <= 1 (rows past nr are zero)
            __syncthreads();
            for (int j = tid; j < DVT; j += NT) {
                float bcv[CS], run = 0.f;
#pragma unroll
                for (int r = 0; r < CS; ++r) {
                    run += (r < nr && j < jn) ? a.log_b[((size_t)bh * a.T + t0 + r) * a.dv + j0 + j] : 0.f;
                    bcv[r] = run;
                }
                gvb[j] = expf(run);
#pragma unroll
                for (int r = 0; r < CS; ++r) vv[r * DVT + j] *= expf(run - bcv[r]);
            }
        }
        __syncthreads();
        // S <- Diag(gamma) S Diag(gamma') + (K (.) Gamma)^T (V (.) Gamma'), 16 columns of one row per step
        float* out = a.Sst + ((size_t)bh * a.nch + c) * dk * a.dv + j0;
        for (int it = tid; it < dk * (DVT / 16); it += NT) {
            const int x = it % dk, g0 = (it / dk) * 4;
            const float gx = gam[x];
            float4 acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 w = ld4(S + swz(x, 4 * (g0 + u)));
                const float4 c = bil ? ld4(gvb + 4 * (g0 + u)) : make_float4(1.f, 1.f, 1.f, 1.f);
                acc[u] = make_float4(gx * w.x * c.x, gx * w.y * c.y, gx * w.z * c.z, gx * w.w * c.w);
            }
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                const float kx = kt[r * dk + x];
#pragma unroll
                for (int u = 0; u < 4; ++u) fma4(acc[u], kx, ld4(vv + r * DVT + 4 * (g0 + u)));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                st4(S + swz(x, 4 * (g0 + u)), acc[u]);
                if (4 * (g0 + u) < jn) st4(out + (size_t)x * a.dv + 4 * (g0 + u), acc[u]);
            }
        }
    }
}

// ---------------------------------------------------------------- reverse sweep per chunk
template <typename Tin>
__global__ void __launch_bounds__(NT) gla_bwd_chunks_kernel(BwdArgs a)
{
    extern __shared__ __align__(16) float smem[];
    const int dk = a.dk, tid = threadIdx.x, lane = tid % 32;
    float* D = smem;                 // [dk][DVT] swizzled: gradient of the state leaving the chunk, via later chunks
    float* Sp = D + dk * DVT;        // [dk][DVT] swizzled: state entering the chunk
    float* qr = Sp + dk * DVT;       // [CS][dk] q, then q (.) Lambda
    float* kr = qr + CS * dk;        // [CS][dk] k, then k (.) Gamma
    float* bc = kr + CS * dk;        // [CS][dk] in-chunk cumulative log gate
    float* vv = bc + CS * dk;        // [CS][DVT] v, this tile's columns
    float* dd = vv + CS * DVT;       // [CS][DVT] dO, this tile's columns
    float* A = dd + CS * DVT;        // [CS][CS] intra scores P_ts (all keys), t >= s
    float* VD = A + CS * CS;         // [CS][CS] v_s . do_t over this tile's columns, t >= s
    float* Aw = VD + CS * CS;        // [NT / 32][CS][CS] per-warp partial scores, summed in a fixed order
    float* gam = Aw + (NT / 32) * CS * CS;   // [dk]
    // bilinear gate only: the column side of the chunk
    float* bcv = gam + dk;           // [CS][DVT] in-chunk cumulative log beta, B'
    float* ddL = bcv + CS * DVT;     // [CS][DVT] dO (.) Lambda', Lambda'_r = exp(B'_r)
    float* vvG = ddL + CS * DVT;     // [CS][DVT] v (.) Gamma', Gamma'_r = exp(B'_end - B'_r)
    float* gvb = vvG + CS * DVT;     // [DVT] gamma' = exp(B'_end)
    float* cst = gvb + DVT;          // [DVT] colsum(dST (.) S_T), added at the last token
    const bool bil = a.gate == GLA_GATE_BILINEAR;
    const int bh = blockIdx.x, tile = blockIdx.y, BH = gridDim.x;
    const int j0 = tile * DVT, jn = min(DVT, a.dv - j0);
    const size_t ST = (size_t)dk * a.dv;
    const Tin* q = static_cast<const Tin*>(a.q) + (size_t)bh * a.T * dk;
    const Tin* k = static_cast<const Tin*>(a.k) + (size_t)bh * a.T * dk;
    const Tin* v = static_cast<const Tin*>(a.v) + (size_t)bh * a.T * a.dv;
    const Tin* dO = static_cast<const Tin*>(a.dO) + (size_t)bh * a.T * a.dv;

    for (int i = tid; i < dk * DVT; i += NT) {
        const int x = i / DVT, j = i % DVT;
        D[swz(x, j)] = (a.dST && j < jn) ? a.dST[(size_t)bh * ST + (size_t)x * a.dv + j0 + j] : 0.f;
    }
    if (a.bnd) {
        const float* Sfin = a.nch > 0 ? a.Sst + ((size_t)bh * a.nch + a.nch - 1) * ST : nullptr;
        for (int x = tid; x < dk; x += NT) {
            float s = 0.f;
            if (a.dST && Sfin)
                for (int j = 0; j < jn; ++j)
                    s = fmaf(a.dST[(size_t)bh * ST + (size_t)x * a.dv + j0 + j], Sfin[(size_t)x * a.dv + j0 + j], s);
            a.bnd[((size_t)tile * BH + bh) * dk + x] = s;
        }
    }
    if (bil) {
        const float* Sfin = a.nch > 0 ? a.Sst + ((size_t)bh * a.nch + a.nch - 1) * ST : nullptr;
        for (int j = tid; j < DVT; j += NT) {
            float s = 0.f;
            if (a.dST && Sfin && j < jn)
                for (int x = 0; x < dk; ++x)
                    s = fmaf(a.dST[(size_t)bh * ST + (size_t)x * a.dv + j0 + j], Sfin[(size_t)x * a.dv + j0 + j], s);
            cst[j] = s;
        }
    }
    const int kk = tid;                       // the key a thread owns in the per-key phases
    const bool warp_on = (tid & ~31) < dk;    // warps with at least one key
    const bool key_on = kk < dk;
    for (int c = a.nch - 1; c >= 0; --c) {
        const int t0 = c * CS, nr = min(CS, a.T - t0);
        __syncthreads();   // the previous chunk is done with every buffer
        for (int i = tid; i < CS * dk; i += NT) {
            const int r = i / dk, x = i % dk;
            const bool ok = r < nr;
            qr[i] = ok ? ld_in<Tin>(q, (size_t)(t0 + r) * dk + x) : 0.f;
            kr[i] = ok ? ld_in<Tin>(k, (size_t)(t0 + r) * dk + x) : 0.f;
        }
        for (int i = tid; i < CS * DVT; i += NT) {
            const int r = i / DVT, j = i % DVT;
            const bool ok = r < nr && j < jn;
            vv[i] = ok ? ld_in<Tin>(v, (size_t)(t0 + r) * a.dv + j0 + j) : 0.f;
            dd[i] = ok ? ld_in<Tin>(dO, (size_t)(t0 + r) * a.dv + j0 + j) : 0.f;
        }
        if (c > 0) {   // the stored state (16-byte aligned rows of the workspace)
            const float* src = a.Sst + ((size_t)bh * a.nch + c - 1) * ST + j0;
            for (int i = tid; i < dk * (DVT / 4); i += NT) {
                const int x = i / (DVT / 4), j = 4 * (i % (DVT / 4));
                st4(Sp + swz(x, j), j < jn ? ld4(src + (size_t)x * a.dv + j) : make_float4(0.f, 0.f, 0.f, 0.f));
            }
        } else {       // S0 (caller memory, 4-byte aligned) or zero
            for (int i = tid; i < dk * DVT; i += NT) {
                const int x = i / DVT, j = i % DVT;
                Sp[swz(x, j)] = (a.S0 && j < jn) ? a.S0[(size_t)bh * ST + (size_t)x * a.dv + j0 + j] : 0.f;
            }
        }
        if (key_on) {
            float run = 0.f;
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                run += r < nr ? log_alpha(a, bh, t0 + r, kk) : 0.f;
                bc[r * dk + kk] = run;
            }
            gam[kk] = expf(run);
        }
        __syncthreads();
        if (bil) {   // the column side: B', gamma', dO (.) Lambda', v (.) Gamma' (rows past nr are zero)
            for (int j = tid; j < DVT; j += NT) {
                float run = 0.f;
#pragma unroll
                for (int r = 0; r < CS; ++r) {
                    run += (r < nr && j < jn) ? a.log_b[((size_t)bh * a.T + t0 + r) * a.dv + j0 + j] : 0.f;
                    bcv[r * DVT + j] = run;
                }
                gvb[j] = expf(run);
#pragma unroll
                for (int r = 0; r < CS; ++r) {
                    const float b = bcv[r * DVT + j];
                    ddL[r * DVT + j] = dd[r * DVT + j] * expf(b);
                    vvG[r * DVT + j] = vv[r * DVT + j] * expf(run - b);
                }
            }
            __syncthreads();
        }
        for (int p = tid; p < CS * CS; p += NT) {
            const int t = p / CS, s = p % CS;
            float acc = 0.f;
            if (s <= t) {
                if (bil) {   // v_s . do_t with the column decay exp(B'_t - B'_s) <= 1
                    for (int j = 0; j < DVT; ++j)
                        acc = fmaf(dd[t * DVT + j] * vv[s * DVT + j], expf(bcv[t * DVT + j] - bcv[s * DVT + j]), acc);
                } else {
#pragma unroll
                    for (int g = 0; g < DVT / 4; ++g)
                        acc = dot4(ld4(dd + t * DVT + 4 * g), ld4(vv + s * DVT + 4 * g), acc);
                }
            }
            VD[p] = acc;
        }
        __syncthreads();
        // pairs t >= s, one thread per key: the scores P_ts (summed over a warp's keys by
        // shuffles, then over warps in a fixed order) and the intra parts of dq and dk
        float dqi[CS], dki[CS];
#pragma unroll
        for (int r = 0; r < CS; ++r) dqi[r] = dki[r] = 0.f;
        if (warp_on) {
#pragma unroll
            for (int t = 0; t < CS; ++t) {
                const float bt = key_on ? bc[t * dk + kk] : 0.f;
                const float qt = key_on ? qr[t * dk + kk] : 0.f;
#pragma unroll
                for (int s = 0; s <= t; ++s) {
                    const float e = key_on ? expf(bt - bc[s * dk + kk]) : 0.f;
                    const float ks = key_on ? kr[s * dk + kk] : 0.f;
                    const float w = VD[t * CS + s];
                    dqi[t] = fmaf(e * ks, w, dqi[t]);
                    dki[s] = fmaf(e * qt, w, dki[s]);
                    float pk = qt * ks * e;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) pk += __shfl_xor_sync(0xffffffffu, pk, o);
                    if (lane == 0) Aw[(tid / 32) * CS * CS + t * CS + s] = pk;
                }
            }
        }
        __syncthreads();
        for (int p = tid; p < CS * CS; p += NT) {
            const int t = p / CS, s = p % CS;
            float acc = 0.f;
            if (s <= t)
                for (int wp = 0; wp * 32 < dk; ++wp) acc += Aw[wp * CS * CS + p];
            A[p] = acc;
        }
        // inter parts (S_[n-1] do_t^T and D_[n] v_t^T over this tile's columns, 4 at a time),
        // then this tile's partials of dq and dk
        if (key_on) {
            float aq[CS], ak[CS];
#pragma unroll
            for (int t = 0; t < CS; ++t) aq[t] = ak[t] = 0.f;
            const float* ddq = bil ? ddL : dd;   // dO (.) Lambda' and v (.) Gamma' with the bilinear gate
            const float* vvk = bil ? vvG : vv;
#pragma unroll 2
            for (int g = 0; g < DVT / 4; ++g) {
                const float4 sp = ld4(Sp + swz(kk, 4 * g)), dg = ld4(D + swz(kk, 4 * g));
#pragma unroll
                for (int t = 0; t < CS; ++t) {
                    aq[t] = dot4(sp, ld4(ddq + t * DVT + 4 * g), aq[t]);
                    ak[t] = dot4(dg, ld4(vvk + t * DVT + 4 * g), ak[t]);
                }
            }
            const float bend = bc[(CS - 1) * dk + kk];
            const size_t prow = ((size_t)tile * BH + bh) * a.T + t0;
#pragma unroll
            for (int t = 0; t < CS; ++t) {
                const float b = bc[t * dk + kk];
                if (t < nr) {
                    a.Pq[(prow + t) * dk + kk] = fmaf(expf(b), aq[t], dqi[t]);
                    a.Pk[(prow + t) * dk + kk] = fmaf(expf(bend - b), ak[t], dki[t]);
                }
                // K (.) Gamma and Q (.) Lambda in place (rows past nr are zero)
                kr[t * dk + kk] *= expf(bend - b);
                qr[t * dk + kk] *= expf(b);
            }
        }
        __syncthreads();
        // dv (this tile): (K (.) Gamma) D + P^T dO over rows t >= s; a thread owns 4 columns of a row
        {
            const int s = tid / (DVT / 4), g = tid % (DVT / 4);
            static_assert(CS * (DVT / 4) == NT, "one float4 of dv per thread");
            if (s < nr && 4 * g < jn && !bil) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int x = 0; x < dk; ++x) fma4(acc, kr[s * dk + x], ld4(D + swz(x, 4 * g)));
                for (int t = s; t < CS; ++t) fma4(acc, A[t * CS + s], ld4(dd + t * DVT + 4 * g));
                float* o = a.gv + ((size_t)bh * a.T + t0 + s) * a.dv + j0 + 4 * g;
                o[0] = acc.x; o[1] = acc.y; o[2] = acc.z; o[3] = acc.w;
            } else if (s < nr && 4 * g < jn) {
                // bilinear gate, per column j: dv_s = Gamma'_s (K (.) Gamma)_s D + sum_{t>=s} P_ts do_t
                // exp(B'_t - B'_s); and the output o_s = Lambda'_s (Q (.) Lambda)_s S_[n-1] +
                // sum_{t<=s} P_st v_t exp(B'_s - B'_t), for the term o_s do_s - v_s dv_s of dlog beta
                float kd[4] = {0.f, 0.f, 0.f, 0.f}, qs[4] = {0.f, 0.f, 0.f, 0.f};
                for (int x = 0; x < dk; ++x) {
                    const float4 dx = ld4(D + swz(x, 4 * g)), sx = ld4(Sp + swz(x, 4 * g));
                    const float kx = kr[s * dk + x], qx = qr[s * dk + x];
                    kd[0] = fmaf(kx, dx.x, kd[0]); kd[1] = fmaf(kx, dx.y, kd[1]);
                    kd[2] = fmaf(kx, dx.z, kd[2]); kd[3] = fmaf(kx, dx.w, kd[3]);
                    qs[0] = fmaf(qx, sx.x, qs[0]); qs[1] = fmaf(qx, sx.y, qs[1]);
                    qs[2] = fmaf(qx, sx.z, qs[2]); qs[3] = fmaf(qx, sx.w, qs[3]);
                }
                const size_t row = (size_t)bh * a.T + t0 + s;
                float* o = a.gv + row * a.dv + j0 + 4 * g;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = 4 * g + c;
                    const float bs = bcv[s * DVT + j], bend = bcv[(CS - 1) * DVT + j];
                    float dvj = kd[c] * expf(bend - bs);
                    for (int t = s; t < CS; ++t)
                        dvj = fmaf(A[t * CS + s] * dd[t * DVT + j], expf(bcv[t * DVT + j] - bs), dvj);
                    float oj = qs[c] * expf(bs);
                    for (int t = 0; t <= s; ++t)
                        oj = fmaf(A[s * CS + t] * vv[t * DVT + j], expf(bs - bcv[t * DVT + j]), oj);
                    o[c] = dvj;
                    float e = oj * dd[s * DVT + j] - vv[s * DVT + j] * dvj;
                    if (t0 + s == a.T - 1) e += cst[j];
                    a.dlbe[row * a.dv + j0 + j] = e;
                }
            }
        }
        __syncthreads();
        // D <- Diag(gamma) D + (Q (.) Lambda)^T dO, 16 columns of one row per step
        for (int it = tid; it < dk * (DVT / 16); it += NT) {
            const int x = it % dk, g0 = (it / dk) * 4;
            const float gx = gam[x];
            const float* ddu = bil ? ddL : dd;   // bilinear gate: D Diag(gamma') and dO (.) Lambda'
            float4 acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 w = ld4(D + swz(x, 4 * (g0 + u)));
                const float4 c = bil ? ld4(gvb + 4 * (g0 + u)) : make_float4(1.f, 1.f, 1.f, 1.f);
                acc[u] = make_float4(gx * w.x * c.x, gx * w.y * c.y, gx * w.z * c.z, gx * w.w * c.w);
            }
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                const float qx = qr[r * dk + x];
#pragma unroll
                for (int u = 0; u < 4; ++u) fma4(acc[u], qx, ld4(ddu + r * DVT + 4 * (g0 + u)));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) st4(D + swz(x, 4 * (g0 + u)), acc[u]);
        }
    }
    __syncthreads();
    if (a.gS0)
        for (int i = tid; i < dk * DVT; i += NT) {
            const int x = i / DVT, j = i % DVT;
            if (j < jn) a.gS0[(size_t)bh * ST + (size_t)x * a.dv + j0 + j] = D[swz(x, j)];
        }
}

// ---------------------------------------------------------------- the bf16 path: intra kernel + tensor-core sweep
// For bf16 inputs with dk in {64, 128, 256} the reverse sweep is split in two:
//  * gla_bwd_intra, parallel over (b,h, chunk): the pair walk (t >= s, exact in fp32 log
//    space) over the full dv width gives the intra parts of dq and dk (written as one
//    more partial plane) and the scores P_ts (kept for the dv product);
//  * gla_bwd_sweep_tc, serial over chunks per (b,h, 64 dv columns): the chunk products
//      dq_inter = dO S_[n-1]^T, dk_inter = V D_[n]^T, dv = (K (.) Gamma) D_[n] + P^T dO,
//      D_[n-1] = Diag(gamma) D_[n] + (Q (.) Lambda)^T dO
//    on the tensor cores (mma.sync m16n8k16, fp32 accumulate). Operands that are not bf16
//    inputs (the state, D, Q (.) Lambda, K (.) Gamma) are split into hi + lo bf16 parts and
//    multiplied as hi*x + lo*x (+ hi*lo for dv), so each product keeps about 16 mantissa
//    bits: the bf16 path is as accurate as the fp32 one. D is carried in fp32 accumulator
//    registers from chunk to chunk.
constexpr int BP = 8;              // bf16 row padding: rows 16 bytes apart in the banks
constexpr int VDC = 256;           // dv columns per staged slice in the intra kernel's v . dO products

__device__ __forceinline__ void ldsm_x4(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(const void* p, uint32_t& r0, uint32_t& r1) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
}
__device__ __forceinline__ void ldsm_x2_t(const void* p, uint32_t& r0, uint32_t& r1) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// x = hi + lo with hi, lo bf16 (lo carries the next 8 mantissa bits)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// ---- forward sweep on the tensor cores (bf16 inputs, dk in {64, 128, 256})
// The same recurrence as gla_bwd_states_kernel, S <- Diag(gamma) S + (K (.) Gamma)^T V per
// 16-row chunk, with the state held in the warps' fp32 mma.sync accumulators: warp w owns
// the 16 x 8 tiles w * TPW .. w * TPW + TPW - 1 (key tile m = id / 8, column tile n = id % 8).
// K (.) Gamma is split into hi + lo bf16 parts and v is bf16, so each product keeps about
// 16 mantissa bits, as in the reverse sweep. Each chunk's state goes to the workspace from
// the accumulators: 8-byte pairs, every 32-byte sector written whole.
template <int DK>
struct StLay {
    static constexpr int RS = DVT + BP;                  // bf16 row of a [CS][64] tile
    static constexpr int RK = DK + BP;                   // bf16 row of a [CS][DK] tile
    static constexpr int VVB = 0;                        // bf16 [CS][RS] v, this tile's columns
    static constexpr int KGH = VVB + CS * RS * 2;        // bf16 [CS][RK] k (.) Gamma, hi
    static constexpr int KGL = KGH + CS * RK * 2;        //   and lo
    static constexpr int GAM = KGL + CS * RK * 2;        // fp32 [DK] chunk decay
    static constexpr int BYTES = GAM + DK * 4;
    static constexpr int TPW = DK / 16;                  // accumulator tiles per warp
    static_assert(KGH % 16 == 0 && KGL % 16 == 0 && GAM % 16 == 0, "ldmatrix rows 16-byte aligned");
};

template <int DK>
__global__ void __launch_bounds__(NT, 2) gla_bwd_states_tc_kernel(BwdArgs a)
{
    using L = StLay<DK>;
    extern __shared__ __align__(16) uint8_t sst[];
    __nv_bfloat16* vvb = reinterpret_cast<__nv_bfloat16*>(sst + L::VVB);
    __nv_bfloat16* kgh = reinterpret_cast<__nv_bfloat16*>(sst + L::KGH);
    __nv_bfloat16* kgl = reinterpret_cast<__nv_bfloat16*>(sst + L::KGL);
    float* gam = reinterpret_cast<float*>(sst + L::GAM);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, g = lane / 4, tq = lane % 4;
    const int bh = blockIdx.x, j0 = blockIdx.y * DVT, jn = min(DVT, a.dv - j0);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k) + (size_t)bh * a.T * DK;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v) + (size_t)bh * a.T * a.dv;

    float Sacc[L::TPW][4];
#pragma unroll
    for (int u = 0; u < L::TPW; ++u) {
        const int id = warp * L::TPW + u, m = id / 8, n = id % 8;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = 16 * m + g + 8 * (e / 2), j = 8 * n + 2 * tq + (e % 2);
            Sacc[u][e] = (a.S0 && j < jn) ? a.S0[((size_t)bh * DK + key) * a.dv + j0 + j] : 0.f;
        }
    }
    const int brow = (lane % 8) + 8 * ((lane / 8) % 2);
    const int mi = lane / 8, arow = (lane % 8) + 8 * (mi / 2), acol = 8 * (mi % 2);
    for (int c = 0; c < a.nch; ++c) {
        const int t0 = c * CS, nr = min(CS, a.T - t0);
        __syncthreads();   // the previous chunk's products are done with the tiles
        if (c + 1 < a.nch) pf_chunk_inputs(a, bh, c + 1, j0, jn, 2, false, false, tid);
        for (int i = tid; i < CS * DVT; i += NT) {
            const int r = i / DVT, j = i % DVT;
            vvb[r * L::RS + j] = (r < nr && j < jn) ? v[(size_t)(t0 + r) * a.dv + j0 + j] : __float2bfloat16_rn(0.f);
        }
        for (int x = tid; x < DK; x += NT) {
            float lg[CS], kv[CS], bcr[CS], run = 0.f;
#pragma unroll
            for (int r = 0; r < CS; ++r) {   // every load first, then the arithmetic
                lg[r] = r < nr ? log_alpha(a, bh, t0 + r, x) : 0.f;
                kv[r] = r < nr ? __bfloat162float(k[(size_t)(t0 + r) * DK + x]) : 0.f;
            }
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                run += lg[r];
                bcr[r] = run;
            }
            gam[x] = expf(run);
#pragma unroll
            for (int r = 0; r < CS; ++r) split_bf16(kv[r] * expf(run - bcr[r]), kgh[r * L::RK + x], kgl[r * L::RK + x]);
        }
        __syncthreads();
        float* out = a.Sst + ((size_t)bh * a.nch + c) * DK * a.dv + j0;
#pragma unroll
        for (int u = 0; u < L::TPW; ++u) {
            const int id = warp * L::TPW + u, m = id / 8, n = id % 8;
            uint32_t a0, a1, a2, a3, b0, b1;
            ldsm_x2_t(vvb + brow * L::RS + 8 * n, b0, b1);
            const float g0 = gam[16 * m + g], g1 = gam[16 * m + g + 8];
            Sacc[u][0] *= g0; Sacc[u][1] *= g0; Sacc[u][2] *= g1; Sacc[u][3] *= g1;
            ldsm_x4_t(kgh + arow * L::RK + 16 * m + acol, a0, a1, a2, a3);
            mma16816(Sacc[u], a0, a1, a2, a3, b0, b1);
            ldsm_x4_t(kgl + arow * L::RK + 16 * m + acol, a0, a1, a2, a3);
            mma16816(Sacc[u], a0, a1, a2, a3, b0, b1);
            const int key = 16 * m + g, j = 8 * n + 2 * tq;   // j even, jn a multiple of 16
            if (j < jn) {
                *reinterpret_cast<float2*>(out + (size_t)key * a.dv + j) = make_float2(Sacc[u][0], Sacc[u][1]);
                *reinterpret_cast<float2*>(out + (size_t)(key + 8) * a.dv + j) = make_float2(Sacc[u][2], Sacc[u][3]);
            }
        }
    }
}

// ---- intra kernel: grid (BH, nch), one thread per key; the pair walk over the full dv width
__global__ void __launch_bounds__(NT) gla_bwd_intra_kernel(BwdArgs a, float* Ag)
{
    extern __shared__ __align__(16) float smi[];
    const int dk = a.dk, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    float* qr = smi;                 // [CS][dk]
    float* kr = qr + CS * dk;        // [CS][dk]
    float* bc = kr + CS * dk;        // [CS][dk]
    float* VD = bc + CS * dk;        // [CS][CS] v_s . do_t over all dv columns
    float* Aw = VD + CS * CS;        // [NT / 32][CS][CS]
    __nv_bfloat16* dsl = reinterpret_cast<__nv_bfloat16*>(Aw + (NT / 32) * CS * CS);   // [CS][VDC] dO slice
    __nv_bfloat16* vsl = dsl + CS * VDC;                                                 // [CS][VDC] v slice
    const int bh = blockIdx.x, c = blockIdx.y, BH = gridDim.x;
    const int t0 = c * CS, nr = min(CS, a.T - t0);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + (size_t)bh * a.T * dk;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k) + (size_t)bh * a.T * dk;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v) + ((size_t)bh * a.T + t0) * a.dv;
    const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(a.dO) + ((size_t)bh * a.T + t0) * a.dv;
    for (int i = tid; i < CS * dk; i += NT) {
        const int r = i / dk, x = i % dk;
        const bool ok = r < nr;
        qr[i] = ok ? __bfloat162float(q[(size_t)(t0 + r) * dk + x]) : 0.f;
        kr[i] = ok ? __bfloat162float(k[(size_t)(t0 + r) * dk + x]) : 0.f;
    }
    const int kk = tid;
    const bool key_on = kk < dk, warp_on = (tid & ~31) < dk;
    if (key_on) {
        float run = 0.f;
#pragma unroll
        for (int r = 0; r < CS; ++r) {
            run += r < nr ? log_alpha(a, bh, t0 + r, kk) : 0.f;
            bc[r * dk + kk] = run;
        }
    }
    // v_s . do_t for t >= s over every dv column (rows past nr are zero): VDC columns at a
    // time, the chunk's dO and v rows staged in shared memory by 16-byte loads; one warp per
    // pair, its lanes splitting the columns, partial sums in registers until the end
    constexpr int NPW = (CS * (CS + 1) / 2 + NT / 32 - 1) / (NT / 32);   // pairs per warp
    float vdp[NPW];
#pragma unroll
    for (int i = 0; i < NPW; ++i) vdp[i] = 0.f;
    // 16-byte loads need 16-byte aligned bases (rows are, dv being a multiple of 16)
    const bool vec = ((reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.dO)) & 15) == 0;
    for (int j0 = 0; j0 < a.dv; j0 += VDC) {
        __syncthreads();   // the previous slice has been read
        for (int i = tid; i < CS * VDC / 8; i += NT) {
            const int r = i / (VDC / 8), j = (i % (VDC / 8)) * 8;
            uint4 d8 = make_uint4(0u, 0u, 0u, 0u), v8 = d8;
            if (r < nr && j0 + j < a.dv) {
                const size_t off = (size_t)r * a.dv + j0 + j;
                if (vec) {
                    d8 = *reinterpret_cast<const uint4*>(dO + off);
                    v8 = *reinterpret_cast<const uint4*>(v + off);
                } else {
                    __nv_bfloat16* dp = reinterpret_cast<__nv_bfloat16*>(&d8);
                    __nv_bfloat16* vp = reinterpret_cast<__nv_bfloat16*>(&v8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        dp[e] = dO[off + e];
                        vp[e] = v[off + e];
                    }
                }
            }
            *reinterpret_cast<uint4*>(dsl + r * VDC + j) = d8;
            *reinterpret_cast<uint4*>(vsl + r * VDC + j) = v8;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NPW; ++i) {
            const int p = warp + i * (NT / 32);
            if (p < CS * (CS + 1) / 2) {
                int t = 0;
                while ((t + 1) * (t + 2) / 2 <= p) ++t;
                const int s2 = p - t * (t + 1) / 2;
                const __nv_bfloat162* dr = reinterpret_cast<const __nv_bfloat162*>(dsl + t * VDC);
                const __nv_bfloat162* vr = reinterpret_cast<const __nv_bfloat162*>(vsl + s2 * VDC);
                float acc = vdp[i];
#pragma unroll
                for (int j = lane; j < VDC / 2; j += 32) {
                    const float2 x = __bfloat1622float2(dr[j]), y = __bfloat1622float2(vr[j]);
                    acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
                }
                vdp[i] = acc;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NPW; ++i) {
        float acc = vdp[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const int p = warp + i * (NT / 32);
        if (lane == 0 && p < CS * (CS + 1) / 2) {
            int t = 0;
            while ((t + 1) * (t + 2) / 2 <= p) ++t;
            const int s2 = p - t * (t + 1) / 2;
            VD[t * CS + s2] = acc;
        }
    }
    __syncthreads();
    float dqi[CS], dki[CS];
#pragma unroll
    for (int r = 0; r < CS; ++r) dqi[r] = dki[r] = 0.f;
    if (warp_on) {
#pragma unroll
        for (int t = 0; t < CS; ++t) {
            const float bt = key_on ? bc[t * dk + kk] : 0.f;
            const float qt = key_on ? qr[t * dk + kk] : 0.f;
#pragma unroll
            for (int s = 0; s <= t; ++s) {
                const float e = key_on ? expf(bt - bc[s * dk + kk]) : 0.f;
                const float ks = key_on ? kr[s * dk + kk] : 0.f;
                const float w = VD[t * CS + s];
                dqi[t] = fmaf(e * ks, w, dqi[t]);
                dki[s] = fmaf(e * qt, w, dki[s]);
                float pk = qt * ks * e;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) pk += __shfl_xor_sync(0xffffffffu, pk, o);
                if (lane == 0) Aw[warp * CS * CS + t * CS + s] = pk;
            }
        }
    }
    if (key_on) {   // the intra plane of the dq / dk partials
        const size_t prow = ((size_t)a.ndvt * BH + bh) * a.T + t0;
#pragma unroll
        for (int t = 0; t < CS; ++t)
            if (t < nr) {
                a.Pq[(prow + t) * dk + kk] = dqi[t];
                a.Pk[(prow + t) * dk + kk] = dki[t];
            }
    }
    __syncthreads();
    for (int p = tid; p < CS * CS; p += NT) {
        const int t = p / CS, s = p % CS;
        float acc = 0.f;
        if (s <= t)
            for (int wp = 0; wp * 32 < dk; ++wp) acc += Aw[wp * CS * CS + p];
        Ag[((size_t)bh * a.nch + c) * CS * CS + p] = acc;
    }
}

size_t intra_smem(int dk) {
    return sizeof(float) * (3 * (size_t)CS * dk + CS * CS + (NT / 32) * CS * CS) + 2 * (size_t)CS * VDC * 2;
}

template <int DK>
struct TcLay {
    static constexpr int RS = DVT + BP;          // bf16 row of a [rows][64] tile
    static constexpr int RK = DK + BP;           // bf16 row of a [16][DK] tile
    static constexpr int SPH = 0;                                  // bf16 [DK][RS] state entering the chunk, hi
    static constexpr int SPL = SPH + DK * RS * 2;                  //   and lo
    static constexpr int DBH = SPL + DK * RS * 2;                  // bf16 [DK][RS] D, hi
    static constexpr int DBL = DBH + DK * RS * 2;                  //   and lo
    static constexpr int DDB = DBL + DK * RS * 2;                  // bf16 [CS][RS] dO
    static constexpr int VVB = DDB + CS * RS * 2;                  // bf16 [CS][RS] v
    static constexpr int QLH = VVB + CS * RS * 2;                  // bf16 [CS][RK] q (.) Lambda, hi
    static constexpr int QLL = QLH + CS * RK * 2;                  //   and lo
    static constexpr int KGH = QLL + CS * RK * 2;                  // bf16 [CS][RK] k (.) Gamma, hi
    static constexpr int KGL = KGH + CS * RK * 2;                  //   and lo
    static constexpr int BC = KGL + CS * RK * 2;                   // fp32 [CS][DK] cumulative log gate
    static constexpr int AA = BC + CS * DK * 4;                    // fp32 [CS][CS] scores of the chunk
    static constexpr int GAM = AA + CS * CS * 4;                   // fp32 [DK]
    static constexpr int BYTES = GAM + DK * 4;
    static constexpr int TPW = DK / 16;                            // D accumulator tiles per warp
    static constexpr int NPW = DK / 64;                            // dq / dk n-tiles (8 keys) per warp
    static_assert(BYTES <= 227 * 1024, "shared memory budget");
    static_assert(SPL % 16 == 0 && DBH % 16 == 0 && DDB % 16 == 0 && QLH % 16 == 0 && KGH % 16 == 0 &&
                  KGL % 16 == 0 && BC % 16 == 0, "ldmatrix rows 16-byte aligned");
};

template <int DK>
__global__ void __launch_bounds__(NT, 1) gla_bwd_sweep_tc_kernel(BwdArgs a, const float* Ag)
{
    using L = TcLay<DK>;
    extern __shared__ __align__(16) uint8_t smb[];
    __nv_bfloat16* Sph = reinterpret_cast<__nv_bfloat16*>(smb + L::SPH);
    __nv_bfloat16* Spl = reinterpret_cast<__nv_bfloat16*>(smb + L::SPL);
    __nv_bfloat16* Dbh = reinterpret_cast<__nv_bfloat16*>(smb + L::DBH);
    __nv_bfloat16* Dbl = reinterpret_cast<__nv_bfloat16*>(smb + L::DBL);
    __nv_bfloat16* ddb = reinterpret_cast<__nv_bfloat16*>(smb + L::DDB);
    __nv_bfloat16* vvb = reinterpret_cast<__nv_bfloat16*>(smb + L::VVB);
    __nv_bfloat16* qlh = reinterpret_cast<__nv_bfloat16*>(smb + L::QLH);
    __nv_bfloat16* qll = reinterpret_cast<__nv_bfloat16*>(smb + L::QLL);
    __nv_bfloat16* kgh = reinterpret_cast<__nv_bfloat16*>(smb + L::KGH);
    __nv_bfloat16* kgl = reinterpret_cast<__nv_bfloat16*>(smb + L::KGL);
    float* bc = reinterpret_cast<float*>(smb + L::BC);
    float* A = reinterpret_cast<float*>(smb + L::AA);
    float* gam = reinterpret_cast<float*>(smb + L::GAM);
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32, g = lane / 4, tq = lane % 4;
    const int bh = blockIdx.x, tile = blockIdx.y, BH = gridDim.x;
    const int j0 = tile * DVT, jn = min(DVT, a.dv - j0);
    const size_t ST = (size_t)DK * a.dv;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + (size_t)bh * a.T * DK;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k) + (size_t)bh * a.T * DK;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v) + (size_t)bh * a.T * a.dv;
    const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(a.dO) + (size_t)bh * a.T * a.dv;

    // D (fp32 accumulator fragments): warp tile u covers keys 16 m .. +15 and columns
    // 8 n .. +7; element e sits at key 16 m + g + 8 (e / 2), column 8 n + 2 tq + (e % 2)
    float Dacc[L::TPW][4];
#pragma unroll
    for (int u = 0; u < L::TPW; ++u) {
        const int id = warp * L::TPW + u, m = id / 8, n = id % 8;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = 16 * m + g + 8 * (e / 2), j = 8 * n + 2 * tq + (e % 2);
            const float d = (a.dST && j < jn) ? a.dST[(size_t)bh * ST + (size_t)key * a.dv + j0 + j] : 0.f;
            Dacc[u][e] = d;
            split_bf16(d, Dbh[key * L::RS + j], Dbl[key * L::RS + j]);
        }
    }
    if (a.bnd) {
        const float* Sfin = a.nch > 0 ? a.Sst + ((size_t)bh * a.nch + a.nch - 1) * ST : nullptr;
        for (int x = tid; x < DK; x += NT) {
            float s = 0.f;
            if (a.dST && Sfin)
                for (int j = 0; j < jn; ++j)
                    s = fmaf(a.dST[(size_t)bh * ST + (size_t)x * a.dv + j0 + j], Sfin[(size_t)x * a.dv + j0 + j], s);
            a.bnd[((size_t)tile * BH + bh) * DK + x] = s;
        }
    }
    const int kk = tid;
    const bool key_on = kk < DK;
    for (int c = a.nch - 1; c >= 0; --c) {
        const int t0 = c * CS, nr = min(CS, a.T - t0);
        __syncthreads();   // the previous chunk is done with every buffer
        if (c > 0) {   // the next chunk of the sweep into L2 while this one computes
            pf_chunk_inputs(a, bh, c - 1, j0, jn, 2, true, true, tid);
            if (c > 1 && tid < DK)
                pf_range(a.Sst + ((size_t)bh * a.nch + c - 2) * ST + (size_t)tid * a.dv + j0, (size_t)jn * 4, 0, 1);
            if (tid == 0) pf_range(Ag + ((size_t)bh * a.nch + c - 1) * CS * CS, CS * CS * 4, 0, 1);
        }
        for (int i = tid; i < CS * DVT; i += NT) {
            const int r = i / DVT, j = i % DVT;
            const bool ok = r < nr && j < jn;
            const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
            vvb[r * L::RS + j] = ok ? v[(size_t)(t0 + r) * a.dv + j0 + j] : z;
            ddb[r * L::RS + j] = ok ? dO[(size_t)(t0 + r) * a.dv + j0 + j] : z;
        }
        // every global load of the chunk is issued before any of them is used
        constexpr int NV = DK * DVT / 4 / NT;   // float4 groups of the state per thread
        float4 sv[NV];
        if (c > 0) {   // the stored state: workspace rows, 16-byte aligned
            const float* src = a.Sst + ((size_t)bh * a.nch + c - 1) * ST + j0;
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int i = tid + u * NT, x = i / (DVT / 4), j = 4 * (i % (DVT / 4));
                sv[u] = j < jn ? ld4(src + (size_t)x * a.dv + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else {       // S0 (caller memory, 4-byte aligned) or zero
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int i = tid + u * NT, x = i / (DVT / 4), j = 4 * (i % (DVT / 4));
                const float* r = a.S0 ? a.S0 + (size_t)bh * ST + (size_t)x * a.dv + j0 + j : nullptr;
                sv[u] = (r && j < jn) ? make_float4(r[0], r[1], r[2], r[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float lg[CS], qv[CS], kv[CS];
        if (key_on) {
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                const bool ok = r < nr;
                lg[r] = ok ? log_alpha(a, bh, t0 + r, kk) : 0.f;
                qv[r] = ok ? __bfloat162float(q[(size_t)(t0 + r) * DK + kk]) : 0.f;
                kv[r] = ok ? __bfloat162float(k[(size_t)(t0 + r) * DK + kk]) : 0.f;
            }
        }
        const float Ai = Ag[((size_t)bh * a.nch + c) * CS * CS + tid];
        static_assert(CS * CS == NT, "one score per thread");
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int i = tid + u * NT, x = i / (DVT / 4), j = 4 * (i % (DVT / 4));
            __nv_bfloat16* h = Sph + x * L::RS + j;
            __nv_bfloat16* l = Spl + x * L::RS + j;
            split_bf16(sv[u].x, h[0], l[0]); split_bf16(sv[u].y, h[1], l[1]);
            split_bf16(sv[u].z, h[2], l[2]); split_bf16(sv[u].w, h[3], l[3]);
        }
        A[tid] = Ai;
        if (key_on) {   // cumulative log gate, gamma, and Q (.) Lambda, K (.) Gamma in hi + lo parts
            float bcr[CS], run = 0.f;
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                run += lg[r];
                bcr[r] = run;
                bc[r * DK + kk] = run;
            }
            gam[kk] = expf(run);
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                split_bf16(qv[r] * expf(bcr[r]), qlh[r * L::RK + kk], qll[r * L::RK + kk]);
                split_bf16(kv[r] * expf(run - bcr[r]), kgh[r * L::RK + kk], kgl[r * L::RK + kk]);
            }
        }
        __syncthreads();
        // dq_inter = dO S_[n-1]^T and dk_inter = V D_[n]^T: warp w owns keys 8 NPW w .. + 8 NPW;
        // scaled by Lambda / Gamma they are this tile's partials of dq and dk
        {
            const int arow = (lane % 8) + 8 * ((lane / 8) % 2), acol = 8 * (lane / 16);
            const int brow = lane % 8, bcol = 8 * ((lane / 8) % 2);
            float cq[L::NPW][4], ck[L::NPW][4];
#pragma unroll
            for (int nt = 0; nt < L::NPW; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) cq[nt][e] = ck[nt][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < DVT / 16; ++ks) {
                uint32_t ad0, ad1, ad2, ad3, av0, av1, av2, av3;
                ldsm_x4(ddb + arow * L::RS + 16 * ks + acol, ad0, ad1, ad2, ad3);
                ldsm_x4(vvb + arow * L::RS + 16 * ks + acol, av0, av1, av2, av3);
#pragma unroll
                for (int nt = 0; nt < L::NPW; ++nt) {
                    const int key0 = 8 * (warp * L::NPW + nt);
                    uint32_t b0, b1;
                    ldsm_x2(Sph + (key0 + brow) * L::RS + 16 * ks + bcol, b0, b1);
                    mma16816(cq[nt], ad0, ad1, ad2, ad3, b0, b1);
                    ldsm_x2(Spl + (key0 + brow) * L::RS + 16 * ks + bcol, b0, b1);
                    mma16816(cq[nt], ad0, ad1, ad2, ad3, b0, b1);
                    ldsm_x2(Dbh + (key0 + brow) * L::RS + 16 * ks + bcol, b0, b1);
                    mma16816(ck[nt], av0, av1, av2, av3, b0, b1);
                    ldsm_x2(Dbl + (key0 + brow) * L::RS + 16 * ks + bcol, b0, b1);
                    mma16816(ck[nt], av0, av1, av2, av3, b0, b1);
                }
            }
            const size_t prow = ((size_t)tile * BH + bh) * a.T + t0;
#pragma unroll
            for (int nt = 0; nt < L::NPW; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = g + 8 * (e / 2), key = 8 * (warp * L::NPW + nt) + 2 * tq + (e % 2);
                    if (t < nr) {
                        const float b = bc[t * DK + key], bend = bc[(CS - 1) * DK + key];
                        a.Pq[(prow + t) * DK + key] = expf(b) * cq[nt][e];
                        a.Pk[(prow + t) * DK + key] = expf(bend - b) * ck[nt][e];
                    }
                }
        }
        // dv (this tile) = (K (.) Gamma) D_[n] + P^T dO: warp w owns columns 8 w .. 8 w + 7
        {
            const int arow = (lane % 8) + 8 * ((lane / 8) % 2), acol = 8 * (lane / 16);
            const int brow = (lane % 8) + 8 * ((lane / 8) % 2);
            float cv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int ks = 0; ks < DK / 16; ++ks) {
                uint32_t ah0, ah1, ah2, ah3, al0, al1, al2, al3, bh0, bh1, bl0, bl1;
                ldsm_x4(kgh + arow * L::RK + 16 * ks + acol, ah0, ah1, ah2, ah3);
                ldsm_x4(kgl + arow * L::RK + 16 * ks + acol, al0, al1, al2, al3);
                ldsm_x2_t(Dbh + (16 * ks + brow) * L::RS + 8 * warp, bh0, bh1);
                ldsm_x2_t(Dbl + (16 * ks + brow) * L::RS + 8 * warp, bl0, bl1);
                mma16816(cv, ah0, ah1, ah2, ah3, bh0, bh1);
                mma16816(cv, ah0, ah1, ah2, ah3, bl0, bl1);
                mma16816(cv, al0, al1, al2, al3, bh0, bh1);
            }
            const int j = 8 * warp + 2 * tq;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s = g + 8 * (e / 2), jj = j + (e % 2);
                float acc = cv[e];
                for (int t = s; t < CS; ++t) acc = fmaf(A[t * CS + s], __bfloat162float(ddb[t * L::RS + jj]), acc);
                if (s < nr && jj < jn) a.gv[((size_t)bh * a.T + t0 + s) * a.dv + j0 + jj] = acc;
            }
        }
        __syncthreads();   // D's bf16 parts are read above and rewritten below
        // D <- Diag(gamma) D + (Q (.) Lambda)^T dO, then its hi + lo parts
        {
            const int brow = (lane % 8) + 8 * ((lane / 8) % 2);
            const int mi = lane / 8, arow = (lane % 8) + 8 * (mi / 2), acol = 8 * (mi % 2);
#pragma unroll
            for (int u = 0; u < L::TPW; ++u) {
                const int id = warp * L::TPW + u, m = id / 8, n = id % 8;
                uint32_t a0, a1, a2, a3, b0, b1;
                ldsm_x2_t(ddb + brow * L::RS + 8 * n, b0, b1);
                const float g0 = gam[16 * m + g], g1 = gam[16 * m + g + 8];
                Dacc[u][0] *= g0; Dacc[u][1] *= g0; Dacc[u][2] *= g1; Dacc[u][3] *= g1;
                ldsm_x4_t(qlh + arow * L::RK + 16 * m + acol, a0, a1, a2, a3);
                mma16816(Dacc[u], a0, a1, a2, a3, b0, b1);
                ldsm_x4_t(qll + arow * L::RK + 16 * m + acol, a0, a1, a2, a3);
                mma16816(Dacc[u], a0, a1, a2, a3, b0, b1);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = 16 * m + g + 8 * (e / 2), j = 8 * n + 2 * tq + (e % 2);
                    split_bf16(Dacc[u][e], Dbh[key * L::RS + j], Dbl[key * L::RS + j]);
                }
            }
        }
    }
    if (a.gS0)
#pragma unroll
        for (int u = 0; u < L::TPW; ++u) {
            const int id = warp * L::TPW + u, m = id / 8, n = id % 8;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = 16 * m + g + 8 * (e / 2), j = 8 * n + 2 * tq + (e % 2);
                if (j < jn) a.gS0[(size_t)bh * ST + (size_t)key * a.dv + j0 + j] = Dacc[u][e];
            }
        }
}

// ---------------------------------------------------------------- dq, dk and dlog b
template <typename Tin>
__global__ void __launch_bounds__(NT) gla_bwd_finish_kernel(BwdArgs a)
{
    const size_t n = (size_t)a.B * a.H * a.T * a.dk, plane = n;
    const int BH = a.B * a.H;
    for (size_t e = (size_t)blockIdx.x * NT + threadIdx.x; e < n; e += (size_t)gridDim.x * NT) {
        float sq = 0.f, sk = 0.f;
        for (int tl = 0; tl < a.nplanes; ++tl) {
            sq += a.Pq[tl * plane + e];
            sk += a.Pk[tl * plane + e];
        }
        a.gq[e] = sq;
        a.gk[e] = sk;
        if (a.dla) {
            float lb = ld_in<Tin>(static_cast<const Tin*>(a.q), e) * sq - ld_in<Tin>(static_cast<const Tin*>(a.k), e) * sk;
            const int kk = (int)(e % a.dk);
            const size_t bt = e / a.dk;
            if ((int)(bt % a.T) == a.T - 1) {
                const int bh = (int)(bt / a.T);
                for (int tl = 0; tl < a.ndvt; ++tl) lb += a.bnd[((size_t)tl * BH + bh) * a.dk + kk];
            }
            a.dla[e] = lb;
        }
    }
}

// ---------------------------------------------------------------- reverse cumulative sum over tokens
// of a [BH][T][width] array (dlog b over keys, or the bilinear gate's terms over value
// columns); grid (BH, ceil(width / 32)); 8 segments of tokens x 32 columns per CTA
constexpr int RS_SEG = NT / 32;
__global__ void __launch_bounds__(NT) gla_bwd_revsum_kernel(BwdArgs a, const float* src, float* out, int width)
{
    __shared__ float tot[RS_SEG][32];
    const int bh = blockIdx.x, lane = threadIdx.x % 32, seg = threadIdx.x / 32;
    const int kk = blockIdx.y * 32 + lane;
    const int L = (a.T + RS_SEG - 1) / RS_SEG;
    const int ta = seg * L, tb = min(a.T, ta + L);
    const bool on = kk < width;
    const float* in = src + (size_t)bh * a.T * width + kk;
    float s = 0.f;
    if (on)
        for (int t = ta; t < tb; ++t) s += in[(size_t)t * width];
    tot[seg][lane] = s;
    __syncthreads();
    float run = 0.f;
    for (int g = RS_SEG - 1; g > seg; --g) run += tot[g][lane];
    if (on) {
        float* o = out + (size_t)bh * a.T * width + kk;
        for (int t = tb - 1; t >= ta; --t) {
            run += in[(size_t)t * width];
            o[(size_t)t * width] = run;
        }
    }
}

// ---------------------------------------------------------------- per-token / per-head gate gradients
// per token: one warp per (bh, t) row sums its dk values
__global__ void __launch_bounds__(NT) gla_bwd_token_gate_kernel(BwdArgs a)
{
    const size_t rows = (size_t)a.B * a.H * a.T;
    const int lane = threadIdx.x % 32;
    for (size_t r = ((size_t)blockIdx.x * NT + threadIdx.x) / 32; r < rows; r += (size_t)gridDim.x * NT / 32) {
        float s = 0.f;
        for (int x = lane; x < a.dk; x += 32) s += a.dla[r * a.dk + x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) a.glog[r] = s;
    }
}

// per head: the sum over b, t and keys in two levels with a fixed partition (bitwise
// reproducible): CTA (h, j) sums slice j of head h's B * T * dk values, then one thread per
// head adds the HG_SPLIT partial sums in order
constexpr int HG_SPLIT = 64;
__global__ void __launch_bounds__(NT) gla_bwd_head_gate_part_kernel(BwdArgs a, float* part)
{
    __shared__ float red[NT];
    const int h = blockIdx.x, j = blockIdx.y;
    const size_t per = (size_t)a.T * a.dk, tot = (size_t)a.B * per;   // per is a multiple of 16
    const size_t L = ((tot + HG_SPLIT - 1) / HG_SPLIT + 3) / 4 * 4;
    const size_t e0 = min(tot, (size_t)j * L), e1 = min(tot, e0 + L);
    float s = 0.f;
    for (size_t e = e0 + (size_t)threadIdx.x * 4; e < e1; e += (size_t)NT * 4) {
        const size_t b = e / per, off = e % per;   // a float4 never crosses from one b to the next
        const float4 v = *reinterpret_cast<const float4*>(a.dla + ((size_t)b * a.H + h) * per + off);
        s += (v.x + v.y) + (v.z + v.w);
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = NT / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) part[(size_t)h * HG_SPLIT + j] = red[0];
}

__global__ void gla_bwd_head_gate_sum_kernel(const float* part, float* glog, int H)
{
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    float s = 0.f;
    for (int j = 0; j < HG_SPLIT; ++j) s += part[(size_t)h * HG_SPLIT + j];
    glog[h] = s;
}

cudaError_t launch_head_gate(const BwdArgs& a, float* part, cudaStream_t s)
{
    gla_bwd_head_gate_part_kernel<<<dim3(a.H, HG_SPLIT), NT, 0, s>>>(a, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    gla_bwd_head_gate_sum_kernel<<<(a.H + 127) / 128, 128, 0, s>>>(part, a.glog, a.H);
    return cudaGetLastError();
}

size_t states_smem(int dk) { return sizeof(float) * ((size_t)dk * DVT + (size_t)CS * dk + CS * DVT + dk + DVT); }
size_t chunks_smem(int dk) {
    return sizeof(float) * (2 * (size_t)dk * DVT + 3 * (size_t)CS * dk + 2 * CS * DVT + 2 * CS * CS +
                            (NT / 32) * CS * CS + dk + 3 * CS * DVT + 2 * DVT);
}

struct BwdPlan {
    int nch = 0, ndvt = 0;
    size_t off_S = 0, off_Pq = 0, off_Pk = 0, off_Ag = 0, off_bnd = 0, off_dla = 0, off_dlbe = 0, off_hpart = 0,
           bytes = 0;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

BwdPlan bwd_plan(const gla_bwd_params* p)
{
    BwdPlan pl;
    const size_t BH = (size_t)p->B * p->H;
    pl.nch = (p->T + CS - 1) / CS;
    pl.ndvt = (p->dv + DVT - 1) / DVT;
    size_t off = 0;
    pl.off_S = off;   off = up256(off + BH * pl.nch * p->dk * p->dv * 4);
    pl.off_Pq = off;  off = up256(off + (size_t)(pl.ndvt + 1) * BH * p->T * p->dk * 4);
    pl.off_Pk = off;  off = up256(off + (size_t)(pl.ndvt + 1) * BH * p->T * p->dk * 4);
    pl.off_Ag = off;  off = up256(off + BH * pl.nch * CS * CS * 4);
    pl.off_bnd = off; off = up256(off + (size_t)pl.ndvt * BH * p->dk * 4);
    pl.off_dla = off; off = up256(off + BH * p->T * p->dk * 4);
    if (p->gate == GLA_GATE_BILINEAR) {
        pl.off_dlbe = off; off = up256(off + BH * p->T * p->dv * 4);
    }
    if (p->gate == GLA_GATE_HEAD_SCALAR) {
        pl.off_hpart = off; off = up256(off + (size_t)p->H * HG_SPLIT * 4);
    }
    pl.bytes = off;
    return pl;
}

bool tc_shape_ok(const gla_bwd_params* p) {
    return p->dtype == GLA_BF16 && (p->dk == 64 || p->dk == 128 || p->dk == 256) && p->gate != GLA_GATE_BILINEAR;
}

// The 64-row chunk-parallel form on tcgen05 (gla_bwd_chunk.cu and the chunk pass's state
// sweeps): bf16, dk in {128, 256}, dv a multiple of 128, q, k, v and grad_O on 16-byte
// boundaries (tensor-memory-access copies).
bool chunk_shape_ok(const gla_bwd_params* p) {
    const long long BH = (long long)p->B * p->H;
    const long long rows = (((long long)p->T + kChunk - 1) / kChunk) * kChunk;
    auto al16 = [](const void* x) { return reinterpret_cast<uintptr_t>(x) % 16 == 0; };
    return p->dtype == GLA_BF16 && (p->dk == 128 || p->dk == 256) && p->dv % kDvTile == 0 &&
           p->gate != GLA_GATE_BILINEAR && BH <= 65535 && BH * rows < (1LL << 31) &&
           BH * (rows / kChunk) * p->dv < (1LL << 31) && al16(p->q) && al16(p->k) && al16(p->v) && al16(p->grad_O);
}

enum BwdKind { BWD_SIMT, BWD_SPLIT, BWD_CHUNK };

BwdKind bwd_kind(const gla_bwd_params* p) {
    if (p->dtype == GLA_FP32 || p->path == GLA_PATH_SIMT) return BWD_SIMT;
    if (p->path == GLA_PATH_SPLIT) return BWD_SPLIT;
    if (p->T > 0 && chunk_shape_ok(p)) return BWD_CHUNK;   // AUTO or TENSOR
    return tc_shape_ok(p) ? BWD_SPLIT : BWD_SIMT;
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 148;
    return n;
}

// Sequence segments of the chunk form's two sweeps: as for the forward pass, a split pays
// when the B * H * dv-tile sweeps are well under one wave and the sequence is long.
int bwd_segments(const gla_bwd_params* p, int nch, int sms)
{
    const long long units = (long long)p->B * p->H * (p->dv / kDvTile);
    if (units * 2 > sms || nch < 16) return 1;
    long long n = sms / units;
    if (n > nch / 8) n = nch / 8;
    return n < 1 ? 1 : (int)n;
}

// Workspace of the chunk form: the prep's Q (.) Lambda, K (.) Gamma (gated), scores and
// chunk decays; the two sweeps' chunk states H and D (bf16); S_T and the boundary term
// (gate gradient with grad_ST); the per-token gate terms (scalar gates; the per-key
// gradient takes them in place) and their per-chunk totals.
struct ChunkPlan {
    int nch = 0, Tpad = 0;
    int nseg = 1, cps = 0;   // the sweeps' sequence split
    size_t off_segS = 0, off_segin = 0;
    bool raw = false;
    size_t off_qt = 0, off_kt = 0, off_A = 0, off_gam = 0, off_H = 0, off_D = 0, off_ST = 0, off_bnd = 0,
           off_dla = 0, off_ctot = 0, off_hpart = 0, bytes = 0;
};

ChunkPlan chunk_plan(const gla_bwd_params* p)
{
    ChunkPlan c;
    const size_t BH = (size_t)p->B * p->H;
    c.nch = (p->T + kChunk - 1) / kChunk;
    c.Tpad = c.nch * kChunk;
    c.raw = p->gate == GLA_GATE_NONE;
    size_t off = 0;
    if (!c.raw) {
        c.off_qt = off; off = up256(off + BH * c.Tpad * p->dk * 2);
        c.off_kt = off; off = up256(off + BH * c.Tpad * p->dk * 2);
    }
    c.off_A = off;   off = up256(off + BH * c.nch * kChunk * kChunk * 2);
    c.off_gam = off; off = up256(off + BH * c.nch * p->dk * 4);
    c.off_H = off;   off = up256(off + BH * c.nch * p->dv * p->dk * 2);
    c.off_D = off;   off = up256(off + BH * c.nch * p->dv * p->dk * 2);
    c.nseg = bwd_segments(p, c.nch, device_sm_count());
    c.cps = (c.nch + c.nseg - 1) / c.nseg;
    c.nseg = (c.nch + c.cps - 1) / c.cps;
    if (c.nseg > 1) {   // each segment's zero-start state, then its entering state (both sweeps in turn)
        c.off_segS = off;  off = up256(off + BH * c.nseg * p->dk * p->dv * 4);
        c.off_segin = off; off = up256(off + BH * c.nseg * p->dk * p->dv * 4);
    }
    if (p->grad_log_g) {
        if (p->grad_ST) {
            c.off_ST = off;  off = up256(off + BH * p->dk * p->dv * 4);
            c.off_bnd = off; off = up256(off + BH * p->dk * 4);
        }
        if (p->gate != GLA_GATE_PER_KEY) {   // the per-key gradient is written in place
            c.off_dla = off; off = up256(off + BH * p->T * p->dk * 4);
        }
        c.off_ctot = off; off = up256(off + BH * c.nch * p->dk * 4);
        if (p->gate == GLA_GATE_HEAD_SCALAR) {
            c.off_hpart = off; off = up256(off + (size_t)p->H * HG_SPLIT * 4);
        }
    }
    c.bytes = off;
    return c;
}

bool span_overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

gla_status bwd_validate(const gla_bwd_params* p)
{
    if (!p) return GLA_ERR_INVALID_ARG;
    if (p->B <= 0 || p->H <= 0 || p->T < 0 || p->dk <= 0 || p->dv <= 0) return GLA_ERR_INVALID_ARG;
    if (p->dtype != GLA_BF16 && p->dtype != GLA_FP32) return GLA_ERR_INVALID_ARG;
    if (p->gate < GLA_GATE_NONE || p->gate > GLA_GATE_BILINEAR) return GLA_ERR_INVALID_ARG;
    const bool bil = p->gate == GLA_GATE_BILINEAR;
    if (bil != (p->log_b != nullptr) && !(bil && p->T == 0)) return GLA_ERR_INVALID_ARG;
    if (!bil && p->grad_log_b) return GLA_ERR_INVALID_ARG;
    if (p->dk % 16 != 0 || p->dv % 16 != 0) return GLA_ERR_INVALID_ARG;
    if ((long long)p->B * p->H > 65535) return GLA_ERR_INVALID_ARG;
    if (p->gate == GLA_GATE_NONE && (p->log_g || p->grad_log_g)) return GLA_ERR_INVALID_ARG;
    if (p->gate != GLA_GATE_NONE && !p->log_g && (p->T > 0 || p->gate == GLA_GATE_HEAD_SCALAR))
        return GLA_ERR_INVALID_ARG;
    if (p->T > 0 && (!p->q || !p->k || !p->v || !p->grad_O || !p->grad_q || !p->grad_k || !p->grad_v))
        return GLA_ERR_INVALID_ARG;
    if (p->path != GLA_PATH_AUTO && p->path != GLA_PATH_TENSOR && p->path != GLA_PATH_SIMT &&
        p->path != GLA_PATH_SPLIT)
        return GLA_ERR_INVALID_ARG;
    if (p->dk > NT) return GLA_ERR_UNSUPPORTED;
    if (p->path == GLA_PATH_TENSOR && !chunk_shape_ok(p)) return GLA_ERR_UNSUPPORTED;
    if (p->path == GLA_PATH_SPLIT && !tc_shape_ok(p)) return GLA_ERR_UNSUPPORTED;
    const size_t e = p->dtype == GLA_BF16 ? 2 : 4;
    if ((p->log_b && reinterpret_cast<uintptr_t>(p->log_b) % 4) ||
        (p->grad_log_b && reinterpret_cast<uintptr_t>(p->grad_log_b) % 4))
        return GLA_ERR_INVALID_ARG;
    const size_t BH = (size_t)p->B * p->H;
    const size_t nq = BH * p->T * p->dk, nv = BH * p->T * p->dv, ns = BH * p->dk * p->dv;
    const size_t ng = (p->gate == GLA_GATE_PER_KEY || p->gate == GLA_GATE_BILINEAR) ? nq
                    : p->gate == GLA_GATE_TOKEN_SCALAR ? BH * p->T
                    : p->gate == GLA_GATE_HEAD_SCALAR ? (size_t)p->H : 0;
    for (const void* ptr : {p->q, p->k, p->v, p->grad_O})
        if (ptr && reinterpret_cast<uintptr_t>(ptr) % e) return GLA_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)p->log_g, (const void*)p->S0, (const void*)p->grad_ST, (const void*)p->grad_q,
                            (const void*)p->grad_k, (const void*)p->grad_v, (const void*)p->grad_log_g,
                            (const void*)p->grad_S0})
        if (ptr && reinterpret_cast<uintptr_t>(ptr) % 4) return GLA_ERR_INVALID_ARG;
    if (p->workspace && reinterpret_cast<uintptr_t>(p->workspace) % 256) return GLA_ERR_INVALID_ARG;
    // outputs overlap no input and no other output
    const void* outs[] = {p->grad_q, p->grad_k, p->grad_v, p->grad_log_g, p->grad_S0, p->grad_log_b};
    const size_t osz[] = {nq * 4, nq * 4, nv * 4, ng * 4, ns * 4, nv * 4};
    const void* ins[] = {p->q, p->k, p->v, p->grad_O, p->log_g, p->S0, p->grad_ST, p->log_b};
    const size_t isz[] = {nq * e, nq * e, nv * e, nv * e, ng * 4, ns * 4, ns * 4, nv * 4};
    for (int i = 0; i < 6; ++i) {
        for (int j = 0; j < 8; ++j)
            if (span_overlap(outs[i], osz[i], ins[j], isz[j])) return GLA_ERR_INVALID_ARG;
        for (int j = i + 1; j < 6; ++j)
            if (span_overlap(outs[i], osz[i], outs[j], osz[j])) return GLA_ERR_INVALID_ARG;
    }
    return GLA_OK;
}

template <int DK>
cudaError_t launch_chunks_tc(const BwdArgs& a, int BH, cudaStream_t s)
{
    cudaError_t e;
    if (a.nch > 0) {
        const int sm1 = (int)intra_smem(DK);
        if ((e = cudaFuncSetAttribute(gla_bwd_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sm1)) !=
            cudaSuccess)
            return e;
        gla_bwd_intra_kernel<<<dim3(BH, a.nch), NT, sm1, s>>>(a, a.Ag);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int smem = TcLay<DK>::BYTES;
    if ((e = cudaFuncSetAttribute(gla_bwd_sweep_tc_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
        return e;
    gla_bwd_sweep_tc_kernel<DK><<<dim3(BH, a.ndvt), NT, smem, s>>>(a, a.Ag);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_states_tc(const BwdArgs& a, int BH, cudaStream_t s)
{
    const int smem = StLay<DK>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(gla_bwd_states_tc_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gla_bwd_states_tc_kernel<DK><<<dim3(BH, a.ndvt), NT, smem, s>>>(a);
    return cudaGetLastError();
}

// The gate gradient from the per-token terms dla: the reverse cumulative sum over tokens
// (per key: straight to grad_log_g), then the sums over keys (per token) or over batch rows,
// tokens and keys (per head).
cudaError_t launch_gate_tail(const BwdArgs& a, const gla_bwd_params& p, float* hpart, cudaStream_t s)
{
    cudaError_t e;
    const int BH = p.B * p.H;
    const size_t n = (size_t)BH * p.T * p.dk;
    if (a.glog && n > 0) {
        const bool per_key = p.gate == GLA_GATE_PER_KEY || p.gate == GLA_GATE_BILINEAR;
        gla_bwd_revsum_kernel<<<dim3(BH, (p.dk + 31) / 32), NT, 0, s>>>(a, a.dla, per_key ? a.glog : a.dla, p.dk);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (p.gate == GLA_GATE_TOKEN_SCALAR) {
            const size_t rows = (size_t)BH * p.T;
            const int grid = (int)((rows * 32 + NT - 1) / NT < 4096 ? (rows * 32 + NT - 1) / NT : 4096);
            gla_bwd_token_gate_kernel<<<grid, NT, 0, s>>>(a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    if (a.glog && p.gate == GLA_GATE_HEAD_SCALAR) {
        if (n == 0) return cudaMemsetAsync(a.glog, 0, (size_t)p.H * sizeof(float), s);
        if ((e = launch_head_gate(a, hpart, s)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}


// The chunk form in stages: the prep (Q (.) Lambda, K (.) Gamma, gamma, scores), the state
// sweep forward (H, and S_T), the sweep of dL/dS backward (D, and dS0), the boundary term
// rowsum(dST (.) S_T), the chunk-parallel gradients, the gate tail (the later chunks' totals
// added to each chunk's in-chunk sums; sums over keys for the scalar gates).
enum ChunkStage {
    CS_PREP, CS_SEG_FWD, CS_SCAN_FWD, CS_SWEEP_FWD, CS_SEG_REV, CS_SCAN_REV, CS_SWEEP_REV, CS_BOUNDARY, CS_GRADS,
    CS_GATE, CS_N
};

const char* chunk_stage_name(int k)
{
    switch (k) {
    case CS_PREP: return "gla_chunk_prep";
    case CS_SEG_FWD: return "gla_chunk_state";
    case CS_SCAN_FWD: return "gla_state_scan";
    case CS_SEG_REV: return "gla_chunk_dstate";
    case CS_SCAN_REV: return "gla_dstate_scan";
    case CS_SWEEP_FWD: return "gla_bwd_state_sweep";
    case CS_SWEEP_REV: return "gla_bwd_dstate_sweep";
    case CS_BOUNDARY: return "gla_bwd_boundary";
    case CS_GRADS: return "gla_bwd_grads";
    case CS_GATE: return "gla_bwd_gate_tail";
    }
    return "?";
}

// the stages the chunk form runs for *p, in order
int chunk_stages(const gla_bwd_params* p, int* out)
{
    const bool split = chunk_plan(p).nseg > 1;
    int n = 0;
    out[n++] = CS_PREP;
    if (split) { out[n++] = CS_SEG_FWD; out[n++] = CS_SCAN_FWD; }
    out[n++] = CS_SWEEP_FWD;
    if (split) { out[n++] = CS_SEG_REV; out[n++] = CS_SCAN_REV; }
    out[n++] = CS_SWEEP_REV;
    if (p->grad_log_g && p->grad_ST) out[n++] = CS_BOUNDARY;
    out[n++] = CS_GRADS;
    if (p->grad_log_g) out[n++] = CS_GATE;
    return n;
}

cudaError_t run_chunk_stage(const gla_bwd_params& p, const ChunkPlan& cp, uint8_t* w, int* status, int k,
                            cudaStream_t s)
{
    cudaError_t e;
    const int sms = device_sm_count();
    const int BH = p.B * p.H;
    const bool gated = p.gate != GLA_GATE_NONE;
    const void* qt = cp.raw ? p.q : static_cast<const void*>(w + cp.off_qt);
    const void* kt = cp.raw ? p.k : static_cast<const void*>(w + cp.off_kt);
    const long long kt_rows = cp.raw ? p.T : cp.Tpad;
    const float* gam = gated ? reinterpret_cast<const float*>(w + cp.off_gam) : nullptr;
    float* ST = cp.off_ST ? reinterpret_cast<float*>(w + cp.off_ST) : nullptr;
    float* bnd = cp.off_bnd ? reinterpret_cast<float*>(w + cp.off_bnd) : nullptr;
    const bool per_key = p.gate == GLA_GATE_PER_KEY;
    float* R = !p.grad_log_g ? nullptr : per_key ? p.grad_log_g : reinterpret_cast<float*>(w + cp.off_dla);
    float* ctot = p.grad_log_g ? reinterpret_cast<float*>(w + cp.off_ctot) : nullptr;
    switch (k) {
    case CS_PREP: {
        gla_fwd_params fp;
        std::memset(&fp, 0, sizeof(fp));
        fp.q = p.q; fp.k = p.k; fp.v = p.v; fp.log_g = p.log_g; fp.S0 = p.S0;
        fp.B = p.B; fp.H = p.H; fp.T = p.T; fp.dk = p.dk; fp.dv = p.dv;
        fp.dtype = p.dtype; fp.gate = p.gate; fp.path = GLA_PATH_TENSOR;
        Plan pl;
        pl.path = GLA_PATH_TENSOR;
        pl.nchunks = cp.nch; pl.Tpad = cp.Tpad; pl.n_dvt = p.dv / kDvTile; pl.raw_qk = cp.raw; pl.sms = sms;
        pl.off_qt = cp.off_qt; pl.off_kt = cp.off_kt; pl.off_A = cp.off_A; pl.off_gam = cp.off_gam;
        return launch_prep(fp, pl, w, status, s, false);
    }
    case CS_SEG_FWD:
    case CS_SEG_REV: {
        // each segment's state (or dL/dS contribution) from a zero start
        SegStateJob j;
        const bool fwd = k == CS_SEG_FWD;
        j.kt = fwd ? kt : qt; j.kt_rows = kt_rows; j.v = fwd ? p.v : p.grad_O; j.gam = gam;
        j.S_out = reinterpret_cast<float*>(w + cp.off_segS);
        j.reverse = !fwd;
        j.BH = BH; j.T = p.T; j.dk = p.dk; j.dv = p.dv; j.nch = cp.nch; j.cps = cp.cps; j.nseg = cp.nseg;
        return launch_seg_state_job(j, status, s);
    }
    case CS_SCAN_FWD:
    case CS_SCAN_REV: {
        // the state entering each segment (from S0), or the dL/dS leaving it (from dST)
        SegScanJob j;
        const bool fwd = k == CS_SCAN_FWD;
        j.S_start = fwd ? p.S0 : p.grad_ST;
        j.S_end = nullptr;
        j.gam = gam;
        j.segS = reinterpret_cast<const float*>(w + cp.off_segS);
        j.segin = reinterpret_cast<float*>(w + cp.off_segin);
        j.reverse = !fwd;
        j.BH = BH; j.dk = p.dk; j.dv = p.dv; j.nch = cp.nch; j.cps = cp.cps; j.nseg = cp.nseg;
        return launch_seg_scan_job(j, s);
    }
    case CS_SWEEP_FWD:
    case CS_SWEEP_REV: {
        StateSweep sw;
        const bool fwd = k == CS_SWEEP_FWD;
        sw.kt = fwd ? kt : qt; sw.kt_rows = kt_rows; sw.v = fwd ? p.v : p.grad_O; sw.gam = gam;
        sw.S_in = cp.nseg > 1 ? reinterpret_cast<const float*>(w + cp.off_segin) : (fwd ? p.S0 : p.grad_ST);
        sw.S_out = fwd ? ST : p.grad_S0;
        sw.Hst = w + (fwd ? cp.off_H : cp.off_D);
        sw.reverse = !fwd;
        sw.BH = BH; sw.T = p.T; sw.dk = p.dk; sw.dv = p.dv; sw.nch = cp.nch;
        sw.nseg = cp.nseg; sw.cps = cp.cps;
        return launch_state_sweep(sw, status, s);
    }
    case CS_BOUNDARY:
        return launch_bwd_boundary(p.grad_ST, ST, bnd, (long long)BH * p.dk, p.dv, sms, s);
    case CS_GRADS: {
        BwdGrads g;
        g.q = p.q; g.k = p.k; g.v = p.v; g.dO = p.grad_O; g.log_g = p.log_g;
        g.qt = qt; g.kt = kt; g.kt_rows = kt_rows;
        g.A = w + cp.off_A; g.gam = gam;
        g.Hst = w + cp.off_H; g.Dst = w + cp.off_D;
        g.bnd = (ST && bnd) ? bnd : nullptr;
        g.gq = p.grad_q; g.gk = p.grad_k; g.gv = p.grad_v;
        g.R = R; g.ctot = ctot;
        g.BH = BH; g.H = p.H; g.T = p.T; g.dk = p.dk; g.dv = p.dv; g.gate = p.gate; g.sms = sms;
        return launch_bwd_grads(g, status, s);
    }
    case CS_GATE: {
        // each chunk's terms are already summed over its later rows: add the totals of the
        // later chunks (their reverse cumulative sum, in place, then a shifted add)
        BwdArgs a;
        std::memset(&a, 0, sizeof(a));
        a.B = p.B; a.H = p.H; a.T = cp.nch; a.dk = p.dk; a.dv = p.dv; a.gate = p.gate;
        gla_bwd_revsum_kernel<<<dim3(BH, (p.dk + 31) / 32), NT, 0, s>>>(a, ctot, ctot, p.dk);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_bwd_gate_fixup(R, ctot, BH, p.T, p.dk, sms, s)) != cudaSuccess) return e;
        if (per_key) return cudaSuccess;
        a.T = p.T;
        a.glog = p.grad_log_g;
        a.dla = R;
        if (p.gate == GLA_GATE_TOKEN_SCALAR) {
            const size_t rows = (size_t)BH * p.T;
            const int grid = (int)((rows * 32 + NT - 1) / NT < 4096 ? (rows * 32 + NT - 1) / NT : 4096);
            gla_bwd_token_gate_kernel<<<grid, NT, 0, s>>>(a);
        } else {
            return launch_head_gate(a, reinterpret_cast<float*>(w + cp.off_hpart), s);
        }
        return cudaGetLastError();
    }
    }
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t launch_all(const BwdArgs& a, const gla_bwd_params& p, cudaStream_t s, bool use_tc)
{
    cudaError_t e;
    const int BH = p.B * p.H;
    if (a.nch > 0 && use_tc) {
        switch (p.dk) {
        case 64: e = launch_states_tc<64>(a, BH, s); break;
        case 128: e = launch_states_tc<128>(a, BH, s); break;
        default: e = launch_states_tc<256>(a, BH, s); break;
        }
        if (e != cudaSuccess) return e;
    } else if (a.nch > 0) {
        const size_t sm1 = states_smem(p.dk);
        if ((e = cudaFuncSetAttribute(gla_bwd_states_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sm1)) != cudaSuccess)
            return e;
        gla_bwd_states_kernel<Tin><<<dim3(BH, a.ndvt), NT, sm1, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // the reverse sweep (with no chunks it only sets dS0 = dST)
    if (use_tc) {
        switch (p.dk) {
        case 64: e = launch_chunks_tc<64>(a, BH, s); break;
        case 128: e = launch_chunks_tc<128>(a, BH, s); break;
        default: e = launch_chunks_tc<256>(a, BH, s); break;
        }
        if (e != cudaSuccess) return e;
    } else {
        const size_t sm2 = chunks_smem(p.dk);
        if ((e = cudaFuncSetAttribute(gla_bwd_chunks_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sm2)) != cudaSuccess)
            return e;
        gla_bwd_chunks_kernel<Tin><<<dim3(BH, a.ndvt), NT, sm2, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const size_t n = (size_t)BH * p.T * p.dk;
    if (n > 0) {
        const int grid = (int)((n + NT - 1) / NT < 4096 ? (n + NT - 1) / NT : 4096);
        gla_bwd_finish_kernel<Tin><<<grid, NT, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.glb && n > 0) {   // bilinear gate: dlog beta from the chunk sweep's per-token terms
        gla_bwd_revsum_kernel<<<dim3(BH, (p.dv + 31) / 32), NT, 0, s>>>(a, a.dlbe, a.glb, p.dv);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return launch_gate_tail(a, p, a.hpart, s);
}

}  // namespace
}  // namespace gla

using namespace gla;

extern "C" size_t gla_bwd_workspace_size(const gla_bwd_params* p)
{
    if (bwd_validate(p) != GLA_OK) return 0;
    return bwd_kind(p) == BWD_CHUNK ? chunk_plan(p).bytes : bwd_plan(p).bytes;
}

extern "C" gla_status gla_bwd(const gla_bwd_params* p, cudaStream_t stream)
{
    gla_status st = bwd_validate(p);
    if (st != GLA_OK) return st;
    const BwdKind kind = bwd_kind(p);
    if (kind == BWD_CHUNK) {
        const ChunkPlan cp = chunk_plan(p);
        if (!p->workspace || p->workspace_bytes < cp.bytes) return GLA_ERR_WORKSPACE;
        int* status = device_status_ptr();
        if (!status) return GLA_ERR_CUDA;
        int st[CS_N];
        const int n = chunk_stages(p, st);
        for (int i = 0; i < n; ++i)
            if (run_chunk_stage(*p, cp, static_cast<uint8_t*>(p->workspace), status, st[i], stream) != cudaSuccess)
                return GLA_ERR_CUDA;
        return GLA_OK;
    }
    const BwdPlan pl = bwd_plan(p);
    if (!p->workspace || p->workspace_bytes < pl.bytes) return GLA_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(p->workspace);
    BwdArgs a;
    a.q = p->q; a.k = p->k; a.v = p->v; a.dO = p->grad_O;
    a.log_g = p->log_g; a.S0 = p->S0; a.dST = p->grad_ST;
    a.gq = p->grad_q; a.gk = p->grad_k; a.gv = p->grad_v; a.glog = p->grad_log_g; a.gS0 = p->grad_S0;
    a.Sst = reinterpret_cast<float*>(w + pl.off_S);
    a.Pq = reinterpret_cast<float*>(w + pl.off_Pq);
    a.Pk = reinterpret_cast<float*>(w + pl.off_Pk);
    a.Ag = reinterpret_cast<float*>(w + pl.off_Ag);
    a.bnd = p->grad_log_g ? reinterpret_cast<float*>(w + pl.off_bnd) : nullptr;
    a.dla = p->grad_log_g ? reinterpret_cast<float*>(w + pl.off_dla) : nullptr;
    a.B = p->B; a.H = p->H; a.T = p->T; a.dk = p->dk; a.dv = p->dv; a.gate = p->gate;
    a.log_b = p->log_b;
    a.glb = p->grad_log_b;
    a.dlbe = p->gate == GLA_GATE_BILINEAR ? reinterpret_cast<float*>(w + pl.off_dlbe) : nullptr;
    a.hpart = p->gate == GLA_GATE_HEAD_SCALAR ? reinterpret_cast<float*>(w + pl.off_hpart) : nullptr;
    a.nch = pl.nch; a.ndvt = pl.ndvt;
    const bool use_tc = kind == BWD_SPLIT;
    a.nplanes = pl.ndvt + (use_tc ? 1 : 0);
    const cudaError_t e = p->dtype == GLA_FP32 ? launch_all<float>(a, *p, stream, false)
                                               : launch_all<__nv_bfloat16>(a, *p, stream, use_tc);
    return e == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

extern "C" int gla_bwd_num_stages(const gla_bwd_params* p)
{
    if (bwd_validate(p) != GLA_OK) return -1;
    if (bwd_kind(p) != BWD_CHUNK) return 1;
    int st[CS_N];
    return chunk_stages(p, st);
}

extern "C" const char* gla_bwd_stage_name(const gla_bwd_params* p, int stage)
{
    const int n = gla_bwd_num_stages(p);
    if (n < 0 || stage < 0 || stage >= n) return "invalid";
    if (bwd_kind(p) != BWD_CHUNK) return bwd_kind(p) == BWD_SPLIT ? "gla_bwd_split" : "gla_bwd_simt";
    int st[CS_N];
    chunk_stages(p, st);
    return chunk_stage_name(st[stage]);
}

extern "C" gla_status gla_bwd_stage(const gla_bwd_params* p, int stage, cudaStream_t stream)
{
    const int n = gla_bwd_num_stages(p);
    if (n < 0) return bwd_validate(p);
    if (stage < 0 || stage >= n) return GLA_ERR_INVALID_ARG;
    if (bwd_kind(p) != BWD_CHUNK) return gla_bwd(p, stream);
    const ChunkPlan cp = chunk_plan(p);
    if (!p->workspace || p->workspace_bytes < cp.bytes) return GLA_ERR_WORKSPACE;
    int* status = device_status_ptr();
    if (!status) return GLA_ERR_CUDA;
    int st[CS_N];
    chunk_stages(p, st);
    return run_chunk_stage(*p, cp, static_cast<uint8_t*>(p->workspace), status, st[stage], stream) == cudaSuccess
               ? GLA_OK
               : GLA_ERR_CUDA;
}
