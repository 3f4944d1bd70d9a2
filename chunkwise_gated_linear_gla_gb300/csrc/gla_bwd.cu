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
//
// Kernels: gla_bwd_states (forward sweep, writes the state after every
// chunk), gla_bwd_chunks (reverse sweep per (b,h, 64 dv columns): partial dq
// and dk over the tile's columns, dv, dS0), gla_bwd_finish (sums the partials
// in a fixed order, dlog b), gla_bwd_revsum (reverse cumulative sum over
// tokens), gla_bwd_token_gate / gla_bwd_head_gate (per-token or per-head gate
// gradients). Every reduction has a fixed order, so results are bitwise
// reproducible.
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
    float* Pq;     // [ndvt][BH][T][dk] dq partial per dv tile
    float* Pk;     // [ndvt][BH][T][dk] dk partial per dv tile
    float* bnd;    // [ndvt][BH][dk] rowsum(dST (.) S_T) partial per dv tile
    float* dla;    // [BH][T][dk] dlog b, then dlog alpha (per key)
    int B, H, T, dk, dv, gate, nch, ndvt;
};

template <typename T> __device__ __forceinline__ float ld_in(const T* p, size_t i);
template <> __device__ __forceinline__ float ld_in<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

// log alpha_t for key kk of head bh (0 without a gate)
__device__ __forceinline__ float log_alpha(const BwdArgs& a, int bh, int t, int kk) {
    switch (a.gate) {
    case GLA_GATE_HEAD_SCALAR: return a.log_g[bh % a.H];
    case GLA_GATE_TOKEN_SCALAR: return a.log_g[(size_t)bh * a.T + t];
    case GLA_GATE_PER_KEY: return a.log_g[((size_t)bh * a.T + t) * a.dk + kk];
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
        for (int i = tid; i < CS * DVT; i += NT) {
            const int r = i / DVT, j = i % DVT;
            vv[i] = (r < nr && j < jn) ? ld_in<Tin>(v, (size_t)(t0 + r) * a.dv + j0 + j) : 0.f;
        }
        for (int x = tid; x < dk; x += NT) {
            float bcr[CS], run = 0.f;
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                run += r < nr ? log_alpha(a, bh, t0 + r, x) : 0.f;
                bcr[r] = run;
            }
            gam[x] = expf(run);
#pragma unroll
            for (int r = 0; r < CS; ++r)
                kt[r * dk + x] = r < nr ? ld_in<Tin>(k, (size_t)(t0 + r) * dk + x) * expf(run - bcr[r]) : 0.f;
        }
        __syncthreads();
        // S <- Diag(gamma) S + (K (.) Gamma)^T V, 16 columns of one row per step, and keep it
        float* out = a.Sst + ((size_t)bh * a.nch + c) * dk * a.dv + j0;
        for (int it = tid; it < dk * (DVT / 16); it += NT) {
            const int x = it % dk, g0 = (it / dk) * 4;
            const float gx = gam[x];
            float4 acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 w = ld4(S + swz(x, 4 * (g0 + u)));
                acc[u] = make_float4(gx * w.x, gx * w.y, gx * w.z, gx * w.w);
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
        for (int p = tid; p < CS * CS; p += NT) {
            const int t = p / CS, s = p % CS;
            float acc = 0.f;
            if (s <= t)
#pragma unroll
                for (int g = 0; g < DVT / 4; ++g) acc = dot4(ld4(dd + t * DVT + 4 * g), ld4(vv + s * DVT + 4 * g), acc);
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
#pragma unroll 2
            for (int g = 0; g < DVT / 4; ++g) {
                const float4 sp = ld4(Sp + swz(kk, 4 * g)), dg = ld4(D + swz(kk, 4 * g));
#pragma unroll
                for (int t = 0; t < CS; ++t) {
                    aq[t] = dot4(sp, ld4(dd + t * DVT + 4 * g), aq[t]);
                    ak[t] = dot4(dg, ld4(vv + t * DVT + 4 * g), ak[t]);
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
            if (s < nr && 4 * g < jn) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int x = 0; x < dk; ++x) fma4(acc, kr[s * dk + x], ld4(D + swz(x, 4 * g)));
                for (int t = s; t < CS; ++t) fma4(acc, A[t * CS + s], ld4(dd + t * DVT + 4 * g));
                float* o = a.gv + ((size_t)bh * a.T + t0 + s) * a.dv + j0 + 4 * g;
                o[0] = acc.x; o[1] = acc.y; o[2] = acc.z; o[3] = acc.w;
            }
        }
        __syncthreads();
        // D <- Diag(gamma) D + (Q (.) Lambda)^T dO, 16 columns of one row per step
        for (int it = tid; it < dk * (DVT / 16); it += NT) {
            const int x = it % dk, g0 = (it / dk) * 4;
            const float gx = gam[x];
            float4 acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 w = ld4(D + swz(x, 4 * (g0 + u)));
                acc[u] = make_float4(gx * w.x, gx * w.y, gx * w.z, gx * w.w);
            }
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                const float qx = qr[r * dk + x];
#pragma unroll
                for (int u = 0; u < 4; ++u) fma4(acc[u], qx, ld4(dd + r * DVT + 4 * (g0 + u)));
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

// ---------------------------------------------------------------- dq, dk and dlog b
template <typename Tin>
__global__ void __launch_bounds__(NT) gla_bwd_finish_kernel(BwdArgs a)
{
    const size_t n = (size_t)a.B * a.H * a.T * a.dk, plane = n;
    const int BH = a.B * a.H;
    for (size_t e = (size_t)blockIdx.x * NT + threadIdx.x; e < n; e += (size_t)gridDim.x * NT) {
        float sq = 0.f, sk = 0.f;
        for (int tl = 0; tl < a.ndvt; ++tl) {
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
// grid (BH, ceil(dk / 32)); 8 segments of tokens x 32 keys per CTA
constexpr int RS_SEG = NT / 32;
__global__ void __launch_bounds__(NT) gla_bwd_revsum_kernel(BwdArgs a, float* out)
{
    __shared__ float tot[RS_SEG][32];
    const int bh = blockIdx.x, lane = threadIdx.x % 32, seg = threadIdx.x / 32;
    const int kk = blockIdx.y * 32 + lane;
    const int L = (a.T + RS_SEG - 1) / RS_SEG;
    const int ta = seg * L, tb = min(a.T, ta + L);
    const bool on = kk < a.dk;
    const float* in = a.dla + (size_t)bh * a.T * a.dk + kk;
    float s = 0.f;
    if (on)
        for (int t = ta; t < tb; ++t) s += in[(size_t)t * a.dk];
    tot[seg][lane] = s;
    __syncthreads();
    float run = 0.f;
    for (int g = RS_SEG - 1; g > seg; --g) run += tot[g][lane];
    if (on) {
        float* o = out + (size_t)bh * a.T * a.dk + kk;
        for (int t = tb - 1; t >= ta; --t) {
            run += in[(size_t)t * a.dk];
            o[(size_t)t * a.dk] = run;
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

// per head: one CTA per h sums b, t and keys
__global__ void __launch_bounds__(NT) gla_bwd_head_gate_kernel(BwdArgs a)
{
    __shared__ float part[NT];
    const int h = blockIdx.x;
    const size_t per = (size_t)a.T * a.dk;
    float s = 0.f;
    for (int b = 0; b < a.B; ++b) {
        const float* p = a.dla + ((size_t)b * a.H + h) * per;
        for (size_t e = threadIdx.x; e < per; e += NT) s += p[e];
    }
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = NT / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) a.glog[h] = part[0];
}

size_t states_smem(int dk) { return sizeof(float) * ((size_t)dk * DVT + (size_t)CS * dk + CS * DVT + dk); }
size_t chunks_smem(int dk) {
    return sizeof(float) * (2 * (size_t)dk * DVT + 3 * (size_t)CS * dk + 2 * CS * DVT + 2 * CS * CS +
                            (NT / 32) * CS * CS + dk);
}

struct BwdPlan {
    int nch = 0, ndvt = 0;
    size_t off_S = 0, off_Pq = 0, off_Pk = 0, off_bnd = 0, off_dla = 0, bytes = 0;
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
    pl.off_Pq = off;  off = up256(off + (size_t)pl.ndvt * BH * p->T * p->dk * 4);
    pl.off_Pk = off;  off = up256(off + (size_t)pl.ndvt * BH * p->T * p->dk * 4);
    pl.off_bnd = off; off = up256(off + (size_t)pl.ndvt * BH * p->dk * 4);
    pl.off_dla = off; off = up256(off + BH * p->T * p->dk * 4);
    pl.bytes = off;
    return pl;
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
    if (p->gate < GLA_GATE_NONE || p->gate > GLA_GATE_TOKEN_SCALAR) return GLA_ERR_INVALID_ARG;
    if (p->dk % 16 != 0 || p->dv % 16 != 0) return GLA_ERR_INVALID_ARG;
    if ((long long)p->B * p->H > 65535) return GLA_ERR_INVALID_ARG;
    if (p->gate == GLA_GATE_NONE && (p->log_g || p->grad_log_g)) return GLA_ERR_INVALID_ARG;
    if (p->gate != GLA_GATE_NONE && !p->log_g && (p->T > 0 || p->gate == GLA_GATE_HEAD_SCALAR))
        return GLA_ERR_INVALID_ARG;
    if (p->T > 0 && (!p->q || !p->k || !p->v || !p->grad_O || !p->grad_q || !p->grad_k || !p->grad_v))
        return GLA_ERR_INVALID_ARG;
    if (p->dk > NT) return GLA_ERR_UNSUPPORTED;
    const size_t e = p->dtype == GLA_BF16 ? 2 : 4;
    const size_t BH = (size_t)p->B * p->H;
    const size_t nq = BH * p->T * p->dk, nv = BH * p->T * p->dv, ns = BH * p->dk * p->dv;
    const size_t ng = p->gate == GLA_GATE_PER_KEY ? nq : p->gate == GLA_GATE_TOKEN_SCALAR ? BH * p->T
                    : p->gate == GLA_GATE_HEAD_SCALAR ? (size_t)p->H : 0;
    for (const void* ptr : {p->q, p->k, p->v, p->grad_O})
        if (ptr && reinterpret_cast<uintptr_t>(ptr) % e) return GLA_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)p->log_g, (const void*)p->S0, (const void*)p->grad_ST, (const void*)p->grad_q,
                            (const void*)p->grad_k, (const void*)p->grad_v, (const void*)p->grad_log_g,
                            (const void*)p->grad_S0})
        if (ptr && reinterpret_cast<uintptr_t>(ptr) % 4) return GLA_ERR_INVALID_ARG;
    if (p->workspace && reinterpret_cast<uintptr_t>(p->workspace) % 256) return GLA_ERR_INVALID_ARG;
    // outputs overlap no input and no other output
    const void* outs[] = {p->grad_q, p->grad_k, p->grad_v, p->grad_log_g, p->grad_S0};
    const size_t osz[] = {nq * 4, nq * 4, nv * 4, ng * 4, ns * 4};
    const void* ins[] = {p->q, p->k, p->v, p->grad_O, p->log_g, p->S0, p->grad_ST};
    const size_t isz[] = {nq * e, nq * e, nv * e, nv * e, ng * 4, ns * 4, ns * 4};
    for (int i = 0; i < 5; ++i) {
        for (int j = 0; j < 7; ++j)
            if (span_overlap(outs[i], osz[i], ins[j], isz[j])) return GLA_ERR_INVALID_ARG;
        for (int j = i + 1; j < 5; ++j)
            if (span_overlap(outs[i], osz[i], outs[j], osz[j])) return GLA_ERR_INVALID_ARG;
    }
    return GLA_OK;
}

template <typename Tin>
cudaError_t launch_all(const BwdArgs& a, const gla_bwd_params& p, cudaStream_t s)
{
    cudaError_t e;
    const int BH = p.B * p.H;
    if (a.nch > 0) {
        const size_t sm1 = states_smem(p.dk);
        if ((e = cudaFuncSetAttribute(gla_bwd_states_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sm1)) != cudaSuccess)
            return e;
        gla_bwd_states_kernel<Tin><<<dim3(BH, a.ndvt), NT, sm1, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // the reverse sweep (with no chunks it only sets dS0 = dST)
    const size_t sm2 = chunks_smem(p.dk);
    if ((e = cudaFuncSetAttribute(gla_bwd_chunks_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sm2)) != cudaSuccess)
        return e;
    gla_bwd_chunks_kernel<Tin><<<dim3(BH, a.ndvt), NT, sm2, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t n = (size_t)BH * p.T * p.dk;
    if (n > 0) {
        const int grid = (int)((n + NT - 1) / NT < 4096 ? (n + NT - 1) / NT : 4096);
        gla_bwd_finish_kernel<Tin><<<grid, NT, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.glog && n > 0) {
        gla_bwd_revsum_kernel<<<dim3(BH, (p.dk + 31) / 32), NT, 0, s>>>(a, p.gate == GLA_GATE_PER_KEY ? a.glog : a.dla);
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
        gla_bwd_head_gate_kernel<<<p.H, NT, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace
}  // namespace gla

using namespace gla;

extern "C" size_t gla_bwd_workspace_size(const gla_bwd_params* p)
{
    if (bwd_validate(p) != GLA_OK) return 0;
    return bwd_plan(p).bytes;
}

extern "C" gla_status gla_bwd(const gla_bwd_params* p, cudaStream_t stream)
{
    gla_status st = bwd_validate(p);
    if (st != GLA_OK) return st;
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
    a.bnd = p->grad_log_g ? reinterpret_cast<float*>(w + pl.off_bnd) : nullptr;
    a.dla = p->grad_log_g ? reinterpret_cast<float*>(w + pl.off_dla) : nullptr;
    a.B = p->B; a.H = p->H; a.T = p->T; a.dk = p->dk; a.dv = p->dv; a.gate = p->gate;
    a.nch = pl.nch; a.ndvt = pl.ndvt;
    const cudaError_t e = p->dtype == GLA_FP32 ? launch_all<float>(a, *p, stream)
                                               : launch_all<__nv_bfloat16>(a, *p, stream);
    return e == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}
