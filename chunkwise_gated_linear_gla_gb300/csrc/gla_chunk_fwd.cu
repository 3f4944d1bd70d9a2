// gla_chunk_fwd: the chunk-serial tensor-core pass of the chunkwise GLA forward
// ("Gated Linear Attention Transformers with Hardware-Efficient Training",
// §4.2; the non-materialised FlashLinearAttention loop of §3.3 / Alg. 1 with
// the gated chunk recurrence). One CTA owns one (b, h), one tile of 128
// columns of dv and one segment of chunks; per chunk n of C = 64 rows:
//
//   epilogue  S   <- Diag(gamma_n) S_[n-1]    (TMEM fp32, gate scales rows)
//   MMA       S^T += V_n^T (K_n (.) Gamma_n)  (state, M=128 N=dk K=64)
//   epilogue  Sb  <- bf16(S_[n-1])            (TMEM, A operand; written once
//                                              the previous inter MMA is done)
//   MMA       O^T  = Sb^T (Q_n (.) Lambda_n)^T (inter, A from TMEM, N=64 K=dk)
//             O^T += V_n^T (P_n (.) M)^T      (intra, N=64 K=64)
//   epilogue  O^T TMEM -> registers -> bf16 smem tile -> TMA store
//
// Everything is transposed (M = dv) so each MMA uses all 128 TMEM lanes and
// the state's columns (dk) line up with the per-key gate. The state stays in
// tensor memory for the whole segment and never goes to HBM; Q (.) Lambda,
// K (.) Gamma, gamma and the masked intra-chunk scores come from
// gla_chunk_prep. Warp roles: 0 TMA producer, 1 MMA issuer (and TMEM
// owner), 2-9 epilogue in two groups of four warps, each owning half of the
// state's columns and half of each output tile. Only the decay of the state
// sits on the chunk-to-chunk critical path (state MMA -> decay -> next state
// MMA); the bf16 copy, the inter and intra MMAs and the output drain overlap
// with it. Every wait is bounded; on a timeout the CTA records an error code
// and winds down.
//
// The bilinear gate G_t = alpha_t^T beta_t (Table 1's DFW row; the chunkwise
// form of the paper's appendix on the general formulation) is the BIL
// instantiation. V arrives as V^ = V (.) D' (gla_value_prep), so the state
// and intra MMAs are unchanged; the decay also scales column j by
// gamma'[j] = exp(B'_C[j]); the inter MMA's bf16 state is S_[n-1] Diag(gamma');
// and the drain scales O[r][j] by exp(B'_r[j] - B'_C[j]), formed from log beta
// (a prefix sum for the first 32 rows, a suffix sum for the last 32). A head
// that gla_value_prep flagged out of range is left to the CUDA-core pass.
#include <cuda_bf16.h>

#include "gla_internal.h"
#include "sm100.cuh"
#include "tma_host.h"

namespace gla {
namespace {

using namespace sm100;

constexpr int C = kChunk;
constexpr int DVT = kDvTile;
constexpr int NSTAGE = 2;
constexpr int NT = 320;
constexpr int NEPI = 256;                         // epilogue threads (warps 2-9)
constexpr int BAR_EPI = 1, BAR_G0 = 2;            // named barriers (0 is __syncthreads)
constexpr uint64_t kTimeoutNs = 2000000000ull;    // 2 s per wait

enum { ERR_PRODUCER = 0x101, ERR_MMA = 0x102, ERR_EPI = 0x103 };

struct FwdArgs {
    const float* S_in;  long long s_in_bh, s_in_seg;
    float* S_out;       long long s_out_bh, s_out_seg;
    const float* gam;   // [BH][nchunks][dk], null without a gate
    int* status;
    int dv, nchunks, cps, mode, gated;
    // bilinear gate: lbc = B'_C [BH][nchunks][dv], the chunk's total log beta per column,
    // lb = log beta [BH][T][dv]. Per-head scalar gate (SCAL): lamh = log lambda [H]; chunks
    // that pass q_factored take raw q, and the drain scales output row r by lambda^(r+1).
    // (The union keeps this struct at 128 bytes, which the compiler keeps in registers; a
    // larger one went to the stack.)
    union { const float* lbc; float* Opart; };   // Opart: key halves (KH), fp32 [BH][T][dv]
    union { const float* lb; const float* lamh; };
    const int* skip;    // [BH] heads left to the CUDA-core pass
    int T, H;
};

template <int DK, bool BIL>
struct Lay {
    static constexpr int QB = DK * C * 2;
    static constexpr int KB = DK * C * 2;
    static constexpr int VB = DVT * C * 2;
    static constexpr int AB = C * C * 2;
    static constexpr int GB = DK * 4;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = QB;
    static constexpr int V_OFF = QB + KB;
    static constexpr int A_OFF = V_OFF + VB;
    static constexpr int G_OFF = A_OFF + AB;
    static constexpr int GVB = BIL ? DVT * 4 : 0;
    static constexpr int GV_OFF = G_OFF + GB;
    static constexpr int STAGE = (GV_OFF + GVB + 1023) / 1024 * 1024;
    static constexpr int OB = C * DVT * 2;
    static constexpr int O_OFF = NSTAGE * STAGE;
    static constexpr int BAR_OFF = O_OFF + 2 * OB;
    static constexpr int SMEM = BAR_OFF + 256 + 1024;
    static constexpr int TCOLS_USED = DK + DK / 2 + 2 * 64;
    static constexpr int TCOLS = TCOLS_USED <= 256 ? 256 : 512;
    static_assert(TCOLS_USED <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void fail(int* status, volatile int* abort_flag, int code) {
    *abort_flag = 1;
    atomicExch(status, code);
}

// All `n` threads of a named-barrier group agree on success (bar.red.or).
__device__ __forceinline__ bool group_all_ok(bool ok, int id, int n) {
    uint32_t bad;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(bad)
        : "r"(ok ? 0u : 1u), "r"(id), "r"(n)
        : "memory");
    return bad == 0;
}

__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// KH (keys wider than the tensor memory holds, dk = 2 DK): 0 = all keys; 1 = keys
// [0, DK) of 2 DK, O written as an fp32 partial (with the intra-chunk term);
// 2 = keys [DK, 2 DK), no intra-chunk term, the partial added before the bf16 store.
// Each half carries its own rows of the state: the gate scales rows, so the two
// halves' recurrences are independent and only their outputs add.
template <int DK, bool BIL, bool SCAL, int KH>
__global__ void __launch_bounds__(NT, 1)
gla_chunk_fwd_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmQr)
{
    using L = Lay<DK, BIL>;
    constexpr int HC = DK / 2;   // state columns per epilogue thread
    constexpr int DKT = KH ? 2 * DK : DK;    // keys of the head
    constexpr int KOFF = KH == 2 ? DK : 0;   // this CTA's first key
    if constexpr (BIL) {
        if (a.skip[blockIdx.y]) return;   // the whole CTA leaves before any setup
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
    uint64_t* full = bar + 0;      // [2] stage filled (TMA transaction count)
    uint64_t* empty = bar + 2;     // [2] stage consumed (MMA commit)
    uint64_t* s_ready = bar + 4;   // state decayed in TMEM (256 arrivals)
    uint64_t* s_done = bar + 5;    // state MMA of the chunk complete
    uint64_t* sb_free = bar + 6;   // inter MMA complete: bf16 state copy reusable
    uint64_t* o_full = bar + 7;    // [2] O accumulator complete
    uint64_t* o_empty = bar + 9;   // [2] O accumulator drained (256 arrivals)
    uint64_t* sb_ready = bar + 11; // bf16 state copy written (256 arrivals)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 12);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 13);
    uint64_t* mma_fin = bar + 14;  // every MMA of the CTA complete (the issuer's last commit)

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y, seg = blockIdx.z;
    const int dv0 = blockIdx.x * DVT;
    const int c_begin = seg * a.cps;
    const int c_end = min(a.nchunks, c_begin + a.cps);
    const int nloc = max(0, c_end - c_begin);
    const bool want_out = a.mode != kModeSegState;
    const bool gated = a.gated != 0;
    // per-head scalar gate: whether chunk ch's query factor is left to this pass (the prep
    // made the same decision on the same float, rows x log lambda)
    const float lam_h = SCAL ? a.lamh[bh % a.H] : 0.f;
    auto q_fac = [&](int ch) -> bool { return SCAL && q_factored((float)min(C, a.T - ch * C) * lam_h); };

    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1); mbar_init(&full[1], 1);
        mbar_init(&empty[0], 1); mbar_init(&empty[1], 1);
        mbar_init(s_ready, NEPI); mbar_init(s_done, 1); mbar_init(sb_free, 1); mbar_init(sb_ready, NEPI);
        mbar_init(&o_full[0], 1); mbar_init(&o_full[1], 1);
        mbar_init(&o_empty[0], NEPI); mbar_init(&o_empty[1], NEPI);
        mbar_init(mma_fin, 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&tmQ); prefetch_tmap(&tmK); prefetch_tmap(&tmV); prefetch_tmap(&tmA); prefetch_tmap(&tmO);
        if (SCAL) prefetch_tmap(&tmQr);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, L::TCOLS);
        tmem_relinquish();
    }
    // Epilogue threads issue every load of their S_in columns (dv column d, HC keys)
    // before the set-up barrier, so the loads overlap the set-up and are all in flight
    // at once; they go to tensor memory after the barrier.
    constexpr int NB = HC / 32;
    uint32_t s_in[NB][32];
    if (warp >= 2) {
        const int d = (warp & 3) * 32 + lane, cb = ((warp - 2) >> 2) * HC;
        const float* sin = a.S_in ? a.S_in + bh * a.s_in_bh + seg * a.s_in_seg + dv0 + d : nullptr;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                s_in[b][i] = sin ? __float_as_uint(sin[(size_t)(cb + b * 32 + i) * a.dv]) : 0u;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS = tmem, tSb = tmem + DK, tO0 = tmem + DK + DK / 2;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int n = 0; n < nloc; ++n) {
                if (*abort_flag) break;
                const int st = n & 1, c = c_begin + n;
                if (n >= 2 && !mbar_wait(&empty[st], ((n >> 1) - 1) & 1, kTimeoutNs)) {
                    fail(a.status, abort_flag, ERR_PRODUCER);
                    break;
                }
                uint8_t* sb = sm + st * L::STAGE;
                const uint32_t bytes = L::KB + L::VB + (gated ? L::GB : 0) +
                                       (want_out ? L::QB + (KH == 2 ? 0 : L::AB) : 0) + L::GVB;
                mbar_arrive_expect_tx(&full[st], bytes);
                if (gated) bulk_load(sb + L::G_OFF, a.gam + ((size_t)bh * a.nchunks + c) * DKT + KOFF, L::GB, &full[st]);
                if constexpr (BIL)
                    bulk_load(sb + L::GV_OFF, a.lbc + ((size_t)bh * a.nchunks + c) * a.dv + dv0, L::GVB, &full[st]);
#pragma unroll
                for (int i = 0; i < DK / 64; ++i)
                    tma_load_3d(sb + L::K_OFF + i * 8192, &tmK, &full[st], KOFF + i * 64, c * C, bh);
                tma_load_3d(sb + L::V_OFF, &tmV, &full[st], dv0, c * C, bh);
                tma_load_3d(sb + L::V_OFF + 8192, &tmV, &full[st], dv0 + 64, c * C, bh);
                if (want_out) {
                    const CUtensorMap* mq = q_fac(c) ? &tmQr : &tmQ;
#pragma unroll
                    for (int i = 0; i < DK / 64; ++i)
                        tma_load_3d(sb + L::Q_OFF + i * 8192, mq, &full[st], KOFF + i * 64, c * C, bh);
                    if (KH != 2) tma_load_2d(sb + L::A_OFF, &tmA, &full[st], 0, (bh * a.nchunks + c) * C);
                }
                // L2 prefetch two chunks ahead, beyond what the two shared-memory stages
                // hold; the tiles all dv-tile CTAs of this head share are split among them
                const int cp = c + 2;
                if (cp < c_end) {
                    prefetch_l2_tile_3d(&tmV, dv0, cp * C, bh);
                    prefetch_l2_tile_3d(&tmV, dv0 + 64, cp * C, bh);
                    const int nt = gridDim.x, me = blockIdx.x;
                    int item = 0;
#pragma unroll
                    for (int i = 0; i < DK / 64; ++i, ++item)
                        if (item % nt == me) prefetch_l2_tile_3d(&tmK, KOFF + i * 64, cp * C, bh);
                    if (want_out) {
                        const CUtensorMap* mq = q_fac(cp) ? &tmQr : &tmQ;
#pragma unroll
                        for (int i = 0; i < DK / 64; ++i, ++item)
                            if (item % nt == me) prefetch_l2_tile_3d(mq, KOFF + i * 64, cp * C, bh);
                        if (KH != 2 && item % nt == me) prefetch_l2_tile_2d(&tmA, 0, (bh * a.nchunks + cp) * C);
                        ++item;
                    }
                    if (gated && item % nt == me)
                        prefetch_l2(a.gam + ((size_t)bh * a.nchunks + cp) * DKT + KOFF, L::GB);
                }
                issued = n + 1;
            }
            // no copy may land after the CTA exits: wait for the last fills
            for (int n = max(0, issued - 2); n < issued; ++n) mbar_wait(&full[n & 1], (n >> 1) & 1, kTimeoutNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_state = idesc_bf16(128, DK, true, true);
            const uint32_t id_inter = idesc_bf16(128, 64, false, false);
            const uint32_t id_intra = idesc_bf16(128, 64, true, false);
            for (int n = 0; n < nloc; ++n) {
                if (*abort_flag) break;
                const int st = n & 1;
                bool ok = mbar_wait(&full[st], (n >> 1) & 1, kTimeoutNs);
                ok = ok && mbar_wait(s_ready, n & 1, kTimeoutNs);
                if (!ok) {
                    fail(a.status, abort_flag, ERR_MMA);
                    break;
                }
                tc_fence_after();
                const uint32_t sb = smem_u32(sm + st * L::STAGE);
                const uint32_t sQ = sb + L::Q_OFF, sK = sb + L::K_OFF, sV = sb + L::V_OFF, sA = sb + L::A_OFF;
                // state: S^T += V^T (K (.) Gamma); both operands MN-major
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tS, sdesc(sV + kk * 2048, 8192, 1024, kSwizzle128),
                           sdesc(sK + kk * 2048, 8192, 1024, kSwizzle128), id_state, 1);
                mma_commit(s_done);
                if (want_out) {
                    ok = mbar_wait(sb_ready, n & 1, kTimeoutNs);
                    if (ok && n >= 2) ok = mbar_wait(&o_empty[n & 1], ((n >> 1) - 1) & 1, kTimeoutNs);
                    if (!ok) {
                        fail(a.status, abort_flag, ERR_MMA);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tO = tO0 + (n & 1) * 64;
                    // inter: O^T = Sb^T (Q (.) Lambda)^T, A (the bf16 state) from TMEM
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk)
                        mma_ts(tO, tSb + kk * 8, sdesc(sQ + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128),
                               id_inter, kk > 0);
                    mma_commit(sb_free);
                    // intra: O^T += V^T (P (.) M)^T (the second key half leaves it to the first)
                    if (KH != 2) {
#pragma unroll
                        for (int kk = 0; kk < C / 16; ++kk)
                            mma_ss(tO, sdesc(sV + kk * 2048, 8192, 1024, kSwizzle128),
                                   sdesc(sA + kk * 32, 16, 1024, kSwizzle128), id_intra, 1);
                    }
                    mma_commit(&o_full[n & 1]);
                }
                mma_commit(&empty[st]);
            }
            // one last commit tracks every MMA issued above: after an abort as on the normal
            // path, none may still run when the TMEM is freed at the end
            mma_commit(mma_fin);
            mbar_wait(mma_fin, 0, kTimeoutNs);
        }
    } else {
        // ---------------------------------------------------------- epilogue warps (2 groups of 4)
        // Group g owns state columns [g*DK/2, (g+1)*DK/2) and output rows [g*32, g*32+32)
        // of every chunk; the warp's TMEM lane quarter is (warp % 4).
        const int grp = (warp - 2) >> 2;
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const int d = (warp & 3) * 32 + lane;   // dv column within the tile
        const int cb = grp * HC;                 // first state column of this group
        const int gt = threadIdx.x - 64 - grp * 128;   // thread index within the group
        const int bar_grp = BAR_G0 + grp;
#pragma unroll
        for (int b = 0; b < NB; ++b) tmem_st32(tS + lb + cb + b * 32, s_in[b]);
        tmem_wait_st();
        // drain the O accumulator of chunk m: TMEM -> registers -> bf16 smem tile -> TMA store;
        // lbc_m is B'_C[d] of chunk m (bilinear gate)
        auto drain = [&](int m, float lbc_m) -> bool {
            const int b = m & 1;
            float w[32];
            const bool fq = SCAL && q_fac(c_begin + m);   // per-head gate: output rows take lambda^(r+1)
            if constexpr (BIL) {
                // log beta of this thread's 32 rows of chunk m (rows past T add nothing), and an
                // L2 prefetch of chunk m+2's rows, one 128-byte line per thread
                const int row0 = (c_begin + m) * C + grp * 32;
                const float* lp = a.lb + ((size_t)bh * a.T + row0) * a.dv + dv0 + d;
#pragma unroll
                for (int t = 0; t < 32; ++t) w[t] = row0 + t < a.T ? lp[(size_t)t * a.dv] : 0.f;
                const int prow = (c_begin + m + 2) * C + gt / 4 + grp * 32;
                if (c_begin + m + 2 < c_end && prow < a.T)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.lb + ((size_t)bh * a.T + prow) * a.dv + dv0 +
                                                                 (gt & 3) * 32));
            }
            const int orow = (c_begin + m) * C + grp * 32;   // this thread's first row of chunk m
            if constexpr (KH == 2) {
                // the first key half's fp32 partial of this thread's 32 rows (rows past T: none)
                const float* pp = a.Opart + ((size_t)bh * a.T + orow) * a.dv + dv0 + d;
#pragma unroll
                for (int t = 0; t < 32; ++t) w[t] = orow + t < a.T ? pp[(size_t)t * a.dv] : 0.f;
            }
            const bool ok = mbar_wait(&o_full[b], (m >> 1) & 1, kTimeoutNs);
            if (!group_all_ok(ok, BAR_EPI, NEPI)) return false;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld32(tO0 + b * 64 + lb + grp * 32, r);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&o_empty[b]);
            if constexpr (BIL) {
                // exp(B'_r - B'_C): rows 0-31 from the prefix sum, rows 32-63 from the suffix sum.
                // Exponents are within [-kVGuard, kVGuard]; the fast exponential's error there is
                // far below the bf16 rounding of O (the parity tests hold the bf16 tolerance).
                if (grp == 0) {
                    float acc = -lbc_m;
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        acc += w[t];
                        w[t] = __expf(acc);
                    }
                } else {
                    float acc = 0.f;
#pragma unroll
                    for (int t = 31; t >= 0; --t) {
                        const float x = w[t];
                        w[t] = __expf(acc);
                        acc -= x;
                    }
                }
#pragma unroll
                for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * w[t]);
            } else if (SCAL && fq) {
                // (r + 1) log lambda lies in [-kQGuard, 0] for every row r of the chunk
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    r[t] = __float_as_uint(__uint_as_float(r[t]) * __expf((float)(grp * 32 + t + 1) * lam_h));
            }
            if constexpr (KH == 2) {
#pragma unroll
                for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) + w[t]);
            }
            if constexpr (KH == 1) {
                // the partial goes out in fp32, one coalesced 128-byte row segment per warp and row
                float* pp = a.Opart + ((size_t)bh * a.T + orow) * a.dv + dv0 + d;
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    if (orow + t < a.T) pp[(size_t)t * a.dv] = __uint_as_float(r[t]);
                return true;
            }
            // the store issued from this half-buffer two chunks ago must have read it
            if (gt == 0) bulk_wait_read1();
            named_bar_sync(bar_grp, 128);
            uint8_t* tile = sm + L::O_OFF + b * L::OB;
            __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(tile) + (d >> 6) * (C * 64) + grp * 32 * 64 + (d & 63);
#pragma unroll
            for (int t = 0; t < 32; ++t) ob[t * 64] = __float2bfloat16_rn(__uint_as_float(r[t]));
            fence_proxy_async_smem();
            named_bar_sync(bar_grp, 128);
            if (gt == 0) {
                const int c = c_begin + m;
                tma_store_3d(&tmO, tile + grp * 32 * 64 * 2, dv0, c * C + grp * 32, bh);
                tma_store_3d(&tmO, tile + C * 64 * 2 + grp * 32 * 64 * 2, dv0 + 64, c * C + grp * 32, bh);
                bulk_commit();
            }
            return true;
        };
        bool alive = true;
        uint32_t P[HC / 2];   // bf16 pairs of S_[n-1] (this thread's columns), kept until the copy is free
        float lbc_prev = 0.f, lbc_cur = 0.f;   // B'_C[d] of chunks n-1 and n (bilinear gate)
        for (int n = 0; n < nloc && alive; ++n) {
            bool ok = true;
            if (n >= 1) ok = mbar_wait(s_done, (n - 1) & 1, kTimeoutNs);
            if (ok && gated) ok = mbar_wait(&full[n & 1], (n >> 1) & 1, kTimeoutNs);
            if (!group_all_ok(ok, BAR_EPI, NEPI)) {
                alive = false;
                break;
            }
            tc_fence_after();
            const float* g = reinterpret_cast<const float*>(sm + (n & 1) * L::STAGE + L::G_OFF) + cb;
            float gvd = 1.f;   // gamma'[d] (bilinear gate)
            if constexpr (BIL) {
                lbc_cur = reinterpret_cast<const float*>(sm + (n & 1) * L::STAGE + L::GV_OFF)[d];
                gvd = expf(lbc_cur);
            }
            // part 1: S <- Diag(gamma_n) S_[n-1] (and keep bf16(S_[n-1]) in registers)
#pragma unroll
            for (int c2 = 0; c2 < HC; c2 += 64) {
                uint32_t r0[32], r1[32];
                tmem_ld32(tS + lb + cb + c2, r0);
                tmem_ld32(tS + lb + cb + c2 + 32, r1);
                tmem_wait_ld();
                if constexpr (BIL) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * gvd);
                        r1[i] = __float_as_uint(__uint_as_float(r1[i]) * gvd);
                    }
                }
                if (want_out) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        P[c2 / 2 + i] = pack_bf16(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                        P[c2 / 2 + 16 + i] = pack_bf16(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
                    }
                }
                if (gated) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * g[c2 + i]);
                        r1[i] = __float_as_uint(__uint_as_float(r1[i]) * g[c2 + 32 + i]);
                    }
                    tmem_st32(tS + lb + cb + c2, r0);
                    tmem_st32(tS + lb + cb + c2 + 32, r1);
                }
            }
            if (gated) tmem_wait_st();
            tc_fence_before();
            mbar_arrive(s_ready);
            if (!want_out) continue;
            // part 2: bf16 copy of S_[n-1] for the inter MMA, once the previous one is consumed
            ok = (n == 0) || mbar_wait(sb_free, (n - 1) & 1, kTimeoutNs);
            if (!group_all_ok(ok, BAR_EPI, NEPI)) {
                alive = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c2 = 0; c2 < HC; c2 += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = P[c2 / 2 + i];
                tmem_st16(tSb + lb + (cb + c2) / 2, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(sb_ready);
            if (n >= 1 && !drain(n - 1, lbc_prev)) {
                alive = false;
                break;
            }
            lbc_prev = lbc_cur;
        }
        // The final state is complete once the last state MMA is (before the last inter
        // and intra MMAs): its stores go out while those run, then the last O drain.
        if (alive && nloc > 0) {
            const bool ok = mbar_wait(s_done, (nloc - 1) & 1, kTimeoutNs);
            if (group_all_ok(ok, BAR_EPI, NEPI)) {
                tc_fence_after();
                if (a.S_out) {
                    float* so = a.S_out + bh * a.s_out_bh + seg * a.s_out_seg + dv0 + d;
#pragma unroll
                    for (int b = 0; b < NB; ++b) tmem_ld32(tS + lb + cb + b * 32, s_in[b]);
                    tmem_wait_ld();
#pragma unroll
                    for (int b = 0; b < NB; ++b)
#pragma unroll
                        for (int i = 0; i < 32; ++i) so[(size_t)(cb + b * 32 + i) * a.dv] = __uint_as_float(s_in[b][i]);
                }
            } else {
                alive = false;
            }
        }
        if (alive && want_out && nloc > 0 && !drain(nloc - 1, lbc_prev)) alive = false;
        if (!alive && gt == 0) fail(a.status, abort_flag, ERR_EPI);
        if (gt == 0) bulk_wait0();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TCOLS);
    }
}

bool map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, CUtensorMapSwizzle swz,
          uint32_t rows = 64) {
    uint64_t dims[3] = {d0, d1, d2};
    uint64_t str[2] = {d0 * 2, d0 * d1 * 2};
    uint32_t box[3] = {64, rows, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box, swz);
}

template <int DK, bool BIL, bool SCAL, int KH = 0>
cudaError_t launch_dk(const FwdArgs& a, dim3 grid, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                      const CUtensorMap& A, const CUtensorMap& o, const CUtensorMap& qr, cudaStream_t s) {
    using L = Lay<DK, BIL>;
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_fwd_kernel<DK, BIL, SCAL, KH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    gla_chunk_fwd_kernel<DK, BIL, SCAL, KH><<<grid, NT, L::SMEM, s>>>(a, q, k, v, A, o, qr);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_fwd(const gla_fwd_params& p, const Plan& pl, void* ws, int mode, int* status, cudaStream_t s,
                             int kh)
{
    uint8_t* base = static_cast<uint8_t*>(ws);
    const uint64_t BH = (uint64_t)p.B * p.H;
    const void* qb = pl.raw_qk ? p.q : base + pl.off_qt;
    const void* kb = pl.raw_qk ? p.k : base + pl.off_kt;
    const uint64_t qrows = pl.raw_qk ? (uint64_t)p.T : (uint64_t)pl.Tpad;
    CUtensorMap mq, mk, mv, ma, mo, mqr;
    if (!map3(&mq, qb, p.dk, qrows, BH, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    // raw q for the chunks of a per-head scalar gate whose query factor this pass applies
    const bool qfac = q_factor_offload(p);
    if (qfac) {
        if (!map3(&mqr, p.q, p.dk, p.T, BH, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    } else {
        mqr = mq;
    }
    if (!map3(&mk, kb, p.dk, qrows, BH, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    const bool bil = p.gate == GLA_GATE_BILINEAR;
    const void* vb = bil ? base + pl.off_vh : p.v;   // bilinear gate: V (.) D' from gla_value_prep
    if (!map3(&mv, vb, p.dv, p.T, BH, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    if (!map3(&mo, p.O, p.dv, p.T, BH, CU_TENSOR_MAP_SWIZZLE_NONE, 32)) return cudaErrorInvalidValue;
    {
        uint64_t dims[2] = {64, BH * (uint64_t)pl.nchunks * 64};
        uint64_t str[1] = {128};
        uint32_t box[2] = {64, 64};
        if (!make_tmap(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base + pl.off_A, dims, str, box,
                       CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    FwdArgs a;
    const long long st = (long long)p.dk * p.dv;
    a.S_in = nullptr; a.s_in_bh = 0; a.s_in_seg = 0;
    a.S_out = nullptr; a.s_out_bh = 0; a.s_out_seg = 0;
    if (mode == kModeFull) {
        a.S_in = p.S0; a.s_in_bh = st;
        a.S_out = p.ST; a.s_out_bh = st;
    } else if (mode == kModeSegState) {
        a.S_out = reinterpret_cast<float*>(base + pl.off_segS); a.s_out_bh = st * pl.nseg; a.s_out_seg = st;
    } else {
        a.S_in = reinterpret_cast<const float*>(base + pl.off_segin); a.s_in_bh = st * pl.nseg; a.s_in_seg = st;
    }
    a.gam = reinterpret_cast<const float*>(base + pl.off_gam);
    a.status = status;
    a.dv = p.dv; a.nchunks = pl.nchunks;
    a.cps = (mode == kModeFull) ? pl.nchunks : pl.chunks_per_seg;
    a.mode = mode;
    a.gated = p.gate != GLA_GATE_NONE;
    a.lbc = bil ? reinterpret_cast<const float*>(base + pl.off_lbc) : nullptr;
    a.lb = p.log_b;
    if (qfac) a.lamh = p.log_g;
    a.skip = bil ? reinterpret_cast<const int*>(base + pl.off_flag) : nullptr;
    a.T = p.T;
    a.H = p.H;
    dim3 grid(pl.n_dvt, (unsigned)BH, mode == kModeFull ? 1 : pl.nseg);
    if (kh) {
        // dk = 512 in two key halves of 256: each half its own rows of S0 / S_T, the first
        // half's O an fp32 partial in the workspace that the second half adds
        if (mode != kModeFull || bil || qfac || p.dk != 512) return cudaErrorInvalidValue;
        const size_t koff = kh == 2 ? 256 : 0;
        a.S_in = p.S0 ? p.S0 + koff * p.dv : nullptr;
        a.S_out = p.ST ? p.ST + koff * p.dv : nullptr;
        a.Opart = reinterpret_cast<float*>(base + pl.off_opart);
        return kh == 1 ? launch_dk<256, false, false, 1>(a, grid, mq, mk, mv, ma, mo, mqr, s)
                       : launch_dk<256, false, false, 2>(a, grid, mq, mk, mv, ma, mo, mqr, s);
    }
    if (bil) {
        if (mode != kModeFull) return cudaErrorInvalidValue;   // no sequence split with the bilinear gate
        switch (p.dk) {
        case 64: return launch_dk<64, true, false>(a, grid, mq, mk, mv, ma, mo, mqr, s);
        case 128: return launch_dk<128, true, false>(a, grid, mq, mk, mv, ma, mo, mqr, s);
        case 256: return launch_dk<256, true, false>(a, grid, mq, mk, mv, ma, mo, mqr, s);
        }
        return cudaErrorInvalidValue;
    }
    if (qfac) {
        switch (p.dk) {
        case 64: return launch_dk<64, false, true>(a, grid, mq, mk, mv, ma, mo, mqr, s);
        case 128: return launch_dk<128, false, true>(a, grid, mq, mk, mv, ma, mo, mqr, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (p.dk) {
    case 64: return launch_dk<64, false, false>(a, grid, mq, mk, mv, ma, mo, mqr, s);
    case 128: return launch_dk<128, false, false>(a, grid, mq, mk, mv, ma, mo, mqr, s);
    case 256: return launch_dk<256, false, false>(a, grid, mq, mk, mv, ma, mo, mqr, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gla
