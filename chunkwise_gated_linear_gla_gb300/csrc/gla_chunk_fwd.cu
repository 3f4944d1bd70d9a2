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
// gla_chunk_prep. Warp roles, by warpgroup: warp 0 TMA producer and warp 1
// MMA issuer (and TMEM owner) in the first; the state epilogue in the second
// and third (two groups of four warps, each owning half of the state's
// columns); the output drain in the fourth (four warps, one per TMEM lane
// quarter, every row of each output tile). setmaxnreg moves registers from
// the producer/MMA and drain warpgroups to the state epilogue. Only the decay
// of the state sits on the chunk-to-chunk critical path (state MMA -> decay ->
// next state MMA); the bf16 copy, the inter and intra MMAs and the output
// drain, on warps of their own, overlap with it. Every wait is bounded; on a
// timeout the CTA records an error code and winds down.
//
// The bilinear gate G_t = alpha_t^T beta_t (Table 1's DFW row; the chunkwise
// form of the paper's appendix on the general formulation) is the BIL
// instantiation. V arrives as V^ = V (.) D' (gla_value_prep), so the state
// and intra MMAs are unchanged; the decay also scales column j by
// gamma'[j] = exp(B'_C[j]); the inter MMA's bf16 state is S_[n-1] Diag(gamma');
// and the drain scales O[r][j] by exp(B'_r[j] - B'_C[j]), formed from log beta
// (a prefix sum for the first 32 rows, a suffix sum for the last 32). A head
// that gla_value_prep flagged out of range is left to the CUDA-core pass.
//
// The SC instantiations (dk <= 128, no gate or a per-head decay) form the
// intra-chunk scores themselves instead of reading the prep's tiles: warp 2's
// lane 0 issues P = Q K^T into spare tensor-memory columns as soon as a
// stage's Q and K have landed (rows in lanes 64-127, see the readout), warps 2
// and 3 mask it, scale it by lambda^-nr for the decay (with K (.) Gamma that is
// (q_r . k_s) lambda^-(s+1), the scores of the query-factored form), and write
// it as the bf16 score tile into the stage, and the intra MMA waits for it.
// Without a gate nothing is prepared at all: the pass reads q, k, v directly.
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
constexpr int NG = 4;                             // gate ring slots
constexpr int G_AHEAD = 2;                        // gate loads run this many chunks ahead of the stages
constexpr int PF_AHEAD = 2;                       // L2 prefetches run this many chunks ahead of the stage loads
constexpr int NT = 512;
constexpr int NEPI = 256;                         // state epilogue threads (warps 4-11)
constexpr int NDR = 128;                          // output drain threads (warps 12-15)
constexpr int BAR_EPI = 1, BAR_DR = 2, BAR_SC = 3;   // named barriers (0 is __syncthreads)
constexpr uint64_t kTimeoutNs = 2000000000ull;    // 2 s per wait
// Registers per thread of each warpgroup after setmaxnreg (the launch gives 128 each):
// producer/MMA, state epilogue (two warpgroups), drain.
// The split that compiles without spills differs between instantiations.
template <int DK, bool BIL, bool SC = false>
struct Regs {
    static constexpr bool wide = DK == 256 && !BIL;
    // SC: warps 2 and 3 of the first warpgroup also read the scores out
    static constexpr int ctl = wide ? 64 : SC ? 96 : 80, epi = wide ? 176 : 160, drain = wide || SC ? 96 : 112;
    static_assert(128 * (ctl + 2 * epi + drain) <= NT * 128, "register split");
};

enum { ERR_PRODUCER = 0x101, ERR_MMA = 0x102, ERR_EPI = 0x103, ERR_DRAIN = 0x104, ERR_READOUT = 0x105 };

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
    // state sweeps (kModeSweep / kModeSweepRev): the state entering each chunk's update,
    // bf16 [BH][nchunks][dv][dk] (row d holds column d of the state)
    __nv_bfloat16* Hst;
};
static_assert(sizeof(FwdArgs) <= 128, "FwdArgs stays within 128 bytes");

// SC: the pass forms the intra-chunk scores itself (see the kernel's header); the stage then
// holds the K tile before the Q tile, so that the score product's 128-row A operand can start
// 64 rows before the Q tile and place the chunk's rows in tensor-memory lanes 64-127.
template <int DK, bool BIL, bool SC = false>
struct Lay {
    static constexpr int QB = DK * C * 2;
    static constexpr int KB = DK * C * 2;
    static constexpr int VB = DVT * C * 2;
    static constexpr int AB = C * C * 2;
    static constexpr int GB = DK * 4;
    static constexpr int Q_OFF = SC ? KB : 0;
    static constexpr int K_OFF = SC ? 0 : QB;
    static constexpr int V_OFF = QB + KB;
    static constexpr int A_OFF = V_OFF + VB;
    static constexpr int STAGE = (A_OFF + AB + 1023) / 1024 * 1024;
    // operand stages: SC with dk <= 128 holds three (a stage is released only after the score
    // readout the intra MMA waits for, so its turnaround is longer), else two
    static constexpr int NST = (SC && DK <= 128) ? 3 : NSTAGE;
    // the gate ring: slot = the chunk's key decays gamma (and, bilinear gate, its column
    // decays' logs B'_C), NG chunks deep, so the decay of the state never waits for a stage
    static constexpr int GVB = BIL ? DVT * 4 : 0;
    static constexpr int GSL = GB + GVB;
    static constexpr int GR_OFF = NST * STAGE;
    static constexpr int OB = C * DVT * 2;
    static constexpr int O_OFF = GR_OFF + NG * GSL;
    static constexpr int BAR_OFF = O_OFF + 2 * OB;
    static constexpr int BARB = SC ? 512 : 256;   // SC: the stage barriers after the first 32 slots
    static constexpr int SMEM = BAR_OFF + BARB + 1024;
    static constexpr int TCOLS_USED = DK + DK / 2 + 2 * 64 + (SC ? 64 : 0);   // + the score accumulator
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
template <int DK, bool BIL, bool SCAL, int KH, bool SC>
__global__ void __launch_bounds__(NT, 1)
gla_chunk_fwd_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmQr)
{
    static_assert(!SC || (!BIL && KH == 0 && DK <= 128), "on-chip scores: no bilinear gate, dk <= 128");
    using L = Lay<DK, BIL, SC>;
    constexpr int HC = DK / 2;   // state columns per epilogue thread
    constexpr int DKT = KH ? 2 * DK : DK;    // keys of the head
    constexpr int KOFF = KH == 2 ? DK : 0;   // this CTA's first key
    if constexpr (BIL) {
        if (a.skip[blockIdx.y]) return;   // the whole CTA leaves before any setup
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
    constexpr int NST = L::NST;
    // [NST] stage's K and V tiles landed (TMA transaction count) / stage consumed (MMA commit)
    uint64_t* full = SC ? bar + 32 : bar + 0;
    uint64_t* empty = SC ? bar + 32 + NST : bar + 2;
    uint64_t* s_ready = bar + 4;   // state decayed in TMEM (256 arrivals)
    uint64_t* s_done = bar + 5;    // state MMA of the chunk complete
    uint64_t* sb_free = bar + 6;   // inter MMA complete: bf16 state copy reusable
    uint64_t* o_full = bar + 7;    // [2] O accumulator complete
    uint64_t* o_empty = bar + 9;   // [2] O accumulator drained (128 arrivals)
    uint64_t* sb_ready = bar + 11; // bf16 state copy written (256 arrivals)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 12);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 13);
    uint64_t* mma_fin = bar + 14;  // every MMA of the CTA complete (the issuer's last commit)
    uint64_t* gfull = bar + 15;    // [NG] gate ring slot filled (transaction count)
    uint64_t* gempty = bar + 15 + NG;   // [NG] gate ring slot read (256 arrivals)
    uint64_t* full_qa = SC ? bar + 32 + 2 * NST : bar + 15 + 2 * NG;   // [NST] stage's Q and score tiles landed
    volatile int* issued_ctr = reinterpret_cast<volatile int*>(bar + 17 + 2 * NG);   // chunks whose loads are out
    uint64_t* p_full = bar + 18 + 2 * NG;    // SC: score product complete
    uint64_t* p_ready = bar + 32 + 3 * NST;  // SC: [NST] masked bf16 scores written to the stage (64 arrivals)

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y, seg = blockIdx.z;
    const int dv0 = blockIdx.x * DVT;
    const int c_begin = seg * a.cps;
    const int c_end = min(a.nchunks, c_begin + a.cps);
    const int nloc = max(0, c_end - c_begin);
    const bool want_out = a.mode == kModeFull || a.mode == kModeSegOut;
    // the state sweeps keep the state entering every chunk; the reverse one walks the chunks
    // from the last (the backward's recurrence for dL/dS)
    const bool sweep = !BIL && !SCAL && !SC && KH == 0 && (a.mode == kModeSweep || a.mode == kModeSweepRev);
    const bool rev = sweep && a.mode == kModeSweepRev;
    auto chunk_of = [&](int j) { return rev ? c_end - 1 - j : c_begin + j; };
    const bool gated = a.gated != 0;
    // per-head scalar gate: whether chunk ch's query factor is left to this pass (the prep
    // made the same decision on the same float, rows x log lambda)
    const float lam_h = SCAL ? a.lamh[bh % a.H] : 0.f;
    auto q_fac = [&](int ch) -> bool { return SCAL && q_factored((float)min(C, a.T - ch * C) * lam_h); };
    // SC: whether chunk ch's scores are formed here (no gate: every chunk; per-head gate: the
    // chunks that take raw q) instead of read from the prep's score tiles
    auto sc_chunk = [&](int ch) -> bool { return SC && (!SCAL || q_fac(ch)); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&full_qa[i], 1);
            mbar_init(&empty[i], 1);
        }
        *issued_ctr = 0;
        mbar_init(s_ready, NEPI); mbar_init(s_done, 1); mbar_init(sb_free, 1); mbar_init(sb_ready, NEPI);
        mbar_init(&o_full[0], 1); mbar_init(&o_full[1], 1);
        mbar_init(&o_empty[0], NDR); mbar_init(&o_empty[1], NDR);
        mbar_init(mma_fin, 1);
        if (SC) {
            mbar_init(p_full, 1);
            for (int i = 0; i < NST; ++i) mbar_init(&p_ready[i], 64);
        }
        for (int i = 0; i < NG; ++i) {
            mbar_init(&gfull[i], 1);
            mbar_init(&gempty[i], NEPI);
        }
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&tmQ); prefetch_tmap(&tmK); prefetch_tmap(&tmV); prefetch_tmap(&tmA); prefetch_tmap(&tmO);
        if (SCAL) prefetch_tmap(&tmQr);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, L::TCOLS);
        tmem_relinquish();
    }
    constexpr int NB = HC / 32;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS = tmem, tSb = tmem + DK, tO0 = tmem + DK + DK / 2;
    const uint32_t tP = tO0 + 128;   // SC: the score accumulator, 64 columns (lanes 64-127)

    const int wg = warp >> 2;
    if (wg == 0) regs_dec<Regs<DK, BIL, SC>::ctl>();   // warp 2 prefetches; SC: warps 2 and 3 read the scores out
    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            // chunk j's gate decays into ring slot j % NG, once chunk j - NG's decay has read it
            auto load_g = [&](int j) -> bool {
                const int sl = j % NG, c = chunk_of(j);
                if (j >= NG && !mbar_wait(&gempty[sl], ((j / NG) - 1) & 1, kTimeoutNs)) return false;
                uint8_t* gs = sm + L::GR_OFF + sl * L::GSL;
                mbar_arrive_expect_tx(&gfull[sl], L::GSL);
                bulk_load(gs, a.gam + ((size_t)bh * a.nchunks + c) * DKT + KOFF, L::GB, &gfull[sl]);
                if constexpr (BIL)
                    bulk_load(gs + L::GB, a.lbc + ((size_t)bh * a.nchunks + c) * a.dv + dv0, L::GVB, &gfull[sl]);
                return true;
            };
            // launched with programmatic stream serialization (see launch_dk), the grid ahead
            // (gate prep or segment scan) may still run: wait for its writes before any load
            grid_dependency_wait();
            int issued = 0, gissued = 0;
            if (gated)
                for (; gissued < G_AHEAD && gissued < nloc; ++gissued) load_g(gissued);
            for (int n = 0; n < nloc; ++n) {
                if (*abort_flag) break;
                const int st = n % NST, c = chunk_of(n);
                if (n >= NST && !mbar_wait(&empty[st], ((n / NST) - 1) & 1, kTimeoutNs)) {
                    fail(a.status, abort_flag, ERR_PRODUCER);
                    break;
                }
                uint8_t* sb = sm + st * L::STAGE;
                // K and V first (the state MMA, on the chunk-to-chunk chain, needs only them),
                // then Q and the scores (the output MMAs) on a barrier of their own
                mbar_arrive_expect_tx(&full[st], L::KB + L::VB);
#pragma unroll
                for (int i = 0; i < DK / 64; ++i)
                    tma_load_3d(sb + L::K_OFF + i * 8192, &tmK, &full[st], KOFF + i * 64, c * C, bh);
                tma_load_3d(sb + L::V_OFF, &tmV, &full[st], dv0, c * C, bh);
                tma_load_3d(sb + L::V_OFF + 8192, &tmV, &full[st], dv0 + 64, c * C, bh);
                if (want_out) {
                    const bool ldA = KH != 2 && !sc_chunk(c);
                    mbar_arrive_expect_tx(&full_qa[st], L::QB + (ldA ? L::AB : 0));
                    const CUtensorMap* mq = q_fac(c) ? &tmQr : &tmQ;
#pragma unroll
                    for (int i = 0; i < DK / 64; ++i)
                        tma_load_3d(sb + L::Q_OFF + i * 8192, mq, &full_qa[st], KOFF + i * 64, c * C, bh);
                    if (ldA) tma_load_2d(sb + L::A_OFF, &tmA, &full_qa[st], 0, (bh * a.nchunks + c) * C);
                }
                *issued_ctr = n + 1;   // paces the L2 prefetches of warp 2
                issued = n + 1;
                if (gated && gissued < nloc) {
                    if (!load_g(gissued)) {
                        fail(a.status, abort_flag, ERR_PRODUCER);
                        break;
                    }
                    ++gissued;
                }
            }
            // no copy may land after the CTA exits: wait for the last fills
            for (int n = max(0, issued - NST); n < issued; ++n) {
                mbar_wait(&full[n % NST], (n / NST) & 1, kTimeoutNs);
                if (want_out) mbar_wait(&full_qa[n % NST], (n / NST) & 1, kTimeoutNs);
            }
            for (int j = max(0, gissued - NG); j < gissued; ++j) mbar_wait(&gfull[j % NG], (j / NG) & 1, kTimeoutNs);
        }
    } else if (warp == 2 || (SC && warp == 3)) {
        // ---------------------------------------------------------- L2 prefetcher (and SC readout)
        // Once the producer has issued chunk m's loads, pull chunk m + PFA's tiles into L2, so
        // that the stage loads, issued only when a stage frees up, find them there. The tiles
        // all dv-tile CTAs of this head share are split among them. Prefetches are hints: if
        // the producer stops (an abort) this thread just stops too.
        constexpr int PFA = SC ? PF_AHEAD + 1 : PF_AHEAD;   // SC: issued after the chunk's readout
        const uint64_t t_start = globaltimer();
        // bounded wait until the producer has issued chunk m's loads
        auto wait_issued = [&](int m) -> bool {
            while (*issued_ctr <= m) {
                if (*abort_flag || globaltimer() - t_start > kTimeoutNs) return false;
                __nanosleep(64);
            }
            return true;
        };
        auto prefetch = [&](int m) -> bool {
            if (!wait_issued(m)) return false;
            const int cp = chunk_of(m + PFA);
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
                if (KH != 2 && !sc_chunk(cp) && item % nt == me)
                    prefetch_l2_tile_2d(&tmA, 0, (bh * a.nchunks + cp) * C);
                ++item;
            }
            if (gated && item % nt == me && m + PFA + G_AHEAD < nloc)
                prefetch_l2(a.gam + ((size_t)bh * a.nchunks + chunk_of(m + PFA + G_AHEAD)) * DKT + KOFF, L::GB);
            return true;
        };
        if (!SC || !want_out) {
            if (warp == 2 && lane == 0)
                for (int m = 0; m + PFA < nloc; ++m)
                    if (!prefetch(m)) break;
        } else {
            // SC: warps 2 and 3 form the chunk's scores. Lane 0 of warp 2 issues the product
            // P = Q K^T (its own MMAs and commit, beside the issuer's) as soon as the stage's Q and
            // K have landed: both operands K-major, A = 128 rows from 64 rows before the Q tile
            // (the K tile's last 64-column slab, or the Q tile's previous one), so that the
            // chunk's rows r = 0..63 land in TMEM lanes 64-127, the lane quarters of warps 2 and 3.
            // Those turn it into the masked bf16 tile the intra MMA reads, in the stage's score
            // slot (which the producer leaves empty for these chunks): row r, 128-byte swizzle, as
            // the prep's tiles. Per-head gate: times lambda^-nr, which with K (.) Gamma gives the
            // factored scores (q_r . k_s) lambda^-(s+1). The product reads the stage, which the
            // issuer releases only after the intra MMA, which waits for this readout, which waits
            // for the product: so it is done before the stage is refilled.
            const int r = (warp - 2) * 32 + lane;
            const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t id_score = idesc_bf16(128, 64, false, false);
            const uint32_t sbase = smem_u32(sm);
            const uint64_t dQm0 = sdesc(sbase + L::Q_OFF - 8192, 16, 1024, kSwizzle128);
            const uint64_t dKk0 = sdesc(sbase + L::K_OFF, 16, 1024, kSwizzle128);
            bool alive = true, pf = true;
            for (int m = 0, j = 0; m < nloc && alive; ++m) {
                const int c = chunk_of(m), st = m % NST;
                if (sc_chunk(c)) {
                    bool ok = true;
                    if (warp == 2) {
                        if (lane == 0) {
                            // chunk m's loads issued first: its stage's barriers are then in chunk
                            // m's phase (chunks skipped above did not wait on them, and chunk m + NST
                            // cannot be loaded before this readout is done)
                            ok = wait_issued(m) && mbar_wait(&full[st], (m / NST) & 1, kTimeoutNs) &&
                                 mbar_wait(&full_qa[st], (m / NST) & 1, kTimeoutNs) && !*abort_flag;
                            if (ok) {
                                tc_fence_after();
                                const uint64_t so = (uint64_t)((st * L::STAGE) >> 4);
#pragma unroll
                                for (int kk = 0; kk < DK / 16; ++kk) {
                                    const uint64_t ko = so + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                                    mma_ss(tP, dQm0 + ko, dKk0 + ko, id_score, kk > 0);
                                }
                                mma_commit(p_full);
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                    }
                    ok = __all_sync(0xffffffffu, ok && mbar_wait(p_full, j & 1, kTimeoutNs) && !*abort_flag);
                    ++j;
                    if (ok) {
                        tc_fence_after();
                        const float fac = SCAL ? __expf(-(float)min(C, a.T - c * C) * lam_h) : 1.f;
                        uint8_t* row = sm + st * L::STAGE + L::A_OFF + r * 128;
                        // 16 bf16 pairs of key rows 32 h .. 32 h + 31 of row r, masked to s <= r
                        auto half = [&](int h, const uint32_t* v) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int col = 32 * h + 2 * i;   // key row s of the chunk
                                float x0 = __uint_as_float(v[2 * i]), x1 = __uint_as_float(v[2 * i + 1]);
                                if (SCAL) { x0 *= fac; x1 *= fac; }
                                pk[i] = pack_bf16(col <= r ? x0 : 0.f, col + 1 <= r ? x1 : 0.f);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                *reinterpret_cast<uint4*>(row + (((4 * h + i) ^ (r & 7)) << 4)) =
                                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        };
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t v[32];
                            tmem_ld32(tP + lb + 32 * h, v);
                            tmem_wait_ld();
                            half(h, v);
                        }
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(&p_ready[st]);
                    }
                    // both warps' loads of the accumulator are done before the next product
                    alive = group_all_ok(ok, BAR_SC, 64);
                    tc_fence_after();
                    if (!alive) break;
                }
                if (warp == 2 && lane == 0 && pf && m + PFA < nloc) pf = prefetch(m);
                __syncwarp();
            }
            if (!alive && lane == 0) fail(a.status, abort_flag, ERR_READOUT);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_state = idesc_bf16(128, DK, true, true);
            const uint32_t id_inter = idesc_bf16(128, 64, false, false);
            const uint32_t id_intra = idesc_bf16(128, 64, true, false);
            // Operand descriptors of stage 0, built once; a stage or a K step only moves the
            // start address, the low 14-bit field (addr >> 4) of the descriptor, and every
            // shared address here is below 2^18, so adding the offset >> 4 never carries out.
            const uint32_t s0 = smem_u32(sm);
            const uint64_t dV0 = sdesc(s0 + L::V_OFF, 8192, 1024, kSwizzle128);
            const uint64_t dK0 = sdesc(s0 + L::K_OFF, 8192, 1024, kSwizzle128);
            const uint64_t dQ0 = sdesc(s0 + L::Q_OFF, 16, 1024, kSwizzle128);
            const uint64_t dA0 = sdesc(s0 + L::A_OFF, 16, 1024, kSwizzle128);
            // bit st: the parity of the chunks in stage st whose scores warps 2 and 3 formed so far
            // (p_ready[st]'s phase: a stage's next readout needs the stage refilled, so it cannot
            // run two phases ahead)
            uint32_t jpar = 0;
            for (int n = 0; n < nloc; ++n) {
                if (*abort_flag) break;
                const int st = n % NST;
                bool ok = mbar_wait(&full[st], (n / NST) & 1, kTimeoutNs);
                ok = ok && mbar_wait(s_ready, n & 1, kTimeoutNs);
                if (!ok) {
                    fail(a.status, abort_flag, ERR_MMA);
                    break;
                }
                tc_fence_after();
                const uint64_t so = (uint64_t)((st * L::STAGE) >> 4);
                const uint64_t dV = dV0 + so, dK = dK0 + so, dQ = dQ0 + so, dA = dA0 + so;
                // state: S^T += V^T (K (.) Gamma); both operands MN-major
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tS, dV + kk * (2048 >> 4), dK + kk * (2048 >> 4), id_state, 1);
                mma_commit(s_done);
                if (want_out) {
                    ok = mbar_wait(sb_ready, n & 1, kTimeoutNs);
                    if (ok && n >= 2) ok = mbar_wait(&o_empty[n & 1], ((n >> 1) - 1) & 1, kTimeoutNs);
                    if (ok) ok = mbar_wait(&full_qa[st], (n / NST) & 1, kTimeoutNs);
                    if (!ok) {
                        fail(a.status, abort_flag, ERR_MMA);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tO = tO0 + (n & 1) * 64;
                    // inter: O^T = Sb^T (Q (.) Lambda)^T, A (the bf16 state) from TMEM
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk)
                        mma_ts(tO, tSb + kk * 8, dQ + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), id_inter, kk > 0);
                    mma_commit(sb_free);
                    // intra: O^T += V^T (P (.) M)^T (the second key half leaves it to the first)
                    if (KH != 2) {
                        if (sc_chunk(chunk_of(n))) {
                            // warps 2 and 3's masked scores in the stage's score slot
                            const bool okp = mbar_wait(&p_ready[st], (jpar >> st) & 1, kTimeoutNs);
                            jpar ^= 1u << st;
                            if (!okp) {
                                fail(a.status, abort_flag, ERR_MMA);
                                break;
                            }
                            tc_fence_after();
                        }
#pragma unroll
                        for (int kk = 0; kk < C / 16; ++kk)
                            mma_ss(tO, dV + kk * (2048 >> 4), dA + kk * (32 >> 4), id_intra, 1);
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
    } else if (wg == 1 || wg == 2) {
        // ---------------------------------------------------------- state epilogue (2 groups of 4 warps)
        // Group g owns state columns [g*DK/2, (g+1)*DK/2); the warp's TMEM lane quarter is
        // (warp % 4) and its thread's dv column d.
        regs_inc<Regs<DK, BIL, SC>::epi>();
        const int grp = wg - 1;
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const int d = (warp & 3) * 32 + lane;   // dv column within the tile
        const int cb = grp * HC;                 // first state column of this group
        const int gt = threadIdx.x - 128 - grp * 128;   // thread index within the group
        // S0 is the caller's and no earlier grid of the pass writes it; the segment scan's
        // start states (sequence split) come from the grid ahead. Without a gate and with the
        // scores formed here (SC, not SCAL) no prep runs first: the grid ahead may then be the
        // caller's previous pass, whose S_T can be this S0, so wait for it too.
        if (a.mode != kModeFull || (SC && !SCAL)) grid_dependency_wait();
        {
            // S_in of this thread's column and HC keys: every load in flight at once, then to TMEM
            const float* sin = a.S_in ? a.S_in + bh * a.s_in_bh + seg * a.s_in_seg + dv0 + d : nullptr;
            uint32_t s_in[NB][32];
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    s_in[b][i] = sin ? __float_as_uint(sin[(size_t)(cb + b * 32 + i) * a.dv]) : 0u;
#pragma unroll
            for (int b = 0; b < NB; ++b) tmem_st32(tS + lb + cb + b * 32, s_in[b]);
            tmem_wait_st();
        }
        bool alive = true;
        uint32_t P[HC / 2];   // bf16 pairs of S_[n-1] (this thread's columns), kept until the copy is free
        for (int n = 0; n < nloc && alive; ++n) {
            bool ok = true;
            if (n >= 1) ok = mbar_wait(s_done, (n - 1) & 1, kTimeoutNs);
            if (ok && gated) ok = mbar_wait(&gfull[n % NG], (n / NG) & 1, kTimeoutNs);
            if (!group_all_ok(ok, BAR_EPI, NEPI)) {
                alive = false;
                break;
            }
            tc_fence_after();
            const uint8_t* gs = sm + L::GR_OFF + (n % NG) * L::GSL;
            const float* g = reinterpret_cast<const float*>(gs) + cb;
            float gvd = 1.f;   // gamma'[d] (bilinear gate)
            if constexpr (BIL) gvd = expf(reinterpret_cast<const float*>(gs + L::GB)[d]);
            // part 1: S <- Diag(gamma_n) S_[n-1] (and keep bf16(S_[n-1]) in registers), 32
            // columns per step. The step's gate values are read from shared memory before its
            // tensor-memory load is issued, so their latency hides behind that load's.
#pragma unroll
            for (int c2 = 0; c2 < HC; c2 += 32) {
                float4 gv[8];
                if (gated) {
                    const float4* g4 = reinterpret_cast<const float4*>(g + c2);
#pragma unroll
                    for (int i = 0; i < 8; ++i) gv[i] = g4[i];
                }
                uint32_t r0[32];
                tmem_ld32(tS + lb + cb + c2, r0);
                tmem_wait_ld();
                if constexpr (BIL) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r0[i] = __float_as_uint(__uint_as_float(r0[i]) * gvd);
                }
                if (want_out || sweep) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        P[c2 / 2 + i] = pack_bf16(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                }
                if (gated) {
                    // two columns per packed multiply (each lane rounds as a single fp32 multiply)
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        mul2_inplace(r0[4 * i], r0[4 * i + 1], make_float2(gv[i].x, gv[i].y));
                        mul2_inplace(r0[4 * i + 2], r0[4 * i + 3], make_float2(gv[i].z, gv[i].w));
                    }
                    tmem_st32(tS + lb + cb + c2, r0);
                }
            }
            if (gated) mbar_arrive(&gempty[n % NG]);   // this thread has read its gate slot
            if (gated) tmem_wait_st();
            tc_fence_before();
            mbar_arrive(s_ready);
            if (sweep) {
                // the state entering this chunk's update, once the decay is handed back (off the
                // chunk-to-chunk chain): this thread's row d and HC keys
                if constexpr (DK >= 128) {
                    // staged in the idle Q tiles as boxes of 64 keys x 128 rows (128-byte
                    // swizzle; a Q tile holds DK / 128 boxes, so both stages' tiles take the
                    // DK / 64 boxes), then TMA stores from one thread, once the previous chunk's
                    // stores have read the tiles
                    constexpr int BPS = DK / 128;   // boxes per stage's Q tile
                    static_assert(L::QB == BPS * 16384, "state boxes fill the Q tiles");
                    if (gt == 0 && grp == 0) bulk_wait_read0();
                    named_bar_sync(BAR_EPI, NEPI);
#pragma unroll
                    for (int m = 0; m < HC / 8; ++m) {
                        const int key = cb + 8 * m, box = key >> 6;
                        uint8_t* bb = sm + (box / BPS) * L::STAGE + L::Q_OFF + (box % BPS) * 16384;
                        *reinterpret_cast<uint4*>(bb + d * 128 + ((((key & 63) >> 3) ^ (d & 7)) << 4)) =
                            make_uint4(P[4 * m], P[4 * m + 1], P[4 * m + 2], P[4 * m + 3]);
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(BAR_EPI, NEPI);
                    if (gt == 0 && grp == 0) {
                        const int row0 = (bh * a.nchunks + chunk_of(n)) * a.dv + dv0;
#pragma unroll
                        for (int box = 0; box < DK / 64; ++box)
                            tma_store_2d(&tmO, sm + (box / BPS) * L::STAGE + L::Q_OFF + (box % BPS) * 16384, 64 * box,
                                         row0);
                        bulk_commit();
                    }
                } else {
                    uint4* hp = reinterpret_cast<uint4*>(
                        a.Hst + (((size_t)bh * a.nchunks + chunk_of(n)) * a.dv + dv0 + d) * DK + cb);
#pragma unroll
                    for (int i = 0; i < HC / 8; ++i)
                        hp[i] = make_uint4(P[4 * i], P[4 * i + 1], P[4 * i + 2], P[4 * i + 3]);
                }
                continue;
            }
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
        }
        // The final state is complete once the last state MMA is (before the last inter
        // and intra MMAs): its stores go out while those run.
        if (alive && nloc > 0) {
            const bool ok = mbar_wait(s_done, (nloc - 1) & 1, kTimeoutNs);
            if (group_all_ok(ok, BAR_EPI, NEPI)) {
                tc_fence_after();
                // (with per-segment start states, only the end state of the segment that ends
                // the walk is kept: the last one, or the first for the reverse sweep)
                const bool keep = a.mode == kModeSegState || a.mode == kModeFull ||
                                  (a.mode == kModeSweepRev ? seg == 0 : seg == (int)gridDim.z - 1);
                if (a.S_out && keep) {
                    float* so = a.S_out + bh * a.s_out_bh + seg * a.s_out_seg + dv0 + d;
#pragma unroll 1
                    for (int b = 0; b < NB; ++b) {
                        uint32_t r[32];
                        tmem_ld32(tS + lb + cb + b * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) so[(size_t)(cb + b * 32 + i) * a.dv] = __uint_as_float(r[i]);
                    }
                }
            } else {
                alive = false;
            }
        }
        if (!alive && gt == 0) fail(a.status, abort_flag, ERR_EPI);
        if (sweep && gt == 0 && grp == 0) bulk_wait0();   // the state tiles' stores
    } else if (wg == 3) {
        // ---------------------------------------------------------- output drain (4 warps)
        // Thread (warp % 4, lane) owns dv column d of the tile in all 64 rows of each chunk:
        // O^T TMEM -> registers -> bf16 smem tile -> TMA store, 32 rows at a time.
        regs_dec<Regs<DK, BIL, SC>::drain>();
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const int d = (warp & 3) * 32 + lane;
        const int dt = threadIdx.x - 384;   // thread index within the drain warps
        auto drain = [&](int m) -> bool {
            const int b = m & 1;
            const int c = c_begin + m;
            float lbc_m = 0.f;   // B'_C[d] of chunk m (bilinear gate)
            if constexpr (BIL) lbc_m = a.lbc[((size_t)bh * a.nchunks + c) * a.dv + dv0 + d];
            const bool fq = SCAL && q_fac(c);   // per-head gate: output rows take lambda^(r+1)
            const bool ok = mbar_wait(&o_full[b], (m >> 1) & 1, kTimeoutNs);
            if (!group_all_ok(ok, BAR_DR, NDR)) return false;
            tc_fence_after();
            uint8_t* tile = sm + L::O_OFF + b * L::OB;
            if constexpr (KH != 1) {
                // the store issued from this tile two chunks ago must have read it
                if (dt == 0) bulk_wait_read1();
                named_bar_sync(BAR_DR, NDR);
            }
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float w[32];
                const int orow = c * C + h * 32;   // first row of this half
                if constexpr (BIL) {
                    // log beta of these 32 rows (rows past T add nothing), and an L2 prefetch of
                    // chunk m+2's rows, one 128-byte line per thread
                    const float* lp = a.lb + ((size_t)bh * a.T + orow) * a.dv + dv0 + d;
#pragma unroll
                    for (int t = 0; t < 32; ++t) w[t] = orow + t < a.T ? lp[(size_t)t * a.dv] : 0.f;
                    const int prow = (c + 2) * C + h * 32 + dt / 4;
                    if (c + 2 < c_end && prow < a.T)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.lb + ((size_t)bh * a.T + prow) * a.dv + dv0 +
                                                                     (dt & 3) * 32));
                }
                if constexpr (KH == 2) {
                    // the first key half's fp32 partial of these rows (rows past T: none)
                    const float* pp = a.Opart + ((size_t)bh * a.T + orow) * a.dv + dv0 + d;
#pragma unroll
                    for (int t = 0; t < 32; ++t) w[t] = orow + t < a.T ? pp[(size_t)t * a.dv] : 0.f;
                }
                uint32_t r[32];
                tmem_ld32(tO0 + b * 64 + lb + h * 32, r);
                tmem_wait_ld();
                if (h == 1) {
                    tc_fence_before();
                    mbar_arrive(&o_empty[b]);
                }
                if constexpr (BIL) {
                    // exp(B'_r - B'_C): rows 0-31 from the prefix sum, rows 32-63 from the suffix
                    // sum. Exponents are within [-kVGuard, kVGuard]; the fast exponential's error
                    // there is far below the bf16 rounding of O (the parity tests hold the bf16
                    // tolerance).
                    if (h == 0) {
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
                        r[t] = __float_as_uint(__uint_as_float(r[t]) * __expf((float)(h * 32 + t + 1) * lam_h));
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
                } else {
                    __nv_bfloat16* ob =
                        reinterpret_cast<__nv_bfloat16*>(tile) + (d >> 6) * (C * 64) + h * 32 * 64 + (d & 63);
#pragma unroll
                    for (int t = 0; t < 32; ++t) ob[t * 64] = __float2bfloat16_rn(__uint_as_float(r[t]));
                }
            }
            if constexpr (KH != 1) {
                fence_proxy_async_smem();
                named_bar_sync(BAR_DR, NDR);
                if (dt == 0) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        tma_store_3d(&tmO, tile + h * 32 * 64 * 2, dv0, c * C + h * 32, bh);
                        tma_store_3d(&tmO, tile + C * 64 * 2 + h * 32 * 64 * 2, dv0 + 64, c * C + h * 32, bh);
                    }
                    bulk_commit();
                }
            }
            return true;
        };
        bool alive = true;
        if (want_out)
            for (int m = 0; m < nloc && alive; ++m) alive = drain(m);
        if (!alive && dt == 0) fail(a.status, abort_flag, ERR_DRAIN);
        if (dt == 0) bulk_wait0();
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

template <int DK, bool BIL, bool SCAL, int KH = 0, bool SC = false>
cudaError_t launch_dk(const FwdArgs& a, dim3 grid, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                      const CUtensorMap& A, const CUtensorMap& o, const CUtensorMap& qr, cudaStream_t s) {
    using L = Lay<DK, BIL, SC>;
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_fwd_kernel<DK, BIL, SCAL, KH, SC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    // the setmaxnreg split redistributes the 128 registers per thread the launch provides
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, gla_chunk_fwd_kernel<DK, BIL, SCAL, KH, SC>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != 128) return cudaErrorInvalidConfiguration;
    // Programmatic stream serialization lets the CTAs start (barriers, tensor memory, S0)
    // while the grid ahead finishes; the producer (and, for segment start states, the state
    // epilogue) waits for that grid before reading what it wrote. Not for the bilinear gate
    // (its head flags and column decays are read at once) or the second key half (it reads
    // the first half's partial output).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (!BIL && KH != 2) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gla_chunk_fwd_kernel<DK, BIL, SCAL, KH, SC>, a, q, k, v, A, o, qr);
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
    // the scores: pl.sc without a gate forms every chunk's in the pass (no score tiles; the
    // q map stands in, never read); with the per-head gate, the steep chunks' come from the prep
    const bool sc = pl.sc && mode != kModeSegState;
    if (sc && p.gate == GLA_GATE_NONE) {
        ma = mq;
    } else {
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
        // segment s starts from the workspace's start state s * sub (sub state-pass pieces per
        // segment; one per segment with the sliding window); the last segment's pass ends at S_T
        a.S_in = reinterpret_cast<const float*>(base + pl.off_segin);
        a.s_in_bh = st * pl.segin_n; a.s_in_seg = st * pl.sub;
        if (p.ST) { a.S_out = p.ST; a.s_out_bh = st; a.s_out_seg = 0; }
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
    a.Hst = nullptr;
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
    if (sc) {
        if (!qfac && p.gate != GLA_GATE_NONE) return cudaErrorInvalidValue;
        switch (p.dk) {
        case 64: return qfac ? launch_dk<64, false, true, 0, true>(a, grid, mq, mk, mv, ma, mo, mqr, s)
                             : launch_dk<64, false, false, 0, true>(a, grid, mq, mk, mv, ma, mo, mqr, s);
        case 128: return qfac ? launch_dk<128, false, true, 0, true>(a, grid, mq, mk, mv, ma, mo, mqr, s)
                              : launch_dk<128, false, false, 0, true>(a, grid, mq, mk, mv, ma, mo, mqr, s);
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

cudaError_t launch_state_sweep(const StateSweep& w, int* status, cudaStream_t s)
{
    if (w.dv % DVT != 0 || w.nch <= 0 || !w.Hst) return cudaErrorInvalidValue;
    if ((long long)w.BH * w.nch * w.dv >= (1LL << 31)) return cudaErrorInvalidValue;   // state rows as TMA coordinates
    const uint64_t BH = (uint64_t)w.BH;
    CUtensorMap mk, mv;
    if (!map3(&mk, w.kt, w.dk, (uint64_t)w.kt_rows, BH, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    if (!map3(&mv, w.v, w.dv, w.T, BH, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    if (w.nseg < 1 || (w.nseg > 1 && (w.cps <= 0 || (long long)w.cps * (w.nseg - 1) >= w.nch)))
        return cudaErrorInvalidValue;
    FwdArgs a;
    const long long st = (long long)w.dk * w.dv;
    a.S_in = w.S_in; a.s_in_bh = w.nseg > 1 ? st * w.nseg : st; a.s_in_seg = w.nseg > 1 ? st : 0;
    a.S_out = w.S_out; a.s_out_bh = st; a.s_out_seg = 0;
    a.gam = w.gam;
    a.status = status;
    a.dv = w.dv; a.nchunks = w.nch; a.cps = w.nseg > 1 ? w.cps : w.nch;
    a.mode = w.reverse ? kModeSweepRev : kModeSweep;
    a.gated = w.gam != nullptr;
    a.lbc = nullptr;
    a.lb = nullptr;
    a.skip = nullptr;
    a.T = w.T;
    a.H = 1;
    a.Hst = static_cast<__nv_bfloat16*>(w.Hst);
    const dim3 grid(w.dv / DVT, (unsigned)BH, (unsigned)w.nseg);
    // the states leave through the O map's slot: [BH * nch * dv rows][dk] bf16, boxes of 64 keys
    // x 128 rows (128-byte swizzle); no Q, score or O tile is read in a sweep, the K map stands
    // in for those arguments
    CUtensorMap mh;
    {
        uint64_t dims[2] = {(uint64_t)w.dk, BH * (uint64_t)w.nch * (uint64_t)w.dv};
        uint64_t str[1] = {(uint64_t)w.dk * 2};
        uint32_t box[2] = {64, 128};
        if (!make_tmap(&mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.Hst, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    switch (w.dk) {
    case 64: return launch_dk<64, false, false>(a, grid, mk, mk, mv, mk, mh, mk, s);
    case 128: return launch_dk<128, false, false>(a, grid, mk, mk, mv, mk, mh, mk, s);
    case 256: return launch_dk<256, false, false>(a, grid, mk, mk, mv, mk, mh, mk, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gla
