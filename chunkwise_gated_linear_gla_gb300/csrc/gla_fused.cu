// gla_chunk_fused: the chunkwise GLA forward pass for the per-key gate in one
// kernel, with the gate preparation inside the chunk-serial loop ("Gated Linear
// Attention Transformers with Hardware-Efficient Training", §4.2-4.3; the
// non-materialised FlashLinearAttention loop of §3.3 / Alg. 1: chunk states
// stay on chip and every input is read from HBM once).
//
// One thread-block cluster per (b, h) with one CTA per 128 columns of dv (4
// CTAs for dv = 512, 2 for dv = 256). CTA r owns dv columns [128 r, 128 r + 128)
// of the state and output, and prepares keys [KS r, KS r + KS) (KS = dk / NC)
// of every chunk for the whole cluster. With Bc the in-chunk inclusive
// cumulative log gate and g = Bc at the chunk's last row:
//
//   Qg     = Q (.) exp(Bc - g)        query factor referenced to the chunk end
//   Kt     = K (.) exp(g - Bc)        K (.) Gamma                       (<= |k|)
//   gamma  = exp(g)                   the chunk's decay of each key
//
// Qg Kt^T gives the intra-chunk scores (Qg_tk Kt_sk = q_tk k_sk exp(Bc_tk - Bc_sk),
// §4.1 Eq. 4), and Qg (Diag(gamma) S_[n-1]) the inter-chunk term (§4.2,
// (Q (.) Lambda) S_[n-1]), so the same two tiles serve the state update, the
// output and the scores. The preparing CTA writes its slabs of Qg, Kt and gamma
// into its own stage and bulk-copies them into the other CTAs' copies of it
// (distributed shared memory); no intermediate touches HBM and no partial
// result crosses CTAs. Per chunk n:
//
//   MMA       P^T   = Qg Kt^T                    (scores, into this chunk's O buffer)
//   readout   A     = bf16((P (.) M))            (TMEM -> registers -> smem tile)
//   epilogue  S     <- Diag(gamma_n) S_[n-1];  Sb <- bf16(S)
//   MMA       S^T  += V_n^T Kt_n                 (state, M=128 N=256 K=64)
//   MMA       O^T   = Sb^T Qg_n^T                (inter, N=64 K=256; overwrites P)
//             O^T  += V_n^T A^T                  (intra, N=64 K=64)
//   epilogue  O^T TMEM -> registers -> bf16 smem tile -> TMA store
//
// Qg stays within exp(kScoreGuard) |q| while the key's whole-chunk log decay
// g >= -kScoreGuard. A steeper key ("steep") takes Q (.) exp(Bc) instead and
// the undecayed state in Sb, which keeps the inter term exact; its score terms
// from the product are then off by the factor gamma < exp(-kScoreGuard), and
// the readout adds its exact terms pairwise in fp32 log space (§4.3's
// full-precision rule, applied to that key's column), so the scores are exact
// to rounding for any gate.
//
// Warp roles (16 warps): 0 TMA producer (v tiles, L2 prefetch of the next
// chunks' q, k, log g and v; lane 1 releases stages to the cluster); 1 MMA
// issuer and TMEM owner; 2-3 score MMA and readout
// (TMEM lanes 64-127: the score product places the chunk's 64 query rows in
// rows 64-127 of its M = 128 operand); 4-11 state/output epilogue (two groups
// of four, each owning half of the state's columns and half of each output
// tile); 12-15 gate preparation. Stage reuse is agreed across the cluster:
// once a CTA's MMAs are done with a stage it tells every CTA (cempty), and a
// CTA writes its slabs into the others' copies of that stage only after all of
// them have. Every wait is bounded; on a timeout the CTA records an error code,
// tells the other CTAs of its cluster to stop, and winds down.
#include <cuda_bf16.h>

#include <mutex>

#include "gla_internal.h"
#include "sm100.cuh"
#include "tma_host.h"

namespace gla {
namespace {

using namespace sm100;

constexpr int C = kChunk;
constexpr int DK = 256;
constexpr int DVT = kDvTile;
constexpr int NT = 512;
constexpr int NEPI = 256;   // epilogue threads (warps 4-11)
constexpr int NPREP = 128;  // preparation threads (warps 12-15)
constexpr int NRD = 64;     // score readout threads (warps 2-3)
constexpr int BAR_EPI = 1, BAR_G0 = 2, BAR_PREP = 4, BAR_RD = 5;   // named barriers (0: __syncthreads)
constexpr uint64_t kTimeoutNs = 2000000000ull;                     // 2 s per wait
constexpr float kScoreGuard = 60.f;

enum { ERR_PRODUCER = 0x301, ERR_MMA = 0x302, ERR_EPI = 0x303, ERR_PREP = 0x304, ERR_READ = 0x305 };

// Register budgets per warpgroup: 0 (producer, MMA, readout), 1-2 (epilogue), 3 (preparation).
// The kernel is launched with 512 threads x 128 registers; the budgets add up to no more.
constexpr int kRegCtl = 64, kRegEpi = 168, kRegPrep = 112;
static_assert(128 * kRegCtl + 256 * kRegEpi + 128 * kRegPrep <= NT * 128, "register split");

template <int NC>
struct FL {
    static constexpr int KS = DK / NC;          // keys one CTA prepares
    static constexpr int NSL = KS / 64;         // its 64-key (128-byte) slabs
    static constexpr int NCG = KS / 8;          // 16-byte key groups
    static constexpr int NRG = NPREP / NCG;     // row groups
    static constexpr int RPT = C / NRG;         // rows per prep thread
    // The output staging tile comes first: the score product reads the 8 KB before each Qg
    // slab as the unused rows 0-63 of its M = 128 operand, and that must be shared memory.
    static constexpr int O_OFF = 0, OB = C * DVT * 2;
    static constexpr int QB = DK * C * 2, KB = QB, VB = DVT * C * 2, AB = C * C * 2, GB = DK * 4, FB = DK;
    static constexpr int Q_OFF = 0, K_OFF = QB, V_OFF = QB + KB, G_OFF = V_OFF + VB;
    static constexpr int F_OFF = G_OFF + GB;    // steep-key flags of the chunk (one byte per key)
    // The score tile the intra MMA reads: four 16-column blocks (one per K step), each 64 rows
    // in the no-swizzle K-major layout (8-row x 16-byte core matrices); CTA r computes and
    // sends blocks [BPC r, BPC r + BPC). Three tiles in a ring of their own (chunk n in slot
    // n % 3), so that a stage is free once the inter MMA has read it.
    static constexpr int BPC = 4 / NC;
    static constexpr int NASLOT = 3;
    static constexpr int STAGE = (F_OFF + FB + 1023) / 1024 * 1024;
    static constexpr int S_OFF = O_OFF + OB;    // stage 0; stage 1 follows
    static constexpr int A_RING = S_OFF + 2 * STAGE;           // [3] score tiles
    static constexpr int X_OFF = A_RING + NASLOT * AB;          // per-warp totals of the gate scan [4][KS]
    static constexpr int COL_OFF = X_OFF + 4 * KS * 4;          // readout: one steep key's column
    static constexpr int BAR_OFF = COL_OFF + 2 * 64 * 4;
    static constexpr int SMEM = BAR_OFF + 256 + 1024;
    // bytes the other CTAs send into one stage of this one: their slabs of Qg and Kt, their
    // gammas and steep flags; the v tile comes by TMA
    static constexpr uint32_t PEER_TX = (NC - 1) * (2 * KS * C * 2 + KS * 4 + KS);
    static constexpr uint32_t STAGE_TX = VB + PEER_TX;
    static constexpr uint32_t BLOCK_TX = (NC - 1) * BPC * 2048;   // the other CTAs' score blocks
    static_assert(NC == 2 || NC == 4, "cluster of 2 or 4 dv tiles");
    static_assert(RPT >= 1 && NRG * RPT == C, "row groups");
    static_assert(KS % 16 == 0, "flag slices are whole 16-byte pieces");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct FusedArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const float* log_g;
    const float* S0;
    float* ST;
    int* status;
    int T, dv, nchunks;
};

// Byte offset of (row, col) in a 64-column bf16 slab in the tensor cores'
// K-major 128-byte-swizzle layout (rows of 128 B, 16-byte groups XOR row % 8).
__device__ __forceinline__ int sw128(int row, int col) {
    return row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1));
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
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

// Bounded wait: sleeps in try_wait until the phase completes; gives up early once another
// role (or another CTA of the cluster) has set the abort flag.
__device__ __forceinline__ bool wait_cta(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kTimeoutNs) return false;
    }
}

template <int NC>
__device__ __forceinline__ void fail_all(int* status, volatile int* abort_flag, int code) {
    *abort_flag = 1;
    const uint32_t fa = smem_u32(const_cast<int*>(abort_flag));
#pragma unroll
    for (uint32_t p = 0; p < NC; ++p) asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa(fa, p)), "r"(1) : "memory");
    atomicExch(status, code);
}

template <int NC>
__global__ void __launch_bounds__(NT, 1)
gla_fused_kernel(FusedArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmO)
{
    using L = FL<NC>;
    constexpr int HC = DK / 2;   // state columns per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so that every access
    // through it stays a shared-memory access (an integer round trip would make them generic)
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
    uint64_t* full = bar + 0;       // [2] stage complete: v (TMA) and every CTA's slabs
    uint64_t* empty = bar + 2;      // [2] this CTA's MMAs are done with the stage
    uint64_t* cempty = bar + 4;     // [2] every CTA's MMAs are done with the stage (NC arrivals)
    uint64_t* s_ready = bar + 6;    // state decayed in TMEM (256 arrivals)
    uint64_t* s_done = bar + 7;     // state MMA of the chunk complete
    uint64_t* sb_free = bar + 8;    // inter MMA complete: bf16 state copy reusable
    uint64_t* sb_ready = bar + 9;   // bf16 state copy written (256 arrivals)
    uint64_t* o_full = bar + 10;    // [2] O accumulator complete
    uint64_t* o_empty = bar + 12;   // [2] O accumulator drained (256 arrivals)
    uint64_t* p_full = bar + 14;    // score product (this CTA's column blocks) complete
    uint64_t* a_ready = bar + 15;   // the scores are out of tensor memory (64 arrivals)
    uint64_t* mma_drain = bar + 16; // every MMA the chain's issuer issued has completed
    uint64_t* sc_drain = bar + 17;  // every score MMA has completed
    uint64_t* a_full = bar + 18;    // [3] every CTA's score blocks are in score slot i
    uint64_t* qk_empty = bar + 21;  // [2] this CTA's inter MMA is done with the stage (so are the
                                    //     state and score MMAs, the decay and the readout)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 23);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 24);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y;
    const uint32_t rank = cluster_ctarank();   // == blockIdx.x: this CTA's dv tile and key slice
    const int dv0 = (int)rank * DVT;
    const int nch = a.nchunks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], 2);   // producer (expect_tx) and this CTA's own slabs
            mbar_init(&empty[i], 1);
            mbar_init(&cempty[i], NC);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], NEPI);
            mbar_init(&qk_empty[i], 1);
        }
        for (int i = 0; i < L::NASLOT; ++i) mbar_init(&a_full[i], 1);   // own readout (expect_tx: the others')
        mbar_init(s_ready, NEPI); mbar_init(s_done, 1); mbar_init(sb_free, 1); mbar_init(sb_ready, NEPI);
        mbar_init(p_full, 1); mbar_init(a_ready, NRD);
        mbar_init(mma_drain, 1);
        mbar_init(sc_drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&tmQ); prefetch_tmap(&tmK); prefetch_tmap(&tmG); prefetch_tmap(&tmV); prefetch_tmap(&tmO);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();   // every CTA's barriers exist before any CTA signals another
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS = tmem, tSb = tmem + DK, tO0 = tmem + DK + DK / 2;
    auto stage = [&](int n) { return sm + L::S_OFF + (n & 1) * L::STAGE; };

    if (warp < 4) {
        regs_dec<kRegCtl>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------ TMA producer
            auto prefetch_chunk = [&](int c) {
#pragma unroll
                for (int s = 0; s < L::NSL; ++s) {
                    prefetch_l2_tile_3d(&tmQ, (int)rank * L::KS + 64 * s, c * C, bh);
                    prefetch_l2_tile_3d(&tmK, (int)rank * L::KS + 64 * s, c * C, bh);
                    prefetch_l2_tile_3d(&tmG, (int)rank * L::KS + 64 * s, c * C, bh);
                }
                prefetch_l2_tile_3d(&tmV, dv0, c * C, bh);
                prefetch_l2_tile_3d(&tmV, dv0 + 64, c * C, bh);
            };
            if (nch > 1) prefetch_chunk(1);
            int issued = 0;
            for (int n = 0; n < nch; ++n) {
                if (*abort_flag) break;
                const int st = n & 1;
                // this CTA's intra MMA must be done with the stage's v tile (chunk n - 2)
                if (n >= 2 && !wait_cta(&empty[st], ((n >> 1) - 1) & 1, abort_flag)) {
                    fail_all<NC>(a.status, abort_flag, ERR_PRODUCER);
                    break;
                }
                uint8_t* sb = stage(n);
                mbar_arrive_expect_tx(&full[st], L::STAGE_TX);
                tma_load_3d(sb + L::V_OFF, &tmV, &full[st], dv0, n * C, bh);
                tma_load_3d(sb + L::V_OFF + 8192, &tmV, &full[st], dv0 + 64, n * C, bh);
                if (n + 2 < nch) prefetch_chunk(n + 2);
                issued = n + 1;
            }
            // no copy may land after the CTA exits: wait (bounded) for the last fills
            for (int n = max(0, issued - 2); n < issued; ++n) mbar_wait(&full[n & 1], (n >> 1) & 1, kTimeoutNs / 20);
        } else if (warp == 0 && lane == 1) {
            // ------------------------------------------------------ stage release
            // Once this CTA's inter MMA of chunk n is done (so are its state and score MMAs, the
            // decay and the readout), the stage's Q, K, gammas and flags may be rewritten: tell
            // every CTA of the cluster, whose preparation of chunk n + 2 waits for all of them.
            for (int n = 0; n + 2 < nch; ++n) {
                if (!wait_cta(&qk_empty[n & 1], (n >> 1) & 1, abort_flag)) {
                    fail_all<NC>(a.status, abort_flag, ERR_PRODUCER);
                    break;
                }
#pragma unroll
                for (uint32_t p = 0; p < NC; ++p) mbar_arrive_cluster(mapa(smem_u32(&cempty[n & 1]), p));
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------ MMA issuer
            const uint32_t id_state = idesc_bf16(128, DK, true, true);
            const uint32_t id_k64 = idesc_bf16(128, 64, false, false);   // inter
            const uint32_t id_intra = idesc_bf16(128, 64, true, false);
            for (int n = 0; n < nch; ++n) {
                if (*abort_flag) break;
                const int st = n & 1;
                const uint32_t tO = tO0 + (n & 1) * 64;
                bool ok = wait_cta(&full[st], (n >> 1) & 1, abort_flag);
                const uint32_t sb = smem_u32(stage(n));
                const uint32_t sQ = sb + L::Q_OFF, sK = sb + L::K_OFF, sV = sb + L::V_OFF;
                const uint32_t sA = smem_u32(sm + L::A_RING + (n % L::NASLOT) * L::AB);
                // descriptors: one base per operand, K steps add their byte offset >> 4 to it
                const uint64_t dV = sdesc(sV, 8192, 1024, kSwizzle128), dK = sdesc(sK, 8192, 1024, kSwizzle128);
                const uint64_t dQ = sdesc(sQ, 16, 1024, kSwizzle128), dA = sdesc(sA, 128, 256, kNoSwizzle);
                if (ok) ok = wait_cta(s_ready, n & 1, abort_flag);
                if (!ok) {
                    fail_all<NC>(a.status, abort_flag, ERR_MMA);
                    break;
                }
                tc_fence_after();
                // state: S^T += V^T (K (.) Gamma); both operands MN-major
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk) mma_ss(tS, dV + kk * 128, dK + kk * 128, id_state, 1);
                mma_commit(s_done);
                ok = wait_cta(sb_ready, n & 1, abort_flag);
                if (ok) ok = wait_cta(a_ready, n & 1, abort_flag);   // the scores are out of O
                if (!ok) {
                    fail_all<NC>(a.status, abort_flag, ERR_MMA);
                    break;
                }
                tc_fence_after();
                // inter: O^T = Sb^T Qg^T, A (the bf16 state) from TMEM; overwrites the scores
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk)
                    mma_ts(tO, tSb + kk * 8, dQ + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), id_k64, kk > 0);
                mma_commit(sb_free);
                mma_commit(&qk_empty[st]);
                if (!wait_cta(&a_full[n % L::NASLOT], (n / L::NASLOT) & 1, abort_flag)) {   // every CTA's blocks
                    fail_all<NC>(a.status, abort_flag, ERR_MMA);
                    break;
                }
                tc_fence_after();
                // intra: O^T += V^T (P (.) M)^T, K step kk reading score block kk
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk) mma_ss(tO, dV + kk * 128, dA + kk * 128, id_intra, 1);
                mma_commit(&o_full[n & 1]);
                mma_commit(&empty[st]);
            }
            // tensor memory is freed only after every MMA issued here has completed
            mma_commit(mma_drain);
            mbar_wait(mma_drain, 0, kTimeoutNs);
        } else if (warp >= 2) {
            // ------------------------------------------------------ score readout (warps 2-3)
            // TMEM lanes 64-127 of this chunk's O buffer hold this CTA's score columns for rows
            // 0-63 (lane 64 + r = row r). Masked (s <= r), the steep keys' exact terms added, bf16,
            // written as this CTA's 16-column blocks of the score tile and sent to the others.
            const int r = (warp - 2) * 32 + lane;
            const uint32_t lq = (uint32_t)((warp & 3) * 32) << 16;
            float* colb = reinterpret_cast<float*>(sm + L::COL_OFF);   // [2][64]: B_s, k_s of one key
            bool ok = true;
            for (int n = 0; n < nch && ok; ++n) {
                const int st = n & 1, t0 = n * C, nr = min(C, a.T - t0);
                uint8_t* sb = stage(n);
                ok = wait_cta(&full[st], (n >> 1) & 1, abort_flag);   // the operands and the steep flags
                if (ok && n >= 2) ok = wait_cta(&o_empty[n & 1], ((n >> 1) - 1) & 1, abort_flag);
                if (ok && warp == 2 && lane == 0) {
                    // scores, this CTA's columns: rows 64-127 of D = Qg Kt[s in this CTA's blocks]^T,
                    // issued from this thread so the chain's MMA issuer keeps its own pace. The A
                    // operand starts 64 rows (8 KB) before each Qg slab, so the chunk's rows are rows
                    // 64-127; the B operand starts at key row 16 BPC rank of each Kt slab.
                    tc_fence_after();
                    const uint32_t sQ = smem_u32(sb + L::Q_OFF), sK = smem_u32(sb + L::K_OFF);
                    const uint64_t dQ = sdesc(sQ - 8192, 16, 1024, kSwizzle128);
                    const uint64_t dK = sdesc(sK + rank * L::BPC * 2048, 16, 1024, kSwizzle128);
                    const uint32_t id_score = idesc_bf16(128, 16 * L::BPC, false, false);
                    const uint32_t tOs = tO0 + (n & 1) * 64;
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk) {
                        const uint64_t off = (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                        mma_ss(tOs, dQ + off, dK + off, id_score, kk > 0);
                    }
                    mma_commit(p_full);
                }
                if (ok) ok = wait_cta(p_full, n & 1, abort_flag);
                if (!group_all_ok(ok, BAR_RD, NRD)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t* fw = reinterpret_cast<const uint32_t*>(sb + L::F_OFF);
                const bool any_steep = __any_sync(0xffffffffu, (fw[lane] | fw[lane + 32]) != 0u);
                const uint32_t tO = tO0 + (n & 1) * 64;
                const int slot = n % L::NASLOT;
                uint8_t* blk = sm + L::A_RING + slot * L::AB + (int)rank * L::BPC * 2048;
#pragma unroll 1
                for (int bb = 0; bb < L::BPC; ++bb) {
                    const int s0 = 16 * ((int)rank * L::BPC + bb);   // first key row of this block
                    uint32_t v[16];
                    tmem_ld16(tO + lq + 16 * bb, v);
                    tmem_wait_ld();
                    float x[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(v[i]);
                    if (any_steep) {
                        for (int key = 0; key < DK; ++key) {
                            if (!reinterpret_cast<const uint8_t*>(fw)[key]) continue;   // uniform
                            const size_t cb0 = ((size_t)bh * a.T + t0) * DK + key;
                            // this key's cumulative log gate down the chunk (rows 0-31 in warp 2,
                            // 32-63 in warp 3) and its k column, through shared memory
                            float lg = r < nr ? a.log_g[cb0 + (size_t)r * DK] : 0.f;
#pragma unroll
                            for (int o = 1; o < 32; o <<= 1) {
                                const float y = __shfl_up_sync(0xffffffffu, lg, o);
                                if (lane >= o) lg += y;
                            }
                            colb[r] = lg;
                            colb[64 + r] = r < nr ? __bfloat162float(a.k[cb0 + (size_t)r * DK]) : 0.f;
                            named_bar_sync(BAR_RD, NRD);
                            const float off32 = colb[31];
                            const float br = lg + (r >= 32 ? off32 : 0.f);
                            const float qv = r < nr ? __bfloat162float(a.q[cb0 + (size_t)r * DK]) : 0.f;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int s = s0 + i;
                                const float bs = colb[s] + (s >= 32 ? off32 : 0.f);
                                if (s <= r && r < nr) x[i] += qv * colb[64 + s] * __expf(br - bs);
                            }
                            named_bar_sync(BAR_RD, NRD);
                        }
                    }
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int s = s0 + 2 * i;
                        pk[i] = pack_bf16(s <= r && r < nr ? x[2 * i] : 0.f, s + 1 <= r && r < nr ? x[2 * i + 1] : 0.f);
                    }
                    // row r of the block: two 16-byte core-matrix rows, 128 bytes apart along K
                    uint8_t* rw = blk + bb * 2048 + (r >> 3) * 256 + (r & 7) * 16;
                    *reinterpret_cast<uint4*>(rw) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4*>(rw + 128) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
                tc_fence_before();
                fence_proxy_async_smem();
                mbar_arrive(a_ready);                // the O buffer may be overwritten now
                named_bar_sync(BAR_RD, NRD);         // every row of this CTA's blocks is written
                if (r == 0) {
                    mbar_arrive_expect_tx(&a_full[slot], L::BLOCK_TX);
#pragma unroll
                    for (uint32_t p = 1; p < NC; ++p) {
                        const uint32_t dst = (rank + p) % NC;
                        bulk_s2s(mapa(smem_u32(blk), dst), blk, L::BPC * 2048, mapa(smem_u32(&a_full[slot]), dst));
                    }
                }
            }
            if (warp == 2 && lane == 0) {
                // tensor memory is freed only after every MMA issued here has completed
                mma_commit(sc_drain);
                mbar_wait(sc_drain, 0, kTimeoutNs);
            }
            if (!ok && lane == 0) fail_all<NC>(a.status, abort_flag, ERR_READ);
        }
    } else if (warp < 12) {
        // ---------------------------------------------------------- epilogue warps (2 groups of 4)
        // Group g owns state columns [g*DK/2, (g+1)*DK/2) and output rows [g*32, g*32+32)
        // of every chunk; the warp's TMEM lane quarter is (warp % 4).
        regs_inc<kRegEpi>();
        const int grp = (warp - 4) >> 2;
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const int d = (warp & 3) * 32 + lane;          // dv column within the tile
        const int cb = grp * HC;                        // first state column of this group
        const int gt = threadIdx.x - 128 - grp * 128;   // thread index within the group
        const int bar_grp = BAR_G0 + grp;
        {
            // S_0 (or zero) into tensor memory: dv column d, this group's HC keys
            constexpr int NB = HC / 32;
            uint32_t s_in[NB][32];
            const float* sin = a.S0 ? a.S0 + (size_t)bh * DK * a.dv + dv0 + d : nullptr;
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    s_in[b][i] = sin ? __float_as_uint(sin[(size_t)(cb + b * 32 + i) * a.dv]) : 0u;
#pragma unroll
            for (int b = 0; b < NB; ++b) tmem_st32(tS + lb + cb + b * 32, s_in[b]);
            tmem_wait_st();
        }
        // drain the O accumulator of chunk m: TMEM -> registers -> bf16 smem tile -> TMA store
        auto drain = [&](int m) -> bool {
            const int b = m & 1;
            const bool ok = wait_cta(&o_full[b], (m >> 1) & 1, abort_flag);
            if (!group_all_ok(ok, BAR_EPI, NEPI)) return false;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld32(tO0 + b * 64 + lb + grp * 32, r);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&o_empty[b]);
            // the store issued from this group's rows of the tile last chunk must have read it
            if (gt == 0) bulk_wait_read0();
            named_bar_sync(bar_grp, 128);
            uint8_t* tile = sm + L::O_OFF;
            __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(tile) + (d >> 6) * (C * 64) + grp * 32 * 64 + (d & 63);
#pragma unroll
            for (int t = 0; t < 32; ++t) ob[t * 64] = __float2bfloat16_rn(__uint_as_float(r[t]));
            fence_proxy_async_smem();
            named_bar_sync(bar_grp, 128);
            if (gt == 0) {
                tma_store_3d(&tmO, tile + grp * 32 * 64 * 2, dv0, m * C + grp * 32, bh);
                tma_store_3d(&tmO, tile + C * 64 * 2 + grp * 32 * 64 * 2, dv0 + 64, m * C + grp * 32, bh);
                bulk_commit();
            }
            return true;
        };
        bool alive = true;
        uint32_t P[HC / 2];   // bf16 pairs for the inter MMA's copy (this thread's columns)
        for (int n = 0; n < nch && alive; ++n) {
            const int st = n & 1;
            bool ok = true;
            if (n >= 1) ok = wait_cta(s_done, (n - 1) & 1, abort_flag);
            if (ok) ok = wait_cta(&full[st], (n >> 1) & 1, abort_flag);
            if (!group_all_ok(ok, BAR_EPI, NEPI)) {
                alive = false;
                break;
            }
            tc_fence_after();
            const float4* g4 = reinterpret_cast<const float4*>(stage(n) + L::G_OFF) + cb / 4;
            const uint32_t* fw = reinterpret_cast<const uint32_t*>(stage(n) + L::F_OFF) + cb / 4;
            // any steep key in this group's columns? (uniform over the group's threads)
            uint32_t fany = 0u;
#pragma unroll
            for (int i = 0; i < HC / 4; i += 4) {
                const uint4 f4 = *reinterpret_cast<const uint4*>(fw + i);
                fany |= f4.x | f4.y | f4.z | f4.w;
            }
            // S <- Diag(gamma_n) S_[n-1]; the copy for the inter MMA is the decayed state, except
            // for steep keys, whose query factor carries the whole decay (undecayed copy). 32
            // columns per tensor-memory round trip.
#pragma unroll
            for (int c2 = 0; c2 < HC; c2 += 32) {
                uint32_t r0[32];
                tmem_ld32(tS + lb + cb + c2, r0);
                tmem_wait_ld();
                if (fany == 0u) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 ga = g4[(c2 + i) / 4];
                        const float y0 = __uint_as_float(r0[i]) * ga.x, y1 = __uint_as_float(r0[i + 1]) * ga.y;
                        const float y2 = __uint_as_float(r0[i + 2]) * ga.z, y3 = __uint_as_float(r0[i + 3]) * ga.w;
                        P[c2 / 2 + i / 2] = pack_bf16(y0, y1);
                        P[c2 / 2 + i / 2 + 1] = pack_bf16(y2, y3);
                        r0[i] = __float_as_uint(y0); r0[i + 1] = __float_as_uint(y1);
                        r0[i + 2] = __float_as_uint(y2); r0[i + 3] = __float_as_uint(y3);
                    }
                } else {
                    const float* g = reinterpret_cast<const float*>(g4);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const uint32_t fa = fw[(c2 + i) / 4] >> (8 * ((c2 + i) & 3));
                        const float xa = __uint_as_float(r0[i]), xb = __uint_as_float(r0[i + 1]);
                        const float ya = xa * g[c2 + i], yb = xb * g[c2 + i + 1];
                        P[c2 / 2 + i / 2] = pack_bf16((fa & 1u) ? xa : ya, ((fa >> 8) & 1u) ? xb : yb);
                        r0[i] = __float_as_uint(ya);
                        r0[i + 1] = __float_as_uint(yb);
                    }
                }
                tmem_st32(tS + lb + cb + c2, r0);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(s_ready);
            // the bf16 copy for the inter MMA, once the previous one is consumed
            ok = (n == 0) || wait_cta(sb_free, (n - 1) & 1, abort_flag);
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
            if (n >= 1 && !drain(n - 1)) {
                alive = false;
                break;
            }
        }
        // The final state is complete once the last state MMA is (before the last inter
        // and intra MMAs): its stores go out while those run, then the last O drain.
        if (alive && nch > 0) {
            const bool ok = wait_cta(s_done, (nch - 1) & 1, abort_flag);
            if (group_all_ok(ok, BAR_EPI, NEPI)) {
                tc_fence_after();
                if (a.ST) {
                    // 32 columns at a time (the stores do not wait; fewer live registers)
                    float* so = a.ST + (size_t)bh * DK * a.dv + dv0 + d;
#pragma unroll 1
                    for (int b = 0; b < HC / 32; ++b) {
                        uint32_t s_out[32];
                        tmem_ld32(tS + lb + cb + b * 32, s_out);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) so[(size_t)(cb + b * 32 + i) * a.dv] = __uint_as_float(s_out[i]);
                    }
                }
            } else {
                alive = false;
            }
        }
        if (alive && nch > 0 && !drain(nch - 1)) alive = false;
        if (!alive && gt == 0) fail_all<NC>(a.status, abort_flag, ERR_EPI);
        if (gt == 0) bulk_wait0();
    } else {
        // ---------------------------------------------------------- gate preparation (warps 12-15)
        // Thread (cg, rg) owns keys [8 cg, 8 cg + 8) of this CTA's slice and rows [RPT rg, RPT rg +
        // RPT) of the chunk; a warp holds 32 / NCG consecutive row groups. A chunk's inputs are
        // loaded while the previous chunk is published, so their latency is off the chain.
        regs_dec<kRegPrep>();
        const int pt = threadIdx.x - 384, pw = warp - 12;
        const int cg = pt % L::NCG, rg = pt / L::NCG;
        constexpr int RGW = 32 / L::NCG;                // row groups per warp
        const int slab = cg >> 3, cgs = cg & 7;          // the 64-key slab of those keys, their 16-byte group
        const int kc0 = (int)rank * L::KS;              // first key of this CTA's slice
        float* W = reinterpret_cast<float*>(sm + L::X_OFF);   // [4 warps][KS] scan totals
        float g[L::RPT][8];
        uint4 qr[L::RPT], kr[L::RPT];
        // this thread's log gates, q and k of chunk c: RPT rows x 8 keys (rows past T read as zero)
        auto load_chunk = [&](int c) {
            const int t0 = c * C, nr = min(C, a.T - t0);
#pragma unroll
            for (int r = 0; r < L::RPT; ++r) {
                const int row = rg * L::RPT + r;
                if (row < nr) {
                    // read once: streaming loads, so they do not evict anything from the small L1
                    const size_t e = ((size_t)bh * a.T + t0 + row) * DK + kc0 + 8 * cg;
                    const float4* gp = reinterpret_cast<const float4*>(a.log_g + e);
                    const float4 x0 = __ldcs(gp), x1 = __ldcs(gp + 1);
                    g[r][0] = x0.x; g[r][1] = x0.y; g[r][2] = x0.z; g[r][3] = x0.w;
                    g[r][4] = x1.x; g[r][5] = x1.y; g[r][6] = x1.z; g[r][7] = x1.w;
                    qr[r] = __ldcs(reinterpret_cast<const uint4*>(a.q + e));
                    kr[r] = __ldcs(reinterpret_cast<const uint4*>(a.k + e));
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) g[r][i] = 0.f;
                    qr[r] = make_uint4(0u, 0u, 0u, 0u);
                    kr[r] = qr[r];
                }
            }
        };
        if (nch > 0) load_chunk(0);
        bool ok = true;
        for (int n = 0; n < nch; ++n) {
            const int st = n & 1;
            uint8_t* sb = stage(n);
            // 1. inclusive cumulative log gate down the chunk: my rows serially, the row groups of
            //    my warp by shuffles, the warps before mine through shared memory
#pragma unroll
            for (int r = 1; r < L::RPT; ++r)
#pragma unroll
                for (int i = 0; i < 8; ++i) g[r][i] += g[r - 1][i];
            float off[8], tot[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float x = g[L::RPT - 1][i];   // inclusive scan over this warp's row groups
#pragma unroll
                for (int o = L::NCG; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                off[i] = x - g[L::RPT - 1][i];                               // row groups before mine
                tot[i] = __shfl_sync(0xffffffffu, x, (RGW - 1) * L::NCG + cg);   // the warp's total
            }
            if (!group_all_ok(ok, BAR_PREP, NPREP)) break;   // also: the last chunk's reads of W are done
            if (lane >= (RGW - 1) * L::NCG) {
                float4* ww = reinterpret_cast<float4*>(W + pw * L::KS + 8 * cg);
                ww[0] = make_float4(tot[0], tot[1], tot[2], tot[3]);
                ww[1] = make_float4(tot[4], tot[5], tot[6], tot[7]);
            }
            named_bar_sync(BAR_PREP, NPREP);
#pragma unroll
            for (int i = 0; i < 8; ++i) tot[i] = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float4* wr = reinterpret_cast<const float4*>(W + w * L::KS + 8 * cg);
                const float4 u0 = wr[0], u1 = wr[1];
                const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (w < pw) off[i] += v[i];
                    tot[i] += v[i];
                }
            }
#pragma unroll
            for (int r = 0; r < L::RPT; ++r)
#pragma unroll
                for (int i = 0; i < 8; ++i) g[r][i] += off[i];
            bool steep[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) steep[i] = tot[i] < -kScoreGuard;
            // 2. Qg = Q (.) exp(Bc - g) (steep keys: Q (.) exp(Bc)) and Kt = K (.) exp(g - Bc), packed
            //    to bf16 (fewer registers than the inputs they replace) while the stage is in use
            uint4 Qp[L::RPT], Kp[L::RPT];
#pragma unroll
            for (int r = 0; r < L::RPT; ++r) {
                float qf[8], kf[8], oq[8], ok_[8];
                unpack8(qr[r], qf);
                unpack8(kr[r], kf);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float b = g[r][i];
                    ok_[i] = kf[i] * __expf(tot[i] - b);                          // exp(g - Bc) <= 1
                    oq[i] = qf[i] * __expf(steep[i] ? b : b - tot[i]);             // <= exp(kScoreGuard)
                }
                Qp[r] = pack8(oq);
                Kp[r] = pack8(ok_);
            }
            // 3. every CTA of the cluster must be done with this stage (chunk n - 2)
            bool ready = true;
            if (n >= 2) ready = wait_cta(&cempty[st], ((n >> 1) - 1) & 1, abort_flag);
            if (!group_all_ok(ready, BAR_PREP, NPREP)) {
                ok = false;
                break;
            }
            // 4. my slabs into this CTA's stage
#pragma unroll
            for (int r = 0; r < L::RPT; ++r) {
                const int o = sw128(rg * L::RPT + r, 8 * cgs);
                *reinterpret_cast<uint4*>(sb + L::Q_OFF + ((int)rank * L::NSL + slab) * 8192 + o) = Qp[r];
                *reinterpret_cast<uint4*>(sb + L::K_OFF + ((int)rank * L::NSL + slab) * 8192 + o) = Kp[r];
            }
            if (rg == 0) {
                float4* gw = reinterpret_cast<float4*>(sb + L::G_OFF + (kc0 + 8 * cg) * 4);
                gw[0] = make_float4(__expf(tot[0]), __expf(tot[1]), __expf(tot[2]), __expf(tot[3]));
                gw[1] = make_float4(__expf(tot[4]), __expf(tot[5]), __expf(tot[6]), __expf(tot[7]));
                uint32_t f0 = 0u, f1 = 0u;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    f0 |= (steep[i] ? 1u : 0u) << (8 * i);
                    f1 |= (steep[i + 4] ? 1u : 0u) << (8 * i);
                }
                *reinterpret_cast<uint2*>(sb + L::F_OFF + kc0 + 8 * cg) = make_uint2(f0, f1);
            }
            // 5. the next chunk's inputs, in flight while this one is published
            if (n + 1 < nch) load_chunk(n + 1);
            fence_proxy_async_smem();
            named_bar_sync(BAR_PREP, NPREP);
            if (pt == 0) {
                // the other CTAs released this stage with cluster-scope arrivals: acquire them at
                // cluster scope before writing into their copies (the phase is already complete)
                if (n >= 2) mbar_try_wait_cluster(&cempty[st], ((n >> 1) - 1) & 1);
                mbar_arrive(&full[st]);
                const uint8_t* qs = sb + L::Q_OFF + (int)rank * L::KS * C * 2;
                const uint8_t* ks = sb + L::K_OFF + (int)rank * L::KS * C * 2;
                const uint8_t* gs = sb + L::G_OFF + kc0 * 4;
                const uint8_t* fs = sb + L::F_OFF + kc0;
#pragma unroll
                for (uint32_t p = 1; p < NC; ++p) {
                    const uint32_t dst = (rank + p) % NC;
                    const uint32_t fb = mapa(smem_u32(&full[st]), dst);
                    bulk_s2s(mapa(smem_u32(qs), dst), qs, L::KS * C * 2, fb);
                    bulk_s2s(mapa(smem_u32(ks), dst), ks, L::KS * C * 2, fb);
                    bulk_s2s(mapa(smem_u32(gs), dst), gs, L::KS * 4, fb);
                    bulk_s2s(mapa(smem_u32(fs), dst), fs, L::KS, fb);
                }
            }
        }
        if (!ok && pt == 0) fail_all<NC>(a.status, abort_flag, ERR_PREP);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (*abort_flag) {
        // let copies and stores the other CTAs may still have in flight into this one land
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 1000000ull) {
        }
    }
    cluster_sync();   // no CTA leaves while another may still signal it or write into it
}

bool map_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, CUtensorMapSwizzle swz,
              uint32_t rows) {
    uint64_t dims[3] = {d0, d1, d2};
    uint64_t str[2] = {d0 * 2, d0 * d1 * 2};
    uint32_t box[3] = {64, rows, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box, swz);
}

template <int NC>
cudaError_t launch_nc(const FusedArgs& a, unsigned BH, const CUtensorMap& q, const CUtensorMap& k,
                      const CUtensorMap& g, const CUtensorMap& v, const CUtensorMap& o, cudaStream_t s) {
    using L = FL<NC>;
    cudaError_t e = cudaFuncSetAttribute(gla_fused_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    // setmaxnreg redistributes the registers the block is launched with: 128 per thread
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, gla_fused_kernel<NC>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != 128) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NC, BH, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = NC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gla_fused_kernel<NC>, a, q, k, g, v, o);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Clusters of NC CTAs of this kernel that the current device can hold at once (0 if none).
template <int NC>
int max_clusters() {
    using L = FL<NC>;
    if (cudaFuncSetAttribute(gla_fused_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NC, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = NC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gla_fused_kernel<NC>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

std::mutex g_fused_mu;
int g_fused_clusters[64][2];   // per device: -1 unknown, else clusters of 4 / of 2 it can hold
bool g_fused_init[64];

}  // namespace

bool fused_available(int dv) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lk(g_fused_mu);
    if (!g_fused_init[dev]) {
        g_fused_clusters[dev][0] = max_clusters<4>();
        g_fused_clusters[dev][1] = max_clusters<2>();
        g_fused_init[dev] = true;
    }
    return g_fused_clusters[dev][dv == 512 ? 0 : 1] > 0;
}

bool fused_shape_ok(const gla_fwd_params& p) {
    return p.dtype == GLA_BF16 && p.gate == GLA_GATE_PER_KEY && p.dk == DK && (p.dv == 512 || p.dv == 256) &&
           (long long)p.B * p.H <= 65535 && p.T > 0;
}

cudaError_t launch_fused(const gla_fwd_params& p, int* status, cudaStream_t s) {
    if (!fused_shape_ok(p)) return cudaErrorInvalidValue;
    const uint64_t BH = (uint64_t)p.B * p.H;
    CUtensorMap mq, mk, mg, mv, mo;
    if (!map_bf16(&mq, p.q, p.dk, p.T, BH, CU_TENSOR_MAP_SWIZZLE_128B, 64)) return cudaErrorInvalidValue;
    if (!map_bf16(&mk, p.k, p.dk, p.T, BH, CU_TENSOR_MAP_SWIZZLE_128B, 64)) return cudaErrorInvalidValue;
    if (!map_bf16(&mv, p.v, p.dv, p.T, BH, CU_TENSOR_MAP_SWIZZLE_128B, 64)) return cudaErrorInvalidValue;
    if (!map_bf16(&mo, p.O, p.dv, p.T, BH, CU_TENSOR_MAP_SWIZZLE_NONE, 32)) return cudaErrorInvalidValue;
    {
        // log gates, fp32 [BH][T][dk]: only for L2 prefetches of the next chunks
        uint64_t dims[3] = {(uint64_t)p.dk, (uint64_t)p.T, BH};
        uint64_t str[2] = {(uint64_t)p.dk * 4, (uint64_t)p.dk * p.T * 4};
        uint32_t box[3] = {64, 64, 1};
        if (!make_tmap(&mg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.log_g, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    FusedArgs a;
    a.q = static_cast<const __nv_bfloat16*>(p.q);
    a.k = static_cast<const __nv_bfloat16*>(p.k);
    a.log_g = p.log_g;
    a.S0 = p.S0;
    a.ST = p.ST;
    a.status = status;
    a.T = p.T;
    a.dv = p.dv;
    a.nchunks = (p.T + C - 1) / C;
    return p.dv == 512 ? launch_nc<4>(a, (unsigned)BH, mq, mk, mg, mv, mo, s)
                       : launch_nc<2>(a, (unsigned)BH, mq, mk, mg, mv, mo, s);
}

}  // namespace gla
