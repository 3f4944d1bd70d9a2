// gla_bwd_grads: the chunk-parallel part of the backward pass on the
// 5th-generation tensor cores, one work item per (b, h, chunk of C = 64 rows).
//
// With Bc the in-chunk inclusive cumulative log gate, Lambda_t = exp(Bc_t),
// Gamma_t = exp(Bc_end - Bc_t), gamma = exp(Bc_end) (per key), and the prep's
// Qt = Q (.) Lambda, Kt = K (.) Gamma and masked scores A (P_ts for s <= t),
// the chunkwise backward of "Gated Linear Attention Transformers with
// Hardware-Efficient Training" (§4.2; the chunk-level states of §3.3) gives,
// for chunk n with H = S_[n-1] (the state entering it) and D = dL/dS_[n]
// (the gradient of the state leaving it),
//
//   dv   = Kt D + A^T dO
//   dq_t = Lambda_t (.) (H do_t^T + sum_{s<=t} dA_ts k_s / Lambda_s)
//   dk_s = Gamma_s  (.) (D v_s^T  + sum_{t>=s} dA_ts q_t / Gamma_t)
//   dA   = (dO V^T) masked to s <= t
//
// (k_s / Lambda_s = Kt_s / gamma and q_t / Gamma_t = Qt_t / gamma, so the
// intra-chunk sums are products of tiles the prep already wrote, rescaled per
// key, and each gradient shares one accumulator between its inter and intra
// terms.) H and D come from the two state sweeps of the chunk pass (bf16,
// [BH][nch][dv][dk]). The gate gradient's per-token term q (.) dq - k (.) dk
// = gamma (Qg (.) Xq - Kg (.) Xk) (Xq, Xk the two accumulators; plus
// rowsum(dL/dS_T (.) S_T) at the last token) is summed over the chunk's later
// rows into R, with each chunk's total in ctot; the gate tail then adds the
// later chunks' totals.
//
// Every product is a tcgen05 MMA with M = 128 and N = 64 (the chunk's rows),
// the accumulators in tensor memory:
//   dq^T [dk x t] += H dO^T      (per dv block)   and  Kg^T dA^T      (Kg = Kt / gamma)
//   dk^T [dk x s] += D V^T       (per dv block)   and  Qg^T dA        (Qg = Qt / gamma)
//   dv^T [dv x s]  = dO^T A + D^T Kt^T (per dv block of 128)
//   dA   [t x s]  += dO V^T      (per dv block; rows 64-127 of the M = 128 product unused)
// H and D stream through shared memory in units of 128 dv rows x 128 keys; dO
// and V in blocks of 128 columns.
//
// The factors Kt / gamma and Qt / gamma reach exp(-Bc_end) <= 1 / gamma. For a
// key whose chunk decay gamma falls below exp(-60) the factored form could
// overflow, so that key's column of Kg and Qg is zeroed (the MMAs add only
// the inter terms) and its thread adds the intra terms pairwise in fp32 log
// space, exp(Bc_t - Bc_s) with t >= s (the paper's full-precision rule).
//
// Warp roles: 0 TMA producer, 1 MMA issuer (and tensor-memory owner), 4-11
// the epilogue, two warpgroups, per chunk in three phases:
//   1. the dv drains (each warpgroup one of the two dv^T buffers);
//   2. 1 / gamma per key, Kt -> Kg as soon as the last dv product has read Kt,
//      dA -> shared memory (bf16, masked), Qt -> Qg;
//   3. the drain, one key per thread (warpgroup e = key half e). It parks its
//      Kg column in the spare tensor-memory columns and signals the producer,
//      which then refills Kt, A and gamma for the next chunk, and reads Qg from
//      the Qt tile, held until the drain is done.
// Persistent: CTA i takes items i, i + grid, ... Every wait is bounded; on a
// timeout the CTA records an error code and winds down.
#include <cuda_bf16.h>

#include "gla_internal.h"
#include "sm100.cuh"
#include "tma_host.h"

namespace gla {
namespace {

using namespace sm100;

constexpr int C = kChunk;
constexpr int NT = 384;
constexpr int NEPI = 256;               // epilogue threads (warps 4-11)
constexpr int NU = 3;                   // H / D unit slots (32 KB each)
constexpr int NBR = 2;                  // dO / V block slots (32 KB each)
constexpr int BAR_EPI = 1;              // named barrier of the epilogue warps
constexpr uint64_t kTimeoutNs = 2000000000ull;
// exp(-60): a key whose chunk decay gamma is below this takes the pairwise intra rule
constexpr float kSteepGamma = 8.7565108e-27f;
constexpr float kLog2e = 1.44269504088896341f;   // 1 / ln 2

enum { ERR_PRODUCER = 0x501, ERR_MMA = 0x502, ERR_EPI = 0x503 };

// tensor-memory columns
constexpr uint32_t TQ = 0;      // dq^T, 64 columns per key half
constexpr uint32_t TK = 128;    // dk^T
constexpr uint32_t TV = 256;    // dv^T, two buffers of 64
constexpr uint32_t TA = 384;    // dA (lanes 0-63)
constexpr uint32_t TG = 448;    // the drain's Kg columns, 32 per key half (bf16 pairs)

// 8 columns of this warp's 32 lanes from tensor memory (32x32b.x8)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

struct GradArgs {
    const __nv_bfloat16* q;   // raw q, k for the gate term q (.) dq - k (.) dk
    const __nv_bfloat16* k;
    const float* log_g;
    const float* gam;         // [BH][nch][dk] or null (no gate)
    const float* bnd;         // [BH][dk] rowsum(dL/dS_T (.) S_T) or null
    float* gq; float* gk; float* gv;
    // gate terms q (.) dq - k (.) dk (+ the boundary term at T-1), summed over the later rows
    // of the same chunk: R [BH][T][dk], and each chunk's total ctot [BH][nch][dk]; null
    // without a gate gradient
    float* R;
    float* ctot;
    int* status;
    int BH, H, T, dv, nch, gate;
};

template <int DK>
struct GL {
    static constexpr int NKH = DK / 128;                  // key halves (M tiles of dq^T, dk^T)
    static constexpr int KTB = DK / 64 * 8192;            // Kt tile: DK/64 boxes of 64 keys x 64 rows
    static constexpr int KT_OFF = 0;
    static constexpr int A_OFF = KTB;                     // A tile [t][s]
    static constexpr int DA_OFF = A_OFF + 8192;           // dA tile [t][s], bf16, written here
    static constexpr int GM_OFF = DA_OFF + 8192;          // gamma [DK] fp32, then 1 / gamma [DK]
    static constexpr int BLK_OFF = GM_OFF + (DK * 8 + 1023) / 1024 * 1024;
    static constexpr int UNIT_OFF = BLK_OFF + NBR * 32768;
    static constexpr int BAR_OFF = UNIT_OFF + NU * 32768;
    static constexpr int SMEM = BAR_OFF + 512 + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void fail(int* status, volatile int* abort_flag, int code) {
    *abort_flag = 1;
    atomicExch(status, code);
}

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

// log alpha of absolute row t and key `key` of head bh (0 without a gate)
template <int DK>
__device__ __forceinline__ float log_alpha(const GradArgs& a, int bh, int t, int key) {
    switch (a.gate) {
    case GLA_GATE_HEAD_SCALAR: return a.log_g[bh % a.H];
    case GLA_GATE_TOKEN_SCALAR: return a.log_g[(size_t)bh * a.T + t];
    case GLA_GATE_PER_KEY: return a.log_g[((size_t)bh * a.T + t) * DK + key];
    }
    return 0.f;
}

// 16-byte chunk cc (8 keys) of row r of a box of 64 keys x rows, 128-byte swizzle
__device__ __forceinline__ uint32_t swz_off(int r, int cc) { return (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4)); }

__device__ __forceinline__ float bf16_at(const uint8_t* p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// Multiplies the keys of a [64 rows x DK] tile (DK/64 swizzled boxes) by the per-key factors
// f (1 / gamma, or 0 for the keys whose gamma is below kSteepGamma). Thread tid of n.
template <int DK>
__device__ __forceinline__ void scale_keys(uint8_t* tile, const float* f, int tid, int n) {
    for (int idx = tid; idx < DK * 8; idx += n) {
        const int j = idx >> 9, r = (idx >> 3) & 63, cc = idx & 7;
        uint4* p = reinterpret_cast<uint4*>(tile + j * 8192 + swz_off(r, cc));
        uint4 w = *p;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
        const float4 f0 = *reinterpret_cast<const float4*>(f + 64 * j + 8 * cc);
        const float4 f1 = *reinterpret_cast<const float4*>(f + 64 * j + 8 * cc + 4);
        const float fs[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(h[e]);
            h[e] = __floats2bfloat162_rn(x.x * fs[2 * e], x.y * fs[2 * e + 1]);
        }
        *p = w;
    }
}

template <int DK>
__global__ void __launch_bounds__(NT, 1)
gla_bwd_grads_kernel(GradArgs a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH,
                     const __grid_constant__ CUtensorMap tmD)
{
    using L = GL<DK>;
    constexpr int NKH = L::NKH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
    uint64_t* res_full = bar + 0;       // Kt, A, gamma landed
    uint64_t* res_empty = bar + 1;      // the chunk's last MMA done with them (and with dA)
    uint64_t* blk_full = bar + 2;       // [NBR]
    uint64_t* blk_empty = bar + 4;      // [NBR]
    uint64_t* unit_full = bar + 6;      // [NU]
    uint64_t* unit_empty = bar + 9;     // [NU]
    uint64_t* dv_full = bar + 12;       // [2]
    uint64_t* dv_empty = bar + 14;      // [2] (128 arrivals: the warpgroup that drains the buffer)
    uint64_t* da_full = bar + 16;       // every MMA of the chunk's blocks done
    uint64_t* dat_ready = bar + 17;     // dA staged, Kg and Qg rescaled (256 arrivals)
    uint64_t* dqdk_full = bar + 18;
    uint64_t* dk_empty = bar + 19;      // dk^T read out (NKH * 128 arrivals)
    uint64_t* dq_empty = bar + 20;      // dq^T read out (NKH * 128 arrivals)
    uint64_t* mma_fin = bar + 21;
    uint64_t* kt_free = bar + 22;       // the chunk's last product reading Kt done
    uint64_t* p3_done = bar + 23;       // the drain done with the Qg tile (NKH * 128 arrivals)
    uint64_t* kg_read = bar + 24;       // the drain has its Kg columns in registers (NKH * 128 arrivals)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 25);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 26);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int items = a.BH * a.nch;
    const int nblk = a.dv / 128;
    const int u_per = 2 * nblk * NKH + 1;   // units per chunk: D and H per block and key half, then Qt
    const bool gated = a.gam != nullptr;

    if (threadIdx.x == 0) {
        mbar_init(res_full, 1); mbar_init(res_empty, 1);
        for (int i = 0; i < NBR; ++i) { mbar_init(&blk_full[i], 1); mbar_init(&blk_empty[i], 1); }
        for (int i = 0; i < NU; ++i) { mbar_init(&unit_full[i], 1); mbar_init(&unit_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&dv_full[i], 1); mbar_init(&dv_empty[i], 128); }
        mbar_init(da_full, 1); mbar_init(dat_ready, NEPI);
        mbar_init(dqdk_full, 1); mbar_init(dk_empty, NKH * 128); mbar_init(dq_empty, NKH * 128);
        mbar_init(mma_fin, 1); mbar_init(kt_free, 1); mbar_init(p3_done, NKH * 128);
        mbar_init(kg_read, NKH * 128);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&tmK); prefetch_tmap(&tmQ); prefetch_tmap(&tmA); prefetch_tmap(&tmO);
        prefetch_tmap(&tmV); prefetch_tmap(&tmH); prefetch_tmap(&tmD);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int u = 0, bc = 0, i = 0, nres = 0;
            bool ok = true;
            // (a slot that held a chunk's Qt tile is refilled once the drain is done with it too)
            auto slot_free = [&](int x) -> bool {
                if (x < NU) return true;
                const int prev = x - NU;
                if (!mbar_wait(&unit_empty[x % NU], (prev / NU) & 1, kTimeoutNs)) return false;
                return prev % u_per != u_per - 1 || mbar_wait(p3_done, (prev / u_per) & 1, kTimeoutNs);
            };
            auto load_unit = [&](const CUtensorMap* m, int c0, int c1, int c2) -> bool {
                const int us = u % NU;
                if (!slot_free(u)) return false;
                uint8_t* ub = sm + L::UNIT_OFF + us * 32768;
                mbar_arrive_expect_tx(&unit_full[us], 32768);
                tma_load_3d(ub, m, &unit_full[us], c0, c1, c2);
                tma_load_3d(ub + 16384, m, &unit_full[us], c0 + 64, c1, c2);
                ++u;
                return true;
            };
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++i) {
                if (*abort_flag) break;
                const int bh = it / a.nch, c = it % a.nch, hc = bh * a.nch + c;
                for (int b = 0; b < nblk && ok; ++b) {
                    const int slot = bc % NBR;
                    if (bc >= NBR && !mbar_wait(&blk_empty[slot], ((bc / NBR) - 1) & 1, kTimeoutNs)) { ok = false; break; }
                    uint8_t* bb = sm + L::BLK_OFF + slot * 32768;
                    mbar_arrive_expect_tx(&blk_full[slot], 32768);
                    tma_load_3d(bb, &tmO, &blk_full[slot], 128 * b, c * C, bh);
                    tma_load_3d(bb + 8192, &tmO, &blk_full[slot], 128 * b + 64, c * C, bh);
                    tma_load_3d(bb + 16384, &tmV, &blk_full[slot], 128 * b, c * C, bh);
                    tma_load_3d(bb + 24576, &tmV, &blk_full[slot], 128 * b + 64, c * C, bh);
                    ++bc;
                    for (int kh = 0; kh < NKH && ok; ++kh) ok = load_unit(&tmD, 128 * kh, 128 * b, hc);
                    if (ok && b == 0) {
                        // Kt, A and gamma, once the previous chunk's last products are done with
                        // them (the first block's tiles are already on their way)
                        if (i >= 1 && (!mbar_wait(res_empty, (i - 1) & 1, kTimeoutNs) ||
                                       !mbar_wait(kg_read, (i - 1) & 1, kTimeoutNs))) { ok = false; break; }
                        mbar_arrive_expect_tx(res_full, L::KTB + 8192 + (gated ? DK * 4 : 0));
#pragma unroll
                        for (int j = 0; j < DK / 64; ++j)
                            tma_load_3d(sm + L::KT_OFF + j * 8192, &tmK, res_full, 64 * j, c * C, bh);
                        tma_load_2d(sm + L::A_OFF, &tmA, res_full, 0, hc * C);
                        if (gated) bulk_load(sm + L::GM_OFF, a.gam + (size_t)hc * DK, DK * 4, res_full);
                        ++nres;
                        // the rows the drain reads (raw q, k and the per-key log gates) into L2
                        const int nr = min(C, a.T - c * C);
                        const size_t rb = (size_t)bh * a.T + (size_t)c * C;
                        prefetch_l2(a.q + rb * DK, (uint32_t)(nr * DK * 2));
                        prefetch_l2(a.k + rb * DK, (uint32_t)(nr * DK * 2));
                        const float* lg = a.log_g + rb * DK;
                        if (a.gate == GLA_GATE_PER_KEY && (reinterpret_cast<uintptr_t>(lg) & 15) == 0)
                            prefetch_l2(lg, (uint32_t)(nr * DK * 4));
                    }
                    for (int kh = 0; kh < NKH && ok; ++kh) ok = load_unit(&tmH, 128 * kh, 128 * b, hc);
                }
                if (!ok) break;
                // the chunk's Qt rows, for the dk intra product
                const int us = u % NU;
                if (!slot_free(u)) { ok = false; break; }
                uint8_t* ub = sm + L::UNIT_OFF + us * 32768;
                mbar_arrive_expect_tx(&unit_full[us], L::KTB);
#pragma unroll
                for (int j = 0; j < DK / 64; ++j) tma_load_3d(ub + j * 8192, &tmQ, &unit_full[us], 64 * j, c * C, bh);
                ++u;
            }
            if (!ok) fail(a.status, abort_flag, ERR_PRODUCER);
            // no copy may land after the CTA exits: wait for the last fills of every ring
            for (int x = max(0, u - NU); x < u; ++x) mbar_wait(&unit_full[x % NU], (x / NU) & 1, kTimeoutNs);
            for (int x = max(0, bc - NBR); x < bc; ++x) mbar_wait(&blk_full[x % NBR], (x / NBR) & 1, kTimeoutNs);
            if (nres > 0) mbar_wait(res_full, (nres - 1) & 1, kTimeoutNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_dvA = idesc_bf16(128, 64, true, true);     // dO^T (MN) x A (MN)
            constexpr uint32_t id_dvD = idesc_bf16(128, 64, false, false);   // D^T (K) x Kt (K)
            constexpr uint32_t id_mnk = idesc_bf16(128, 64, true, false);    // H, D, Kg^T (MN) x dO, V, dA^T (K)
            constexpr uint32_t id_kk = idesc_bf16(128, 64, false, false);    // dO (K) x V (K)
            constexpr uint32_t id_mnmn = idesc_bf16(128, 64, true, true);    // Qg^T (MN) x dA (MN)
            const uint32_t s0 = smem_u32(sm);
            const uint32_t sKT = s0 + L::KT_OFF, sA = s0 + L::A_OFF, sDA = s0 + L::DA_OFF;
            int u = 0, bc = 0, dvc = 0, i = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++i) {
                if (*abort_flag) { ok = false; break; }
                ok = mbar_wait(res_full, i & 1, kTimeoutNs);
                for (int b = 0; b < nblk && ok; ++b) {
                    const int slot = bc % NBR;
                    ok = mbar_wait(&blk_full[slot], (bc / NBR) & 1, kTimeoutNs);
                    const int buf = dvc & 1;
                    if (ok && dvc >= 2) ok = mbar_wait(&dv_empty[buf], ((dvc >> 1) - 1) & 1, kTimeoutNs);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sB = s0 + L::BLK_OFF + slot * 32768;   // dO: +0, +8192; V: +16384, +24576
                    const uint32_t tDV = tmem + TV + buf * 64;
                    // dv^T = dO^T A: dO^T MN-major (dv contiguous), A as MN-major B (s contiguous)
#pragma unroll
                    for (int kk = 0; kk < C / 16; ++kk)
                        mma_ss(tDV, sdesc(sB + kk * 2048, 8192, 1024, kSwizzle128),
                               sdesc(sA + kk * 2048, 8192, 1024, kSwizzle128), id_dvA, kk > 0);
                    for (int kh = 0; kh < NKH && ok; ++kh) {
                        const int us = u % NU;
                        ok = mbar_wait(&unit_full[us], (u / NU) & 1, kTimeoutNs);
                        if (ok && b == 0 && kh == 0 && i >= 1) ok = mbar_wait(dk_empty, (i - 1) & 1, kTimeoutNs);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t sU = s0 + L::UNIT_OFF + us * 32768;   // D rows 128b.., keys 128kh..
                        // dv^T += D^T Kt^T over these 128 keys: D^T K-major (keys contiguous)
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tDV, sdesc(sU + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128),
                                   sdesc(sKT + (2 * kh + (kk >> 2)) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128),
                                   id_dvD, 1);
                        // dk^T[kh] += D V^T over these 128 dv columns: D MN-major (keys contiguous)
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tmem + TK + kh * 64, sdesc(sU + kk * 2048, 16384, 1024, kSwizzle128),
                                   sdesc(sB + 16384 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128),
                                   id_mnk, (b > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&unit_empty[us]);
                        ++u;
                    }
                    if (!ok) break;
                    mma_commit(&dv_full[buf]);
                    ++dvc;
                    if (b == nblk - 1) mma_commit(kt_free);   // every product reading Kt is issued
                    // dA += dO V^T over these 128 dv columns (rows 64-127 of the product unused)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + TA, sdesc(sB + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128),
                               sdesc(sB + 16384 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128), id_kk,
                               (b > 0 || kk > 0) ? 1u : 0u);
                    for (int kh = 0; kh < NKH && ok; ++kh) {
                        const int us = u % NU;
                        ok = mbar_wait(&unit_full[us], (u / NU) & 1, kTimeoutNs);
                        if (ok && b == 0 && kh == 0 && i >= 1) ok = mbar_wait(dq_empty, (i - 1) & 1, kTimeoutNs);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t sU = s0 + L::UNIT_OFF + us * 32768;   // H rows 128b.., keys 128kh..
                        // dq^T[kh] += H dO^T: H MN-major, dO K-major
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tmem + TQ + kh * 64, sdesc(sU + kk * 2048, 16384, 1024, kSwizzle128),
                                   sdesc(sB + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128), id_mnk,
                                   (b > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&unit_empty[us]);
                        ++u;
                    }
                    if (!ok) break;
                    mma_commit(&blk_empty[slot]);
                    ++bc;
                }
                if (!ok) break;
                mma_commit(da_full);
                // the intra terms, once dA is staged and Kt, Qt are rescaled
                const int us = u % NU;
                ok = mbar_wait(&unit_full[us], (u / NU) & 1, kTimeoutNs);
                if (ok) ok = mbar_wait(dat_ready, i & 1, kTimeoutNs);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sQ = s0 + L::UNIT_OFF + us * 32768;
                for (int kh = 0; kh < NKH; ++kh) {
                    // dq^T[kh] += Kg^T dA^T: Kg^T MN-major, dA^T K-major (s contiguous in a row t)
#pragma unroll
                    for (int kk = 0; kk < C / 16; ++kk)
                        mma_ss(tmem + TQ + kh * 64, sdesc(sKT + 2 * kh * 8192 + kk * 2048, 8192, 1024, kSwizzle128),
                               sdesc(sDA + kk * 32, 16, 1024, kSwizzle128), id_mnk, 1);
                    // dk^T[kh] += Qg^T dA: Qg^T MN-major, dA as MN-major B (s contiguous)
#pragma unroll
                    for (int kk = 0; kk < C / 16; ++kk)
                        mma_ss(tmem + TK + kh * 64, sdesc(sQ + 2 * kh * 8192 + kk * 2048, 8192, 1024, kSwizzle128),
                               sdesc(sDA + kk * 2048, 8192, 1024, kSwizzle128), id_mnmn, 1);
                }
                mma_commit(dqdk_full);
                mma_commit(&unit_empty[us]);
                ++u;
                mma_commit(res_empty);
            }
            if (!ok) fail(a.status, abort_flag, ERR_MMA);
            // one last commit tracks every MMA issued above: none may still run when the
            // tensor memory is freed
            mma_commit(mma_fin);
            mbar_wait(mma_fin, 0, kTimeoutNs);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- epilogue (2 warpgroups)
        const int e = (warp - 4) >> 2;                 // warpgroup
        const int row = (warp & 3) * 32 + lane;        // tensor-memory lane
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const int et = threadIdx.x - 128;              // 0..255
        const float* gm = reinterpret_cast<const float*>(sm + L::GM_OFF);
        int jd = 0;   // dv drains done by this warpgroup
        int i = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x, ++i) {
            const int bh = it / a.nch, c = it % a.nch;
            const int nr = min(C, a.T - c * C);
            const size_t rb = (size_t)bh * a.T + (size_t)c * C;   // first row of the chunk
            bool ok = *abort_flag == 0;
            // this key's log gates over the chunk, loaded at once (rows past T read as 0): the
            // latency overlaps the chunk's products
            const int key = 128 * e + row;
            float Bc[C];
            if (e < NKH) {
                const float* lg = nullptr;
                size_t st = 0;
                if (a.gate == GLA_GATE_PER_KEY) { lg = a.log_g + rb * DK + key; st = DK; }
                else if (a.gate == GLA_GATE_TOKEN_SCALAR) { lg = a.log_g + rb; st = 1; }
                else if (a.gate == GLA_GATE_HEAD_SCALAR) { lg = a.log_g + bh % a.H; st = 0; }
#pragma unroll
                for (int t = 0; t < C; ++t) Bc[t] = (lg && t < nr) ? lg[(size_t)t * st] : 0.f;
            }
            // phase 1: this warpgroup's dv blocks (buffer e), each thread one dv column
            for (int b = 0; b < nblk && ok; ++b) {
                if (((i * nblk + b) & 1) != e) continue;
                ok = __all_sync(0xffffffffu, mbar_wait(&dv_full[e], jd & 1, kTimeoutNs));   // warp-uniform
                ++jd;
                if (!ok) break;
                tc_fence_after();
                float* out = a.gv + rb * a.dv + 128 * b + row;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lb + TV + e * 64 + 32 * h, r);
                    tmem_wait_ld();
                    if (h == 1) {
                        tc_fence_before();
                        mbar_arrive(&dv_empty[e]);
                    }
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (32 * h + t < nr) out[(size_t)(32 * h + t) * a.dv] = __uint_as_float(r[t]);
                }
            }
            // every epilogue thread is past the previous chunk's use of the dA tile
            if (!group_all_ok(ok, BAR_EPI, NEPI)) break;
            // phase 2: the per-key factors 1 / gamma (0 for a steep key), Kt to Kg once the dv
            // products are done with it, dA to shared memory (bf16, masked), Qt to Qg
            float* ginv = reinterpret_cast<float*>(sm + L::GM_OFF) + DK;
            ok = mbar_wait(res_full, i & 1, kTimeoutNs);
            if (ok && gated && et < DK) {
                const float g = gm[et];
                ginv[et] = g >= kSteepGamma ? 1.f / g : 0.f;
            }
            if (!group_all_ok(ok, BAR_EPI, NEPI)) break;
            ok = mbar_wait(kt_free, i & 1, kTimeoutNs);
            if (ok && gated) scale_keys<DK>(sm + L::KT_OFF, ginv, et, NEPI);
            if (ok) ok = mbar_wait(da_full, i & 1, kTimeoutNs);
            ok = __all_sync(0xffffffffu, ok);   // the tensor-memory loads below are warp-wide
            if (ok) {
                tc_fence_after();
                if (e == 0 && row < C) {
                    const int t = row;
                    uint8_t* drow = sm + L::DA_OFF;
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lb + TA + 32 * h, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int g = 0; g < 4; ++g) {   // 16-byte chunk 4h + g: columns 32h + 8g ..
                            uint32_t w[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const int s = 32 * h + 8 * g + 2 * x;
                                const float v0 = (s <= t && t < nr) ? __uint_as_float(r[8 * g + 2 * x]) : 0.f;
                                const float v1 = (s + 1 <= t && t < nr) ? __uint_as_float(r[8 * g + 2 * x + 1]) : 0.f;
                                w[x] = pack_bf16(v0, v1);
                            }
                            *reinterpret_cast<uint4*>(drow + swz_off(t, 4 * h + g)) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
            const int uq = i * u_per + 2 * nblk * NKH;
            const int usq = uq % NU;
            if (ok) ok = mbar_wait(&unit_full[usq], (uq / NU) & 1, kTimeoutNs);
            if (ok && gated) scale_keys<DK>(sm + L::UNIT_OFF + usq * 32768, ginv, et, NEPI);
            const float gk = (gated && e < NKH) ? gm[key] : 1.f;   // read before the slot is reloaded
            fence_proxy_async_smem();
            // every thread's rescale is done before any drain thread reads a Kg or Qg column (the
            // tiles stay until the drain is done with them)
            if (!group_all_ok(ok, BAR_EPI, NEPI)) break;
            const uint8_t* qcol = sm + L::UNIT_OFF + usq * 32768 + (key >> 6) * 8192 + (key & 7) * 2;
            const uint8_t* kcol = sm + L::KT_OFF + (key >> 6) * 8192 + (key & 7) * 2;   // read once, below
            mbar_arrive(dat_ready);
            // phase 3: dq and dk of key `key` (warpgroup e = key half e), rows from the last,
            // with the gate terms summed over the later rows of the chunk
            if (ok && e < NKH) {
                Bc[0] *= kLog2e;
#pragma unroll
                for (int t = 1; t < C; ++t) Bc[t] = fmaf(Bc[t], kLog2e, Bc[t - 1]);   // Bc_t / ln 2; rows past T add 0
                const float tot = Bc[C - 1];                       // Bc_end / ln 2
                ok = __all_sync(0xffffffffu, mbar_wait(dqdk_full, i & 1, kTimeoutNs));
                if (ok) {
                    tc_fence_after();
                    const bool steep = gated && !(gk >= kSteepGamma);
                    float* oq = a.gq + rb * DK + key;
                    float* ok_ = a.gk + rb * DK + key;
                    float* oR = a.R ? a.R + rb * DK + key : nullptr;
                    const __nv_bfloat16* qr = a.q + rb * DK + key;
                    const __nv_bfloat16* kr = a.k + rb * DK + key;
                    const float bnd = (a.bnd && c == a.nch - 1) ? a.bnd[(size_t)bh * DK + key] : 0.f;
                    // rows from the last: dq, dk and the gate term q (.) dq - k (.) dk =
                    // gamma (Qg (.) Xq - Kg (.) Xk) (q Lambda = Qt = gamma Qg, k Gamma = Kt =
                    // gamma Kg), summed over the later rows of the chunk
                    const int cc = (key & 63) >> 3;
                    // this key's Kg column into the spare tensor-memory columns (bf16 pairs, this
                    // thread's lane), so that the next chunk's Kt can land in the tile while the
                    // drain runs
                    {
                        uint32_t kg2[C / 2];
#pragma unroll
                        for (int t = 0; t < C; t += 2) {
                            const uint32_t lo = *reinterpret_cast<const uint16_t*>(kcol + swz_off(t, cc));
                            const uint32_t hi = *reinterpret_cast<const uint16_t*>(kcol + swz_off(t + 1, cc));
                            kg2[t / 2] = lo | (hi << 16);
                        }
                        tmem_st32(tmem + lb + TG + 32 * e, kg2);
                        tmem_wait_st();
                    }
                    mbar_arrive(kg_read);
                    float rsum = 0.f;
#pragma unroll
                    for (int qd = C / 16 - 1; qd >= 0; --qd) {
                        uint32_t xq[16], xk[16], kq[8];
                        tmem_ld16(tmem + lb + TQ + e * 64 + 16 * qd, xq);
                        tmem_ld16(tmem + lb + TK + e * 64 + 16 * qd, xk);
                        tmem_ld8(tmem + lb + TG + 32 * e + 8 * qd, kq);
                        tmem_wait_ld();
                        if (qd == 0) {
                            tc_fence_before();
                            mbar_arrive(dk_empty);
                            mbar_arrive(dq_empty);
                        }
#pragma unroll
                        for (int j = 15; j >= 0; --j) {
                            const int r = 16 * qd + j;
                            if (r < nr) {
                                const float Xq = __uint_as_float(xq[j]), Xk = __uint_as_float(xk[j]);
                                oq[(size_t)r * DK] = exp2f(Bc[r]) * Xq;          // Lambda_r Xq
                                ok_[(size_t)r * DK] = exp2f(tot - Bc[r]) * Xk;   // Gamma_r Xk
                                if (oR) {
                                    const float qg = bf16_at(qcol + swz_off(r, cc));
                                    const uint32_t kp = kq[j >> 1];
                                    const float kg = __uint_as_float(j & 1 ? kp & 0xffff0000u : kp << 16);
                                    rsum += gk * (qg * Xq - kg * Xk);
                                    if (c * C + r == a.T - 1) rsum += bnd;
                                    oR[(size_t)r * DK] = rsum;
                                }
                            }
                        }
                    }
                    mbar_arrive(p3_done);
                    if (steep) {
                        // the intra terms of this key, pairwise: exp(Bc_t - Bc_s) <= 1 for t >= s;
                        // then the gate terms again from the completed dq and dk
                        const uint8_t* dat = sm + L::DA_OFF;
                        float Bs[C];
                        float acc = 0.f;
                        for (int t = 0; t < nr; ++t) {
                            acc += log_alpha<DK>(a, bh, c * C + t, key);
                            Bs[t] = acc;
                        }
                        for (int t = 0; t < nr; ++t) {
                            float sq = 0.f, sk = 0.f;
                            for (int s2 = 0; s2 <= t; ++s2)
                                sq += bf16_at(dat + swz_off(t, s2 >> 3) + (s2 & 7) * 2) *
                                      __bfloat162float(kr[(size_t)s2 * DK]) * expf(Bs[t] - Bs[s2]);
                            for (int u2 = t; u2 < nr; ++u2)
                                sk += bf16_at(dat + swz_off(u2, t >> 3) + (t & 7) * 2) *
                                      __bfloat162float(qr[(size_t)u2 * DK]) * expf(Bs[u2] - Bs[t]);
                            oq[(size_t)t * DK] += sq;
                            ok_[(size_t)t * DK] += sk;
                        }
                        if (oR) {
                            rsum = 0.f;
                            for (int t = nr - 1; t >= 0; --t) {
                                rsum += __bfloat162float(qr[(size_t)t * DK]) * oq[(size_t)t * DK] -
                                        __bfloat162float(kr[(size_t)t * DK]) * ok_[(size_t)t * DK];
                                if (c * C + t == a.T - 1) rsum += bnd;
                                oR[(size_t)t * DK] = rsum;
                            }
                        }
                    }
                    if (a.ctot) a.ctot[((size_t)bh * a.nch + c) * DK + key] = rsum;
                }
            }
            if (!ok) {
                fail(a.status, abort_flag, ERR_EPI);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// rowsum(dL/dS_T (.) S_T) per (b, h, key): one warp per row of dk x dv
__global__ void __launch_bounds__(256) gla_bwd_boundary_kernel(const float* dST, const float* ST, float* bnd, long long rows,
                                                              int dv)
{
    const int lane = threadIdx.x % 32;
    for (long long r = ((long long)blockIdx.x * 256 + threadIdx.x) / 32; r < rows; r += (long long)gridDim.x * 8) {
        const float* x = dST + r * dv;
        const float* y = ST + r * dv;
        float s = 0.f;
        for (int j = lane; j < dv; j += 32) s += x[j] * y[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) bnd[r] = s;
    }
}

// out[bh][t][k] += crev[bh][c(t) + 1][k], c(t) = t / C: the gate terms of the later chunks
// (crev: per chunk, the sum over that chunk and all after it). One float4 of keys per thread.
__global__ void __launch_bounds__(256) gla_bwd_gate_fixup_kernel(float* out, const float* crev, long long BH, int T,
                                                                int dk, int nch)
{
    const int q4 = dk / 4;
    const long long n = BH * T * q4;
    for (long long e = (long long)blockIdx.x * 256 + threadIdx.x; e < n; e += (long long)gridDim.x * 256) {
        const int kq = (int)(e % q4);
        const long long bt = e / q4;
        const int t = (int)(bt % T);
        const long long bh = bt / T;
        const int c = t / C + 1;
        if (c >= nch) continue;
        float4* o = reinterpret_cast<float4*>(out) + e;
        const float4 add = reinterpret_cast<const float4*>(crev)[(bh * nch + c) * q4 + kq];
        float4 v = *o;
        v.x += add.x; v.y += add.y; v.z += add.z; v.w += add.w;
        *o = v;
    }
}

bool map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t rows) {
    uint64_t dims[3] = {d0, d1, d2};
    uint64_t str[2] = {d0 * 2, d0 * d1 * 2};
    uint32_t box[3] = {64, rows, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int DK>
cudaError_t launch_grads_dk(const GradArgs& a, const CUtensorMap* m, int sms, cudaStream_t s)
{
    using L = GL<DK>;
    cudaError_t e = cudaFuncSetAttribute(gla_bwd_grads_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    const int items = a.BH * a.nch;
    const int grid = items < sms ? items : sms;
    gla_bwd_grads_kernel<DK><<<grid, NT, L::SMEM, s>>>(a, m[0], m[1], m[2], m[3], m[4], m[5], m[6]);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_grads(const BwdGrads& g, int* status, cudaStream_t s)
{
    if ((g.dk != 128 && g.dk != 256) || g.dv % 128 != 0 || g.T <= 0) return cudaErrorInvalidValue;
    const uint64_t BH = (uint64_t)g.BH;
    const int nch = (g.T + C - 1) / C;
    CUtensorMap m[7];
    if (!map3(&m[0], g.kt, g.dk, (uint64_t)g.kt_rows, BH, 64) || !map3(&m[1], g.qt, g.dk, (uint64_t)g.kt_rows, BH, 64))
        return cudaErrorInvalidValue;
    {   // A as [BH * nch * 64 rows][64] bf16
        uint64_t dims[2] = {64, BH * (uint64_t)nch * 64};
        uint64_t str[1] = {128};
        uint32_t box[2] = {64, 64};
        if (!make_tmap(&m[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (!map3(&m[3], g.dO, g.dv, g.T, BH, 64) || !map3(&m[4], g.v, g.dv, g.T, BH, 64)) return cudaErrorInvalidValue;
    // H and D: [BH * nch][dv][dk], boxes of 64 keys x 128 dv rows
    if (!map3(&m[5], g.Hst, g.dk, g.dv, BH * nch, 128) || !map3(&m[6], g.Dst, g.dk, g.dv, BH * nch, 128))
        return cudaErrorInvalidValue;
    GradArgs a;
    a.q = static_cast<const __nv_bfloat16*>(g.q);
    a.k = static_cast<const __nv_bfloat16*>(g.k);
    a.log_g = g.log_g;
    a.gam = g.gam;
    a.bnd = g.bnd;
    a.gq = g.gq; a.gk = g.gk; a.gv = g.gv; a.R = g.R; a.ctot = g.ctot;
    a.status = status;
    a.BH = g.BH; a.H = g.H; a.T = g.T; a.dv = g.dv; a.nch = nch; a.gate = g.gate;
    const int sms = g.sms > 0 ? g.sms : 148;
    return g.dk == 128 ? launch_grads_dk<128>(a, m, sms, s) : launch_grads_dk<256>(a, m, sms, s);
}

cudaError_t launch_bwd_gate_fixup(float* out, const float* crev, long long BH, int T, int dk, int sms, cudaStream_t s)
{
    const int nch = (T + C - 1) / C;
    if (nch <= 1 || dk % 4 != 0) return nch <= 1 ? cudaSuccess : cudaErrorInvalidValue;
    const long long n = BH * T * (dk / 4);
    long long blocks = (n + 255) / 256;
    const long long cap = (long long)(sms > 0 ? sms : 148) * 8;
    if (blocks > cap) blocks = cap;
    gla_bwd_gate_fixup_kernel<<<(unsigned)blocks, 256, 0, s>>>(out, crev, BH, T, dk, nch);
    return cudaGetLastError();
}

cudaError_t launch_bwd_boundary(const float* dST, const float* ST, float* bnd, long long rows, int dv, int sms,
                                cudaStream_t s)
{
    if (rows <= 0) return cudaSuccess;
    long long blocks = (rows + 7) / 8;
    const long long cap = (long long)(sms > 0 ? sms : 148) * 8;
    if (blocks > cap) blocks = cap;
    gla_bwd_boundary_kernel<<<(unsigned)blocks, 256, 0, s>>>(dST, ST, bnd, rows, dv);
    return cudaGetLastError();
}

}  // namespace gla
