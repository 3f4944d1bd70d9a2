// gla_chunk_prep: the per-chunk, dv-independent part of the chunkwise GLA
// forward pass ("Gated Linear Attention Transformers with Hardware-Efficient
// Training", §4.2-4.3). One work item per (b, h, chunk of C = 64 rows):
//
//   Bc     in-chunk inclusive cumulative log gate (fp32, on chip only)
//   Qt     = Q (.) Lambda,  Lambda_r = exp(Bc_r)            -> workspace, bf16
//   Kt     = K (.) Gamma,   Gamma_r  = exp(Bc_end - Bc_r)   -> workspace, bf16
//   gamma  = exp(Bc_end)                                    -> workspace, fp32
//   A      = (P (.) M), P_rs = sum_k Q_rk K_sk exp(Bc_rk - Bc_sk), r >= s
//                                                            -> workspace, bf16
//
// The intra-chunk scores take one of two forms, chosen per chunk.
//
// Chunk reference (§4.2 with the normaliser at the middle of the chunk). With
// R_k = Bc at row 31 of key k, P = (Q (.) exp(Bc - R)) (K (.) exp(R - Bc))^T,
// one 64 x 64 x dk product on the 5th-generation tensor cores (tcgen05, the
// accumulator in tensor memory). Every factor is exp of a log-gate difference
// within half a chunk; the form is used when all of them lie within
// exp(+-kRefGuard), so nothing overflows and each product is exact to
// rounding. Entries above the diagonal (r < s) are discarded by the mask.
//
// Secondary chunking (§4.3), for chunks with a steeper gate, with sub-chunks
// of c = 16 rows. For a query sub-chunk j and an earlier key sub-chunk u
// (j > u) the factors are referenced to the first row of j (f_j) and the
// last row of u (l_u):
//     P_ju = (Q_j (.) exp(Bc - f_j)) Diag(exp(f_j - l_u)) (K_u (.) exp(l_u - Bc))^T,
// where every exponent is <= 0, so nothing overflows however steep the gate
// (the paper's P_[i][j] with Lambda, Gamma and b_iC / b_(j+1)C). These run on
// the tensor cores (mma.sync, bf16 in, fp32 accumulate). A diagonal block
// (j = u) needs exp(Bc_r - Bc_s) for r >= s inside one sub-chunk; the same
// factors give it with a per-key scale exp(f_j - l_j) >= 1. While that scale
// stays below exp(kGuard) the product cannot overflow and is exact to
// rounding. A key column whose log gate falls by more than kGuard inside one
// sub-chunk is taken out of the MMA and added pairwise in fp32 log space
// instead (Eq. 4), which is the paper's full-precision intra-sub-chunk rule,
// applied only where it is needed.
//
// Thread layout of the element-wise phase: thread t owns 8 consecutive key
// columns (one 16-byte vector of bf16) and RPT = dk/32 consecutive rows. The
// cumulative gate is a two-level scan: a serial sum over the thread's rows,
// then the totals of the row groups above it. The q and k rows of the chunk
// arrive by TMA in the 128-byte-swizzled K-major layout the tensor cores read
// (rows past the end of the sequence zero-filled), and each thread scales its
// own 16-byte chunks in place.
#include <cuda_bf16.h>

#include "gla_internal.h"
#include "sm100.cuh"
#include "tma_host.h"

namespace gla {
namespace {

using namespace sm100;

constexpr int C = kChunk;
constexpr int SC = 16;                          // sub-chunk rows
constexpr int NSUB = C / SC;                    // 4
constexpr int NPAIR = NSUB * (NSUB + 1) / 2;    // 10 lower (j >= u) blocks
constexpr int NTRI = SC * (SC + 1) / 2;         // 136 pairs r >= s in a block
constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int ALD = C + 8;                      // bf16 row stride of the staged A tile
constexpr int kRefRow = 31;                     // row of the chunk reference
constexpr int kTmemCols = 64;                   // the 64 x 64 fp32 score accumulator (lanes 0-63)
constexpr float kGuard = 60.f;
constexpr float kRefGuard = 60.f;

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
    int qfac;   // per-head scalar gate: chunks that pass q_factored leave Lambda to the chunk pass
    int sc;     // with qfac: those chunks' scores are formed by the chunk pass too (only K (.) Gamma here)
    // read first by the next stages (see prefetch_next_stage): S0, and v by heads
    const uint8_t* pf_s0;   size_t pf_s0_bytes;
    const uint8_t* pf_v;    size_t pf_v_stride;   uint32_t pf_v_bytes;
};

// After its last item a CTA pulls into L2 what the stages after this one read
// first: the initial state S0 (read before the first chunk can be decayed) and
// the first two chunks of v of every head. The stages then start from L2
// instead of competing for DRAM at once. The work goes to the CTAs that have
// one item fewer than the others, which finish first, one bulk prefetch per
// piece from one thread each.
__device__ __forceinline__ void prefetch_next_stage(const PrepArgs& a, int total)
{
    const int extra = total % (int)gridDim.x;   // CTAs [0, extra) run one more item
    const int lo = extra, n = extra ? (int)gridDim.x - extra : (int)gridDim.x;
    if (threadIdx.x != 0 || (int)blockIdx.x < lo) return;
    const int me = (int)blockIdx.x - lo;
    constexpr size_t kPiece = 64 * 1024;
    if (a.pf_s0) {
        const size_t per = ((a.pf_s0_bytes + n - 1) / n + 15) / 16 * 16;
        for (size_t off = (size_t)me * per, end = min(a.pf_s0_bytes, off + per); off < end; off += kPiece)
            prefetch_l2(a.pf_s0 + off, (uint32_t)min(kPiece, end - off));
    }
    if (a.pf_v)
        for (int bh = me; bh < a.BH; bh += n) prefetch_l2(a.pf_v + (size_t)bh * a.pf_v_stride, a.pf_v_bytes);
}

constexpr uint64_t kTimeoutNs = 2000000000ull;   // bounded waits: bulk copies, score MMA
constexpr int ERR_PREP = 0x201;

template <int DK>
struct PL {
    static constexpr int NCG = DK / 8;          // column groups of 8
    static constexpr int NRG = NT / NCG;        // row groups
    static constexpr int RPT = C / NRG;         // rows per thread (dk / 32)
    static constexpr int QS_OFF = 0;                              // [C][DK] bf16 q tile (raw, then swizzled)
    static constexpr int KS_OFF = QS_OFF + C * DK * 2;            // [C][DK] bf16 k tile
    static constexpr int W_OFF = KS_OFF + C * DK * 2;             // [NPAIR][DK] fp32
    static constexpr int X_OFF = W_OFF + NPAIR * DK * 4;          // [2][NRG][DK] fp32 (totals, then first/last)
    static constexpr int CORR_OFF = X_OFF + 2 * NRG * DK * 4;     // [NSUB][NTRI] fp32
    static constexpr int STEEP_OFF = CORR_OFF + NSUB * NTRI * 4;  // [NSUB][DK] u8
    static constexpr int ANY_OFF = STEEP_OFF + NSUB * DK;         // [NSUB] int
    static constexpr int BAR_OFF = (ANY_OFF + 16 + 7) / 8 * 8;    // mbarriers: bulk copies, score MMA
    static constexpr int TM_OFF = BAR_OFF + 16;                   // tensor-memory address
    static constexpr int SMEM = TM_OFF + 16 + 1024;               // + alignment of the tiles to 1024 B
    static_assert(RPT >= 1 && SC % RPT == 0, "a thread's rows lie in one sub-chunk");
    static_assert(kRefRow % RPT == RPT - 1, "the reference row ends a row group");
    static_assert(DK / 8 >= 8, "a 16-byte column group per thread, eight per 128-byte row");
    static_assert(C * ALD * 2 <= 2 * C * DK * 2, "A staging fits in the Q/K tiles");
};

// Element offset of (row, col) in a [C][DK] bf16 tile in the tensor cores'
// K-major 128-byte-swizzle layout: slabs of 64 columns, each 64 rows x 128 B,
// the 16-byte chunks of a row XOR-permuted by (row % 8). The 8 rows of an
// mma.sync fragment load therefore hit 8 different bank groups too.
template <int DK>
__device__ __forceinline__ int opi(int row, int col) {
    return (col >> 6) * (C * 64) + row * 64 + ((((col & 63) >> 3) ^ (row & 7)) << 3) + (col & 7);
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

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Scores on the tensor cores: D[r][s] = sum_k Qs[r][k] Ks[s][k] for the 64 rows of
// the chunk, D in tensor memory lanes 0-63 (an M = 128 product whose rows 64-127,
// read from the memory after the q tile, are discarded). One elected thread.
template <int DK>
__device__ __forceinline__ void score_mma(const uint8_t* Qs, const uint8_t* Ks, uint32_t tmem, uint64_t* bar) {
    const uint32_t id = idesc_bf16(128, 64, false, false);
    const uint64_t dQ = sdesc(smem_u32(Qs), 16, 1024, kSwizzle128);
    const uint64_t dK = sdesc(smem_u32(Ks), 16, 1024, kSwizzle128);
#pragma unroll
    for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * (C * 128) + (kk & 3) * 32) >> 4;
        mma_ss(tmem, dQ + off, dK + off, id, kk > 0);
    }
    mma_commit(bar);
}

// Warps 0 and 1 (tensor-memory lanes 0-63 = rows of the chunk): scores to the
// masked bf16 rows of A, staged in `stage` (64 x 64, 128-byte swizzle, free once
// the MMA is done) and written by one TMA store from thread 0, which also waits
// for that store to read the stage before the stage is reused. With free_bar >= 0
// the stage is written only after the named barrier free_bar (free_n threads)
// says its other readers are done.
// lam: log of the per-head decay (scores scaled by lambda^(r-s)), 0 otherwise.
// TOK (per-token scalar gate): Lc is the chunk's inclusive cumulative log gate in
// shared memory; the scores are then scaled by exp(Lc[r] - Lc[s]) and lam is unused.
// With `fq` (a per-head scalar gate whose chunk passes q_factored) the query
// row's factor lambda^(r+1) is left out: the scores are (q_r . k_s) lambda^-(s+1),
// and the chunk pass multiplies output row r by lambda^(r+1).
template <bool TOK = false>
__device__ __forceinline__ bool score_readout(uint32_t tmem, uint64_t* bar, uint32_t phase, int nr, float lam,
                                              __nv_bfloat16* stage, const CUtensorMap* tmA, int arow,
                                              int free_bar = -1, int free_n = 0, const float* Lc = nullptr,
                                              bool fq = false) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool ok = mbar_wait(bar, phase, kTimeoutNs);
    tc_fence_after();
    const int r = warp * 32 + lane;
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    uint4* dst = reinterpret_cast<uint4*>(stage + r * 64);
    uint32_t p[2][16];
    const float lr = TOK ? Lc[r] : 0.f;
    const int rr = fq ? -1 : r;   // the per-head gate's exponent (rr - s) lam
#pragma unroll
    for (int h = 0; h < 2; ++h) {   // columns 32h .. 32h + 31, one half at a time
        uint32_t v[32];
        tmem_ld32(tmem + lb + 32 * h, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float x[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int s = 32 * h + 2 * i + e;
                const bool keep = s <= r && r < nr;   // the decay only where s <= r: it is <= 1 there
                if (TOK)
                    x[e] = keep ? __uint_as_float(v[2 * i + e]) * __expf(lr - Lc[s]) : 0.f;
                else
                    x[e] = keep ? __uint_as_float(v[2 * i + e]) * (lam != 0.f ? __expf((rr - s) * lam) : 1.f) : 0.f;
            }
            p[h][i] = pack_bf16(x[0], x[1]);
        }
    }
    if (free_bar >= 0) named_bar_sync(free_bar, free_n);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i)   // 16-byte chunk 4h + i of row r, XOR-swizzled by (r % 8)
            dst[(4 * h + i) ^ (r & 7)] = make_uint4(p[h][4 * i], p[h][4 * i + 1], p[h][4 * i + 2], p[h][4 * i + 3]);
    tc_fence_before();
    fence_proxy_async_smem();
    named_bar_sync(1, 64);
    if (threadIdx.x == 0) {
        tma_store_2d(tmA, stage, 0, arow);
        bulk_commit();
    }
    return ok;
}

// Resident CTAs per SM: the kernel is latency-bound, so smaller heads run three
// CTAs per SM (shared memory allows it; registers are bounded to fit).
template <int DK>
constexpr int prep_ctas_per_sm() { return DK <= 128 ? 3 : DK <= 256 ? 2 : 1; }

template <int DK>
__global__ void __launch_bounds__(NT, prep_ctas_per_sm<DK>())
gla_chunk_prep_kernel(PrepArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmA)
{
    // the chunk pass may start (its set-up, its S0 loads) while this grid's last items run;
    // it waits for this grid's writes before it reads them
    launch_dependents();
    using L = PL<DK>;
    constexpr int RPT = L::RPT, NRG = L::NRG;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = align1k(smem_raw);
    // Qs/Ks first receive the q/k rows of the chunk (TMA, swizzled), then are
    // scaled in place for the chunk's score form.
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem + L::QS_OFF);
    __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem + L::KS_OFF);
    uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);     // bulk copies
    uint64_t* mbar = cbar + 1;                                             // score MMA
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::TM_OFF);
    float* W = reinterpret_cast<float*>(smem + L::W_OFF);                     // [NPAIR][DK] exp(f_j - l_u)
    float* X = reinterpret_cast<float*>(smem + L::X_OFF);
    float* corr = reinterpret_cast<float*>(smem + L::CORR_OFF);               // [NSUB][NTRI]
    uint8_t* steep = smem + L::STEEP_OFF;                                     // [NSUB][DK]
    int* steep_any = reinterpret_cast<int*>(smem + L::ANY_OFF);
    __nv_bfloat16* As = Qs;                                                   // [C][ALD], after the MMAs

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        mbar_init(cbar, 1);
        mbar_init(mbar, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // Persistent: work items (b*H+h, chunk) in order, strided by the grid. While
    // one item is computed, the next one's rows are prefetched into L2.
    const int total = a.BH * a.nchunks;
    uint32_t mphase = 0;
    for (int item = blockIdx.x, it = 0; item < total; item += gridDim.x, ++it) {
    const int c = item % a.nchunks, bh = item / a.nchunks;
    const int t0 = c * C;
    const int nr = min(C, a.T - t0);
    const int cg = tid % L::NCG, rg = tid / L::NCG;
    const int col0 = cg * 8, row0 = rg * RPT;
    const int j = row0 / SC;   // the sub-chunk this thread's rows lie in

    if (tid < NSUB) steep_any[tid] = 0;
    for (int i = tid; i < NSUB * DK; i += NT) steep[i] = 0;
    if (tid == 0) {
        bulk_wait_read0();   // the previous item's A store has read its stage (the q tile)
        // every box is full-size: rows at or past T arrive as zeros
        mbar_arrive_expect_tx(cbar, 2 * C * DK * 2);
#pragma unroll
        for (int i = 0; i < DK / 64; ++i) {
            tma_load_3d(Qs + i * C * 64, &tmq, cbar, i * 64, t0, bh);
            tma_load_3d(Ks + i * C * 64, &tmk, cbar, i * 64, t0, bh);
        }
        // the next item's log gates (read by plain loads) into L2; its q and k tiles come by TMA
        const int nx = item + gridDim.x;
        if (nx < total) {
            const int c2 = nx % a.nchunks, bh2 = nx / a.nchunks, nr2 = min(C, a.T - c2 * C);
            const size_t row = (size_t)bh2 * a.T + (size_t)c2 * C;
            prefetch_l2(a.log_g + row * DK, (uint32_t)nr2 * DK * 4);
        }
    }

    // ---- 1. log gates of my rows and their running sum
    float Bc[RPT][8];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
        if (row0 + r < nr) {
            const float4* g = reinterpret_cast<const float4*>(a.log_g + ((size_t)bh * a.T + t0 + row0 + r) * DK + col0);
            x0 = __ldg(g);
            x1 = __ldg(g + 1);
        }
        Bc[r][0] = x0.x; Bc[r][1] = x0.y; Bc[r][2] = x0.z; Bc[r][3] = x0.w;
        Bc[r][4] = x1.x; Bc[r][5] = x1.y; Bc[r][6] = x1.z; Bc[r][7] = x1.w;
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

    // ---- 2. the chunk's score form, then the scaled operands, Q (.) Lambda and K (.) Gamma
    // Chunk reference R = Bc at row kRefRow: usable when, for every key, the largest
    // factors exp(Bc_0 - R) (rows above it) and exp(R - Bc_63) (rows below) stay bounded.
    bool steep_ref = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float R = last[(kRefRow / RPT) * DK + col0 + i];
        steep_ref |= (first[col0 + i] - R) > kRefGuard || (R - last[(NRG - 1) * DK + col0 + i]) > kRefGuard;
    }
    const bool use_ref = !__syncthreads_or(steep_ref);
    // the references of this thread's rows: the query side's (f) and the key side's (l)
    const float* fsrc = use_ref ? last + (kRefRow / RPT) * DK : first + (j * SC / RPT) * DK;
    const float* lsrc = use_ref ? last + (kRefRow / RPT) * DK : last + ((j * SC + SC - 1) / RPT) * DK;
    if (!use_ref && row0 == j * SC) {
        bool any = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool s = (fsrc[col0 + i] - lsrc[col0 + i]) > kGuard;
            steep[j * DK + col0 + i] = s ? 1 : 0;
            any |= s;
        }
        if (any) atomicOr(&steep_any[j], 1);
    }
    {
        const bool ok = mbar_wait(cbar, it & 1, kTimeoutNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicExch(a.status, ERR_PREP);
            break;
        }
    }
    // q rows, then k rows, scaled in place (each thread its own 16-byte chunks)
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        __nv_bfloat16* T = pass == 0 ? Qs : Ks;
        __nv_bfloat16* out = pass == 0 ? a.Qt : a.Kt;
        float ref[8], e[8];   // the reference of this tensor per key, and its output factor
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ref[i] = pass == 0 ? fsrc[col0 + i] : lsrc[col0 + i];
            e[i] = pass == 0 ? __expf(ref[i]) : __expf(last[(NRG - 1) * DK + col0 + i] - ref[i]);
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = row0 + r;
            uint4* slot = reinterpret_cast<uint4*>(T + opi<DK>(row, col0));
            float v[8];
            unpack8(*slot, v);
#pragma unroll
            for (int i = 0; i < 8; ++i)   // factors <= 1 on the sub-chunk form; within exp(+-kRefGuard) on the chunk form
                v[i] *= pass == 0 ? __expf(Bc[r][i] - ref[i]) : __expf(ref[i] - Bc[r][i]);
            *slot = pack8(v);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= e[i];
            *reinterpret_cast<uint4*>(out + ((size_t)bh * a.Tpad + t0 + row) * DK + col0) = pack8(v);
        }
    }
    for (int col = tid; col < DK; col += NT)
        a.gam[((size_t)bh * a.nchunks + c) * DK + col] = __expf(last[(NRG - 1) * DK + col]);
    __nv_bfloat16* Ao = a.A + ((size_t)bh * a.nchunks + c) * C * C;

    if (use_ref) {
        // ---- 3. scores on the tensor cores, one product for the whole chunk
        fence_proxy_async_smem();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            if (lane == 0) score_mma<DK>(reinterpret_cast<uint8_t*>(Qs), reinterpret_cast<uint8_t*>(Ks), tmem, mbar);
            __syncwarp();
        }
        bool ok = true;
        if (warp < 2) ok = score_readout(tmem, mbar, mphase, nr, 0.f, Qs, &tmA, (bh * a.nchunks + c) * C);
        mphase ^= 1u;
        if (__syncthreads_or(!ok)) {   // also: the tiles and the accumulator are reused by the next item
            if (tid == 0) atomicExch(a.status, ERR_PREP);
            break;
        }
        continue;
    }

    // ---- 3'. sub-chunk form: per-pair key factors and exact log-space scores for steep key columns
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
    __syncthreads();
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
                    for (int i = S + 1; i <= R; ++i) lg += a.log_g[((size_t)bh * a.T + t0 + i) * DK + col];
                    const float qv = __bfloat162float(a.q[((size_t)bh * a.T + t0 + R) * DK + col]);
                    const float kv = __bfloat162float(a.k[((size_t)bh * a.T + t0 + S) * DK + col]);
                    acc += qv * kv * __expf(lg);
                }
            }
            corr[jj * NTRI + p] = acc;
        }
    }

    // ---- 4'. lower blocks of A on the tensor cores (mma.sync)
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
            const uint32_t a0 = *reinterpret_cast<const uint32_t*>(Qs + opi<DK>(ra, k0 + 2 * c4));
            const uint32_t a1 = *reinterpret_cast<const uint32_t*>(Qs + opi<DK>(ra + 8, k0 + 2 * c4));
            const uint32_t a2 = *reinterpret_cast<const uint32_t*>(Qs + opi<DK>(ra, k0 + 8 + 2 * c4));
            const uint32_t a3 = *reinterpret_cast<const uint32_t*>(Qs + opi<DK>(ra + 8, k0 + 8 + 2 * c4));
            const float2 w01 = *reinterpret_cast<const float2*>(w + k0 + 2 * c4);
            const float2 w89 = *reinterpret_cast<const float2*>(w + k0 + 2 * c4 + 8);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int rb = ub * SC + nt * 8 + g8;
                uint32_t b0 = *reinterpret_cast<const uint32_t*>(Ks + opi<DK>(rb, k0 + 2 * c4));
                uint32_t b1 = *reinterpret_cast<const uint32_t*>(Ks + opi<DK>(rb, k0 + 8 + 2 * c4));
                b0 = scale_bf16x2(b0, w01.x, w01.y);
                b1 = scale_bf16x2(b1, w89.x, w89.y);
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
    for (int idx = tid; idx < C * C / 8; idx += NT) {
        const int r = idx / (C / 8), s = (idx % (C / 8)) * 8;
        *reinterpret_cast<uint4*>(Ao + r * C + s) = *reinterpret_cast<const uint4*>(As + r * ALD + s);
    }
    __syncthreads();   // shared tiles are refilled by the next item
    }
    prefetch_next_stage(a, total);
    if (tid == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Uniform gates (none, or one fixed decay lambda per head): the cumulative log
// gate of row r in a chunk is (r+1) log(lambda) for every key, so Lambda, Gamma
// and gamma are per-row scalars and the intra-chunk scores have the closed
// form P_rs = (q_r . k_s) lambda^(r-s), r >= s (the decay mask M_ij =
// lambda^(i-j) of "Lightning Attention-2", §3.2.1 Alg. 1). The per-token scalar
// gate (G_t = gamma_t 1^T 1, Table 1 of the GLA paper, §4.1) has the same
// structure with a data-dependent decay: with B_r the chunk's inclusive cumulative
// log gate, P_rs = (q_r . k_s) exp(B_r - B_s), Q rows scale by exp(B_r), K rows by
// exp(B_end - B_r) and gamma = exp(B_end), every factor <= 1. The scores are one
// plain q k^T product on the tensor cores (tcgen05), scaled and masked when
// they are read out; no per-element exponentials of q or k are needed.
// Items of a CTA run in order (load, product, readout), so the SM is kept busy by
// many CTAs: without a gate, small ones (four warps, as many per SM as shared
// memory allows); with the per-head decay, eight warps share the Q and K scaling.
template <int DK>
constexpr int prep_uniform_bufs() { return 1; }
// (the per-token gate at dk = 256 runs two: three left it 80 registers and a 72-byte spill, and
// two measured 2% faster on the 1.3B-shaped layer)
template <int DK, int NTU, int GATE>
constexpr int prep_uniform_ctas_per_sm() {
    return DK > 256 ? 1 : DK > 128 ? (GATE == GLA_GATE_TOKEN_SCALAR ? 2 : 3) : (NTU == 128 ? 6 : 4);
}
template <int DK>
constexpr int prep_uniform_smem() { return prep_uniform_bufs<DK>() * 2 * C * DK * 2 + 64 + C * 4 + 1024; }

// L2 prefetch hints for the bytes [p, p + n) (n > 0) of a row of 4-byte values;
// only addresses of elements inside the row are named.
__device__ __forceinline__ void prefetch_row_l2(const float* p, int n) {
    for (int i = 0; i < n; i += 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + i));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p + n - 1));
}

template <int DK, int NTU, int GATE>
__global__ void __launch_bounds__(NTU, prep_uniform_ctas_per_sm<DK, NTU, GATE>())
gla_chunk_prep_uniform_kernel(PrepArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                              const __grid_constant__ CUtensorMap tmA)
{
    launch_dependents();   // as in gla_chunk_prep_kernel
    constexpr int NCG = DK / 8, NRG = NTU / NCG, RPT = C / NRG;
    static_assert(RPT >= 1 && C % NRG == 0, "rows split evenly over the row groups");
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = align1k(smem_raw);
    constexpr int NBUF = prep_uniform_bufs<DK>();
    constexpr int TILE = C * DK;   // bf16 elements of one q or k tile
    // buffer b: q tile at b * 2 * TILE, k tile after it ([C][DK] each, TMA, swizzled)
    __nv_bfloat16* tiles = reinterpret_cast<__nv_bfloat16*>(smem);
    uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + NBUF * 2 * TILE * 2);   // [NBUF] tile loads
    uint64_t* mbar = cbar + 2;                                                  // score MMA
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(cbar + 3);
    float* Lc = reinterpret_cast<float*>(cbar + 8);   // [C] cumulative log gate (per-token gate)

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        mbar_init(&cbar[0], 1);
        mbar_init(&cbar[1], 1);
        mbar_init(mbar, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int total = a.BH * a.nchunks;
    constexpr bool gated = GATE != GLA_GATE_NONE;
    constexpr bool tok = GATE == GLA_GATE_TOKEN_SCALAR;
    // the q/k tiles of an item (every box full-size: rows at or past T arrive as zeros)
    // per-head gate: whether an item's chunk leaves Lambda, and with a.sc its scores, to the chunk pass
    auto factored = [&](int item) -> bool {
        const int c = item % a.nchunks, h = (item / a.nchunks) % a.H;
        return GATE == GLA_GATE_HEAD_SCALAR && a.qfac && q_factored(min(C, a.T - c * C) * a.log_g[h]);
    };
    auto load = [&](int item, int b) {
        const int c = item % a.nchunks, bh = item / a.nchunks;
        __nv_bfloat16* Qb = tiles + b * 2 * TILE;
        const bool kq = !(a.sc && factored(item));   // only K (.) Gamma: no q tile
        bulk_wait_read0();   // an earlier item's A store has read its stage (a q tile)
        mbar_arrive_expect_tx(&cbar[b], (kq ? 2 : 1) * TILE * 2);
#pragma unroll
        for (int i = 0; i < DK / 64; ++i) {
            if (kq) tma_load_3d(Qb + i * C * 64, &tmq, &cbar[b], i * 64, c * C, bh);
            tma_load_3d(Qb + TILE + i * C * 64, &tmk, &cbar[b], i * 64, c * C, bh);
        }
    };
    // a load issued and not yet waited for (thread 0): no copy may land after the CTA exits
    int pend_b = -1;
    uint32_t pend_par = 0;
    if (tid == 0 && (int)blockIdx.x < total) {
        load(blockIdx.x, 0);
        pend_b = 0;
    }
    uint32_t mphase = 0;
    for (int item = blockIdx.x, it = 0; item < total; item += gridDim.x, ++it) {
    const int c = item % a.nchunks, bh = item / a.nchunks, h = bh % a.H;
    const int t0 = c * C;
    const int nr = min(C, a.T - t0);
    const float lam = GATE == GLA_GATE_HEAD_SCALAR ? a.log_g[h] : 0.f;   // log(lambda_h) <= 0
    const int cg = tid % NCG, rg = tid / NCG;
    const int col0 = cg * 8, row0 = rg * RPT;
    const int b = NBUF == 2 ? (it & 1) : 0;
    const uint32_t parity = NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
    __nv_bfloat16* Qs = tiles + b * 2 * TILE;
    __nv_bfloat16* Ks = Qs + TILE;

    if (tid == 0) {
        const int nx = item + gridDim.x;
        // the other buffer was last read by the previous item's MMA, which has completed
        if (NBUF == 2 && nx < total) {
            load(nx, b ^ 1);
            pend_b = b ^ 1;
            pend_par = ((it + 1) >> 1) & 1;
        } else {
            pend_b = -1;
        }
        const int nx2 = NBUF == 2 ? nx + gridDim.x : nx;
        if (nx2 < total) {
            const int c2 = nx2 % a.nchunks, bh2 = nx2 / a.nchunks, nr2 = min(C, a.T - c2 * C);
            const size_t row = (size_t)bh2 * a.T + (size_t)c2 * C;
            if (!(a.sc && factored(nx2))) prefetch_l2(a.q + row * DK, (uint32_t)nr2 * DK * 2);
            prefetch_l2(a.k + row * DK, (uint32_t)nr2 * DK * 2);
            if (tok) prefetch_row_l2(a.log_g + row, nr2);
        }
    }
    if (gated && !tok)
        for (int col = tid; col < DK; col += NTU) a.gam[((size_t)bh * a.nchunks + c) * DK + col] = __expf(nr * lam);
    if (tok && warp == 2) {
        // inclusive cumulative log gate of the chunk's rows, two rows per lane; rows at or
        // past T add 0 (the previous item's readers of Lc finished at its last barrier)
        const float* gr = a.log_g + (size_t)bh * a.T + t0;
        const float g0 = 2 * lane < nr ? gr[2 * lane] : 0.f;
        const float g1 = 2 * lane + 1 < nr ? gr[2 * lane + 1] : 0.f;
        float run = g0 + g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, run, o);
            if (lane >= o) run += u;
        }
        Lc[2 * lane] = run - g1;
        Lc[2 * lane + 1] = run;
    }
    // The tiles come from TMA and are not written here, so the product can start as soon
    // as they land; Q (.) Lambda (warps 2-3, meanwhile) and K (.) Gamma (warps 0-1, after
    // the readout) are per-row scalings of the same tiles.
    // per-head gate: a chunk whose decay stays within exp(-kQGuard) leaves Lambda to the chunk pass,
    // and with a.sc its scores too (block-uniform)
    const bool fq = GATE == GLA_GATE_HEAD_SCALAR && a.qfac && q_factored(nr * lam);
    const bool only_k = a.sc && fq;
    bool ok = mbar_wait(&cbar[b], parity, kTimeoutNs);
    if (warp == 0 && !only_k) {
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            if (lane == 0) score_mma<DK>(reinterpret_cast<uint8_t*>(Qs), reinterpret_cast<uint8_t*>(Ks), tmem, mbar);
        }
        __syncwarp();
    }
    // nothing proceeds (the readout waits on the product) unless every thread saw its tiles
    if (__syncthreads_or(!ok)) {
        if (tid == 0) atomicExch(a.status, ERR_PREP);
        break;
    }
    if (tok)
        for (int col = tid; col < DK; col += NTU) a.gam[((size_t)bh * a.nchunks + c) * DK + col] = __expf(Lc[C - 1]);
    // Q (pass 0) or K (pass 1), rows [r0, r1), by nth threads
    auto scale_rows = [&](int pass, int r0, int r1, int t, int nth) {
        const __nv_bfloat16* T = pass == 0 ? Qs : Ks;
        __nv_bfloat16* out = pass == 0 ? a.Qt : a.Kt;
        for (int idx = r0 * NCG + t; idx < r1 * NCG; idx += nth) {
            const int row = idx / NCG, col = (idx % NCG) * 8;
            const float fac = row >= nr ? 0.f
                            : tok ? (pass == 0 ? __expf(Lc[row]) : __expf(Lc[C - 1] - Lc[row]))
                            : pass == 0 ? __expf((row + 1) * lam)          // b_row / b_start
                                        : __expf((nr - 1 - row) * lam);    // b_end / b_row
            float v[8];
            unpack8(*reinterpret_cast<const uint4*>(T + opi<DK>(row, col)), v);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= fac;
            *reinterpret_cast<uint4*>(out + ((size_t)bh * a.Tpad + t0 + row) * DK + col) = pack8(v);
        }
    };
    // the readout stages A in the q tile once the other warps are done reading it
    // (named barrier 2); the K rows are split in proportion to the threads
    constexpr int KSPLIT = C * (NTU - 64) / NTU;
    if (only_k) {
        scale_rows(1, 0, C, tid, NTU);
    } else if (warp < 2) {
        ok = score_readout<tok>(tmem, mbar, mphase, nr, lam, Qs, &tmA, (bh * a.nchunks + c) * C, 2, NTU, Lc, fq);
        if (gated) scale_rows(1, KSPLIT, C, tid, 64);
    } else {
        if (gated && !fq) scale_rows(0, 0, C, tid - 64, NTU - 64);
        named_bar_arrive(2, NTU);
        if (gated) scale_rows(1, 0, KSPLIT, tid - 64, NTU - 64);
    }
    if (!only_k) mphase ^= 1u;
    if (__syncthreads_or(!ok)) {   // also: the tiles and the accumulator are reused by the next item
        if (tid == 0) atomicExch(a.status, ERR_PREP);
        break;
    }
    if (NBUF == 1 && tid == 0 && item + (int)gridDim.x < total) {
        load(item + gridDim.x, 0);
        pend_b = 0;
        pend_par = (it + 1) & 1;
    }
    }
    if (tid == 0 && pend_b >= 0) mbar_wait(&cbar[pend_b], pend_par, kTimeoutNs);
    prefetch_next_stage(a, total);
    if (tid == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// q or k as a [BH][T][dk] bf16 tensor, boxes of 64 rows x 64 columns, 128-byte swizzle
bool map_rows(CUtensorMap* m, const void* base, int dk, int T, int BH) {
    uint64_t dims[3] = {(uint64_t)dk, (uint64_t)T, (uint64_t)BH};
    uint64_t str[2] = {(uint64_t)dk * 2, (uint64_t)dk * T * 2};
    uint32_t box[3] = {64, 64, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int DK, int NTU, int GATE>
cudaError_t launch_prep_uniform_nt(const PrepArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                                   const CUtensorMap& mA, int sms, cudaStream_t s)
{
    const int smem = prep_uniform_smem<DK>();
    const int total = a.BH * a.nchunks;
    const int resident = prep_uniform_ctas_per_sm<DK, NTU, GATE>() * sms;
    const dim3 grid(total < resident ? total : resident);
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_prep_uniform_kernel<DK, NTU, GATE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gla_chunk_prep_uniform_kernel<DK, NTU, GATE><<<grid, NTU, smem, s>>>(a, mq, mk, mA);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_prep_uniform_dk(const PrepArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                                   const CUtensorMap& mA, int sms, cudaStream_t s)
{
    switch (a.gate) {
    case GLA_GATE_NONE: return launch_prep_uniform_nt<DK, 128, GLA_GATE_NONE>(a, mq, mk, mA, sms, s);
    case GLA_GATE_HEAD_SCALAR: return launch_prep_uniform_nt<DK, 256, GLA_GATE_HEAD_SCALAR>(a, mq, mk, mA, sms, s);
    case GLA_GATE_TOKEN_SCALAR: return launch_prep_uniform_nt<DK, 256, GLA_GATE_TOKEN_SCALAR>(a, mq, mk, mA, sms, s);
    }
    return cudaErrorInvalidValue;
}

template <int DK>
cudaError_t launch_prep_dk(const PrepArgs& a, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mA,
                          int sms, cudaStream_t s)
{
    using L = PL<DK>;
    const int total = a.BH * a.nchunks;
    const int resident = prep_ctas_per_sm<DK>() * sms;
    const dim3 grid(total < resident ? total : resident);
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_prep_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    gla_chunk_prep_kernel<DK><<<grid, NT, L::SMEM, s>>>(a, mq, mk, mA);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s,
                        bool allow_qfac)
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
    a.qfac = allow_qfac && q_factor_offload(p);
    a.sc = a.qfac && pl.sc;
    a.pf_s0 = static_cast<const uint8_t*>(static_cast<const void*>(p.S0));
    a.pf_s0_bytes = p.S0 ? (size_t)a.BH * p.dk * p.dv * 4 : 0;
    a.pf_v = static_cast<const uint8_t*>(p.v);
    a.pf_v_stride = (size_t)p.T * p.dv * 2;
    a.pf_v_bytes = (uint32_t)((size_t)min(p.T, 2 * C) * p.dv * 2);
    const int sms = pl.sms > 0 ? pl.sms : 148;
    CUtensorMap mq, mk, mA;
    if (!map_rows(&mq, p.q, p.dk, p.T, a.BH) || !map_rows(&mk, p.k, p.dk, p.T, a.BH)) return cudaErrorInvalidValue;
    {   // A as [BH * nchunks * 64 rows][64] bf16, one 64 x 64 tile per store
        uint64_t dims[2] = {64, (uint64_t)a.BH * pl.nchunks * 64};
        uint64_t str[1] = {128};
        uint32_t box[2] = {64, 64};
        if (!make_tmap(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (p.gate != GLA_GATE_PER_KEY && p.gate != GLA_GATE_BILINEAR) {   // the bilinear gate's key side is per key
        switch (p.dk) {
        case 64: return launch_prep_uniform_dk<64>(a, mq, mk, mA, sms, s);
        case 128: return launch_prep_uniform_dk<128>(a, mq, mk, mA, sms, s);
        case 256: return launch_prep_uniform_dk<256>(a, mq, mk, mA, sms, s);
        case 512: return launch_prep_uniform_dk<512>(a, mq, mk, mA, sms, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (p.dk) {
    case 64: return launch_prep_dk<64>(a, mq, mk, mA, sms, s);
    case 128: return launch_prep_dk<128>(a, mq, mk, mA, sms, s);
    case 256: return launch_prep_dk<256>(a, mq, mk, mA, sms, s);
    case 512: return launch_prep_dk<512>(a, mq, mk, mA, sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gla
