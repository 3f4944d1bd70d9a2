// gla_chunk_state: the state-only pass of the sequence split. For every
// (b, h), tile of 128 dv columns and segment s it computes the state the
// segment leaves from a zero start,
//
//     S*_s = sum over the segment's chunks n of (Kt_n (.) sfx_n)^T V_n,
//     sfx_n = prod over the later chunks m of the segment of gamma_m (per key),
//
// which is the chunk recurrence S_n = Diag(gamma_n) S_(n-1) + Kt_n^T V_n
// ("Gated Linear Attention Transformers with Hardware-Efficient Training",
// §4.2) unrolled: each chunk's contribution decays to the segment end by the
// product of the gates after it. Walking the chunks from the segment's end,
// sfx is a running product, so each chunk's K tile is scaled once in shared
// memory (every factor <= 1) and the tensor cores only accumulate; no state
// is rescaled in tensor memory between chunks. The gla_state_scan kernel then
// chains the segments with the segment decays. (In the forward pass the
// "segments" are the split's state-pass pieces: the chunks before the chunk
// pass's last segment, cut finer than its segments so that they fill the GPU.)
//
// Warp roles: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2-9 scale the K
// tiles and finally read the state out (two groups of four warps, one TMEM
// lane quarter per warp, half of the state's columns per group). Every wait
// is bounded; on a timeout the CTA records an error code and winds down.
#include <cuda_bf16.h>

#include "gla_internal.h"
#include "sm100.cuh"
#include "tma_host.h"

namespace gla {
namespace {

using namespace sm100;

constexpr int C = kChunk;
constexpr int DVT = kDvTile;
constexpr int NT = 320;
constexpr int NS = 4;                             // operand stages in flight
constexpr int NSC = 256;                          // scaling threads (warps 2-9)
constexpr int BAR_SC = 1;                         // named barrier of the scaling warps
constexpr uint64_t kTimeoutNs = 2000000000ull;    // 2 s per wait

enum { ERR_PRODUCER = 0x301, ERR_MMA = 0x302, ERR_SCALE = 0x303 };

struct StateArgs {
    const float* gam;   // [BH][nchunks][dk], null without a gate
    float* S_out;       // segment states: [BH][nseg][dk][dv]
    long long s_out_bh, s_out_seg;
    int* status;
    int dv, nchunks, cps, gated;
    int win;            // > 0: segment s covers the win chunks before chunk s * cps (sliding window)
    int rev;            // walk from the segment's first chunk (the decay runs over the earlier chunks)
};

template <int DK>
struct SL {
    static constexpr int KB = DK * C * 2;
    static constexpr int VB = DVT * C * 2;
    static constexpr int GB = DK * 4;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = KB;
    static constexpr int G_OFF = KB + VB;
    static constexpr int STAGE = (G_OFF + GB + 1023) / 1024 * 1024;
    static constexpr int BAR_OFF = NS * STAGE;
    static constexpr int SMEM = BAR_OFF + 8 * (3 * NS + 3) + 1024;
    static constexpr int TCOLS = DK < 32 ? 32 : DK;
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

template <int DK>
__global__ void __launch_bounds__(NT, 1)
gla_chunk_state_kernel(StateArgs a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV)
{
    using L = SL<DK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
    uint64_t* full = bar + 0;           // [NS] stage filled
    uint64_t* empty = bar + NS;         // [NS] stage consumed by the MMA
    uint64_t* scaled = bar + 2 * NS;    // [NS] K tile scaled (256 arrivals)
    uint64_t* done = bar + 3 * NS;      // all MMAs complete
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 3 * NS + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 3 * NS + 2);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.y, seg = blockIdx.z;
    const int dv0 = blockIdx.x * DVT;
    const int c_begin = a.win > 0 ? max(0, seg * a.cps - a.win) : seg * a.cps;
    const int c_end = a.win > 0 ? seg * a.cps : min(a.nchunks, c_begin + a.cps);
    const int nloc = max(0, c_end - c_begin);
    const bool gated = a.gated != 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&scaled[i], NSC);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, L::TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer, last chunk first
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nloc; ++j) {
                if (*abort_flag) break;
                const int st = j % NS, c = a.rev ? c_begin + j : c_end - 1 - j;
                if (j >= NS && !mbar_wait(&empty[st], ((j / NS) - 1) & 1, kTimeoutNs)) {
                    fail(a.status, abort_flag, ERR_PRODUCER);
                    break;
                }
                uint8_t* sb = sm + st * L::STAGE;
                mbar_arrive_expect_tx(&full[st], L::KB + L::VB + (gated ? L::GB : 0));
                if (gated) bulk_load(sb + L::G_OFF, a.gam + ((size_t)bh * a.nchunks + c) * DK, L::GB, &full[st]);
#pragma unroll
                for (int i = 0; i < DK / 64; ++i) tma_load_3d(sb + L::K_OFF + i * 8192, &tmK, &full[st], i * 64, c * C, bh);
                tma_load_3d(sb + L::V_OFF, &tmV, &full[st], dv0, c * C, bh);
                tma_load_3d(sb + L::V_OFF + 8192, &tmV, &full[st], dv0 + 64, c * C, bh);
                const int cp = a.rev ? c + NS : c - NS;   // NS chunks ahead in this order
                if (a.rev ? cp < c_end : cp >= c_begin) {
                    prefetch_l2_tile_3d(&tmV, dv0, cp * C, bh);
                    prefetch_l2_tile_3d(&tmV, dv0 + 64, cp * C, bh);
                    const int nt = gridDim.x, me = blockIdx.x;
#pragma unroll
                    for (int i = 0; i < DK / 64; ++i)
                        if (i % nt == me) prefetch_l2_tile_3d(&tmK, i * 64, cp * C, bh);
                }
                issued = j + 1;
            }
            for (int j = max(0, issued - NS); j < issued; ++j) mbar_wait(&full[j % NS], (j / NS) & 1, kTimeoutNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_state = idesc_bf16(128, DK, true, true);
            bool ok = true;
            for (int j = 0; j < nloc; ++j) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                const int st = j % NS;
                ok = mbar_wait(&full[st], (j / NS) & 1, kTimeoutNs);
                if (ok && gated) ok = mbar_wait(&scaled[st], (j / NS) & 1, kTimeoutNs);
                if (!ok) {
                    fail(a.status, abort_flag, ERR_MMA);
                    break;
                }
                tc_fence_after();
                const uint32_t sb = smem_u32(sm + st * L::STAGE);
                // S*^T += V^T (K (.) sfx); both operands MN-major
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tS, sdesc(sb + L::V_OFF + kk * 2048, 8192, 1024, kSwizzle128),
                           sdesc(sb + L::K_OFF + kk * 2048, 8192, 1024, kSwizzle128), id_state, (j > 0 || kk > 0));
                mma_commit(&empty[st]);
            }
            // the commit tracks every MMA issued above; the lane waits for it, so that on an
            // abort as on the normal path no MMA still runs when the TMEM is freed (the
            // readout warps also check the abort flag before they trust `done`)
            mma_commit(done);
            mbar_wait(done, 0, kTimeoutNs);
            (void)ok;
        }
    } else {
        // ---------------------------------------------------------- K scaling, then the state readout
        const int t = threadIdx.x - 64;
        const int grp = (warp - 2) >> 2;
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const int d = (warp & 3) * 32 + lane;
        const int cb = grp * (DK / 2);
        bool alive = true;
        if (gated) {
            // The K tile is DK / 64 slabs of 64 rows x 128 B in the 128-byte swizzle.
            // Thread t scales the 16-byte pieces t + NSC u (u < DK / 32): piece u lies in
            // slab u / 2, row t / 8 + 32 (u % 2), and holds keys (u / 2) 64 + kq .. + 7 with
            // kq = 8 ((t % 8) ^ (t / 8 % 8)). So a thread only ever touches 8 keys per slab
            // and keeps their running decays in registers.
            constexpr int NU = DK / 32, NSL = DK / 64;
            const int kq = ((t & 7) ^ ((t >> 3) & 7)) << 3;
            float f[NSL][8];
#pragma unroll
            for (int sl = 0; sl < NSL; ++sl)
#pragma unroll
                for (int e = 0; e < 8; ++e) f[sl][e] = 1.f;   // the last chunk's contribution is not decayed
            for (int j = 0; j < nloc; ++j) {
                const int st = j % NS;
                if (!mbar_wait(&full[st], (j / NS) & 1, kTimeoutNs)) {
                    alive = false;
                    break;
                }
                uint8_t* sb = sm + st * L::STAGE;
                uint4* kp = reinterpret_cast<uint4*>(sb + L::K_OFF) + t;
                uint4 v[NU];
#pragma unroll
                for (int u = 0; u < NU; ++u) v[u] = kp[u * NSC];
#pragma unroll
                for (int u = 0; u < NU; ++u) {
                    const float* fu = f[u >> 1];
                    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v[u]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = __bfloat1622float2(h[e]);
                        h[e] = __floats2bfloat162_rn(x.x * fu[2 * e], x.y * fu[2 * e + 1]);
                    }
                }
#pragma unroll
                for (int u = 0; u < NU; ++u) kp[u * NSC] = v[u];
                // the decay for the next (earlier) chunk: times this chunk's gamma, read
                // before the stage is handed to the MMA (which then releases it to the producer)
                const float* g = reinterpret_cast<const float*>(sb + L::G_OFF) + kq;
#pragma unroll
                for (int sl = 0; sl < NSL; ++sl) {
                    const float4 g0 = *reinterpret_cast<const float4*>(g + sl * 64);
                    const float4 g1 = *reinterpret_cast<const float4*>(g + sl * 64 + 4);
                    f[sl][0] *= g0.x; f[sl][1] *= g0.y; f[sl][2] *= g0.z; f[sl][3] *= g0.w;
                    f[sl][4] *= g1.x; f[sl][5] *= g1.y; f[sl][6] *= g1.z; f[sl][7] *= g1.w;
                }
                fence_proxy_async_smem();
                mbar_arrive(&scaled[st]);
            }
            if (!alive) fail(a.status, abort_flag, ERR_SCALE);
        }
        if (nloc > 0) {
            // every scaling thread reaches this barrier, whatever happened above
            const bool ok = alive && !*abort_flag && mbar_wait(done, 0, kTimeoutNs);
            if (group_all_ok(ok, BAR_SC, NSC)) {
                tc_fence_after();
                float* so = a.S_out + bh * a.s_out_bh + seg * a.s_out_seg + dv0 + d;
#pragma unroll 1
                for (int c0 = cb; c0 < cb + DK / 2; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tS + lb + c0, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) so[(size_t)(c0 + i) * a.dv] = __uint_as_float(r[i]);
                }
            } else if (t == 0) {
                fail(a.status, abort_flag, ERR_SCALE);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tS, L::TCOLS);
    }
}

bool map_tiles(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2) {
    uint64_t dims[3] = {d0, d1, d2};
    uint64_t str[2] = {d0 * 2, d0 * d1 * 2};
    uint32_t box[3] = {64, 64, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int DK>
cudaError_t launch_state_dk(const StateArgs& a, dim3 grid, const CUtensorMap& k, const CUtensorMap& v, cudaStream_t s) {
    using L = SL<DK>;
    cudaError_t e = cudaFuncSetAttribute(gla_chunk_state_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    gla_chunk_state_kernel<DK><<<grid, NT, L::SMEM, s>>>(a, k, v);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_seg_state(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s,
                             float* S_out)
{
    if (S_out && pl.nseg != 1) return cudaErrorInvalidValue;
    uint8_t* base = static_cast<uint8_t*>(ws);
    const uint64_t BH = (uint64_t)p.B * p.H;
    const void* kb = pl.raw_qk ? p.k : base + pl.off_kt;
    const uint64_t krows = pl.raw_qk ? (uint64_t)p.T : (uint64_t)pl.Tpad;
    CUtensorMap mk, mv;
    if (!map_tiles(&mk, kb, p.dk, krows, BH)) return cudaErrorInvalidValue;
    if (!map_tiles(&mv, p.v, p.dv, p.T, BH)) return cudaErrorInvalidValue;
    StateArgs a;
    const long long st = (long long)p.dk * p.dv;
    a.gam = reinterpret_cast<const float*>(base + pl.off_gam);
    // one segment: the whole sequence to S_out; the split: its st_nseg pieces to the workspace
    const int nz = S_out ? 1 : pl.st_nseg;
    if (nz < 1) return cudaErrorInvalidValue;
    a.S_out = S_out ? S_out : reinterpret_cast<float*>(base + pl.off_segS);
    a.s_out_bh = st * nz;
    a.s_out_seg = st;
    a.status = status;
    a.dv = p.dv; a.nchunks = pl.nchunks; a.cps = S_out ? pl.chunks_per_seg : pl.st_cps;
    a.gated = p.gate != GLA_GATE_NONE;
    a.win = 0;
    a.rev = 0;
    dim3 grid(pl.n_dvt, (unsigned)BH, nz);
    switch (p.dk) {
    case 64: return launch_state_dk<64>(a, grid, mk, mv, s);
    case 128: return launch_state_dk<128>(a, grid, mk, mv, s);
    case 256: return launch_state_dk<256>(a, grid, mk, mv, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_seg_window(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s)
{
    if (pl.window <= 0 || pl.nseg < 2) return cudaErrorInvalidValue;
    uint8_t* base = static_cast<uint8_t*>(ws);
    const uint64_t BH = (uint64_t)p.B * p.H;
    const size_t st = (size_t)p.dk * p.dv;
    float* segin = reinterpret_cast<float*>(base + pl.off_segin);
    // segment 0 starts from S0 (or zero): [BH] blocks of st floats, nseg * st apart
    cudaError_t e = p.S0 ? cudaMemcpy2DAsync(segin, pl.segin_n * st * 4, p.S0, st * 4, st * 4, BH,
                                             cudaMemcpyDeviceToDevice, s)
                         : cudaMemset2DAsync(segin, pl.segin_n * st * 4, 0, st * 4, BH, s);
    if (e != cudaSuccess) return e;
    const void* kb = pl.raw_qk ? p.k : base + pl.off_kt;
    const uint64_t krows = pl.raw_qk ? (uint64_t)p.T : (uint64_t)pl.Tpad;
    CUtensorMap mk, mv;
    if (!map_tiles(&mk, kb, p.dk, krows, BH)) return cudaErrorInvalidValue;
    if (!map_tiles(&mv, p.v, p.dv, p.T, BH)) return cudaErrorInvalidValue;
    StateArgs a;
    a.gam = reinterpret_cast<const float*>(base + pl.off_gam);
    a.S_out = segin;   // segment s's window state goes to its start state; segment 0 has no window
    a.s_out_bh = (long long)st * pl.segin_n;
    a.s_out_seg = (long long)st;
    a.status = status;
    a.dv = p.dv; a.nchunks = pl.nchunks; a.cps = pl.chunks_per_seg;
    a.gated = p.gate != GLA_GATE_NONE;
    a.win = pl.window;
    a.rev = 0;
    dim3 grid(pl.n_dvt, (unsigned)BH, pl.nseg);
    switch (p.dk) {
    case 64: return launch_state_dk<64>(a, grid, mk, mv, s);
    case 128: return launch_state_dk<128>(a, grid, mk, mv, s);
    case 256: return launch_state_dk<256>(a, grid, mk, mv, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_seg_state_job(const SegStateJob& j, int* status, cudaStream_t s)
{
    if (j.dv % DVT != 0 || j.nseg < 1) return cudaErrorInvalidValue;
    const uint64_t BH = (uint64_t)j.BH;
    CUtensorMap mk, mv;
    if (!map_tiles(&mk, j.kt, j.dk, (uint64_t)j.kt_rows, BH)) return cudaErrorInvalidValue;
    if (!map_tiles(&mv, j.v, j.dv, j.T, BH)) return cudaErrorInvalidValue;
    StateArgs a;
    const long long st = (long long)j.dk * j.dv;
    a.gam = j.gam;
    a.S_out = j.S_out;
    a.s_out_bh = st * j.nseg;
    a.s_out_seg = st;
    a.status = status;
    a.dv = j.dv; a.nchunks = j.nch; a.cps = j.cps;
    a.gated = j.gam != nullptr;
    a.win = 0;
    a.rev = j.reverse ? 1 : 0;
    dim3 grid(j.dv / DVT, (unsigned)BH, j.nseg);
    switch (j.dk) {
    case 64: return launch_state_dk<64>(a, grid, mk, mv, s);
    case 128: return launch_state_dk<128>(a, grid, mk, mv, s);
    case 256: return launch_state_dk<256>(a, grid, mk, mv, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gla
