// Test-only probe of the tcgen05 operand conventions the chunk kernel relies
// on: TMA loads into 128-byte-swizzled slabs, shared-memory descriptors for
// K-major and MN-major operands, an A operand in tensor memory, and the
// accumulator layout read back with tcgen05.ld. One CTA, one product:
//   mode 0  D[128x256] = V^T K      (A MN-major, B MN-major, K = 64)
//   mode 1  D[128x64]  = V^T P^T    (A MN-major, B K-major,  K = 64)
//   mode 2  D[128x64]  = Sb  Q^T    (A in TMEM,  B K-major,  K = 256)
#include <cstdio>
#include <cuda_bf16.h>

#include "sm100.cuh"
#include "tma_host.h"

using namespace gla;
using namespace gla::sm100;

namespace {

constexpr uint64_t kTimeout = 2000000000ull;  // 2 s

struct ProbeArgs {
    int mode;
    int swap;                  // swap LBO/SBO of MN-major descriptors (diagnostic)
    const __nv_bfloat16* sb;   // mode 2: [128][256]
    float* D;                  // [128][N]
    int* err;
};

__global__ void __launch_bounds__(128) umma_probe_kernel(ProbeArgs a, const __grid_constant__ CUtensorMap mA,
                                                         const __grid_constant__ CUtensorMap mB)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* As = base;               // 32 KB
    uint8_t* Bs = base + 32768;       // 32 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + 65536);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + 65536 + 64);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int N = a.mode == 0 ? 256 : 64;

    if (warp == 0) tmem_alloc(tmem_holder, 512);
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (a.mode == 2) {
        // row m of Sb -> TMEM lane m, columns [256, 384), two bf16 per column
        const int m = threadIdx.x;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(a.sb + (size_t)m * 256);
        for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            for (int i = 0; i < 32; ++i) r[i] = row[c * 32 + i];
            tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + 256 + c * 32, r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool ok = true;
    if (threadIdx.x == 0) {
        uint32_t bytes = 0;
        if (a.mode == 0) bytes = 2 * 8192 + 4 * 8192;
        if (a.mode == 1) bytes = 2 * 8192 + 8192;
        if (a.mode == 2) bytes = 4 * 8192;
        mbar_arrive_expect_tx(&bars[0], bytes);
        if (a.mode != 2) {
            tma_load_2d(As, &mA, &bars[0], 0, 0);
            tma_load_2d(As + 8192, &mA, &bars[0], 64, 0);
        }
        const int nb = a.mode == 1 ? 1 : 4;
        for (int i = 0; i < nb; ++i) tma_load_2d(Bs + i * 8192, &mB, &bars[0], i * 64, 0);
        ok = mbar_wait(&bars[0], 0, kTimeout);
        if (ok) {
            tc_fence_after();
            const uint32_t lbo_mn = a.swap ? 1024 : 8192, sbo_mn = a.swap ? 8192 : 1024;
            if (a.mode == 0) {
                const uint32_t id = idesc_bf16(128, 256, true, true);
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem, sdesc(smem_u32(As) + kk * 2048, lbo_mn, sbo_mn, kSwizzle128),
                           sdesc(smem_u32(Bs) + kk * 2048, lbo_mn, sbo_mn, kSwizzle128), id, kk > 0);
            } else if (a.mode == 1) {
                const uint32_t id = idesc_bf16(128, 64, true, false);
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem, sdesc(smem_u32(As) + kk * 2048, lbo_mn, sbo_mn, kSwizzle128),
                           sdesc(smem_u32(Bs) + kk * 32, 16, 1024, kSwizzle128), id, kk > 0);
            } else {
                const uint32_t id = idesc_bf16(128, 64, false, false);
                for (int kk = 0; kk < 16; ++kk)
                    mma_ts(tmem, tmem + 256 + kk * 8,
                           sdesc(smem_u32(Bs) + (kk / 4) * 8192 + (kk % 4) * 32, 16, 1024, kSwizzle128), id, kk > 0);
            }
            mma_commit(&bars[1]);
        } else {
            atomicExch(a.err, 1);
        }
    }
    __syncthreads();
    if (*((volatile int*)a.err) == 0) {
        if (!mbar_wait(&bars[1], 0, kTimeout)) {
            atomicExch(a.err, 2);
        } else {
            tc_fence_after();
            const int m = warp * 32 + lane;
            for (int c = 0; c < N / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
                tmem_wait_ld();
                for (int i = 0; i < 32; ++i) a.D[(size_t)m * N + c * 32 + i] = __uint_as_float(r[i]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

// A and B are device pointers to bf16 row-major arrays:
//   mode 0: A = V [64][128], B = K [64][256]
//   mode 1: A = V [64][128], B = P [64][64]
//   mode 2: A = Sb [128][256] (read by threads), B = Q [64][256]
// D is a device fp32 array [128][N]. Returns 0 on success.
extern "C" int umma_probe(int mode, int swap, const void* A, const void* B, float* D)
{
    CUtensorMap mA, mB;
    memset(&mA, 0, sizeof(mA));
    uint32_t box[2] = {64, 64};
    if (mode != 2) {
        uint64_t dims[2] = {128, 64}, str[1] = {128 * 2};
        if (!make_tmap(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return 10;
    }
    {
        uint64_t bw = mode == 1 ? 64 : 256;
        uint64_t dims[2] = {bw, 64}, str[1] = {bw * 2};
        if (!make_tmap(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return 11;
    }
    int* err = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return 12;
    cudaMemset(err, 0, sizeof(int));
    ProbeArgs a{mode, swap, static_cast<const __nv_bfloat16*>(A), D, err};
    const int smem = 65536 + 1024 + 1024;
    cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    umma_probe_kernel<<<1, 128, smem>>>(a, mA, mB);
    cudaError_t e = cudaDeviceSynchronize();
    int h = 0;
    cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(err);
    if (e != cudaSuccess) {
        fprintf(stderr, "umma_probe: %s\n", cudaGetErrorString(e));
        return 20;
    }
    return h;
}
