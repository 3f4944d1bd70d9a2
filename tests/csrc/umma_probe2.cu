// Test-only probe of two more tcgen05 operand conventions, each one CTA and one
// product, read back from tensor memory:
//   mode 3  D[128x64] = V^T P^T with B (P, 64 x 64, K-major) stored as four 16-column
//           blocks in the no-swizzle layout: 8-row x 16-byte core matrices, block kk
//           at kk * 2048, core (row / 8, col / 8) at (row / 8) * 256 + (col / 8) * 128,
//           i.e. SBO = 256 (next 8 rows), LBO = 128 (next 8 columns along K)
//   mode 4  rows 64..127 of D[128x16] = Q K[16c, 16c + 16)^T, K = 256 keys: the A
//           operand starts 8 KB (64 rows) before each 128-byte-swizzled slab of Q, so
//           the 64 query rows are rows 64-127 of an M = 128 product, and N = 16 rows
//           of K start 16 c rows into its slabs; read by the warps of TMEM lanes 64-127
//           with 16-column loads.
#include <cstdio>
#include <cstring>
#include <cuda_bf16.h>

#include "sm100.cuh"
#include "tma_host.h"

using namespace gla;
using namespace gla::sm100;

namespace {

constexpr uint64_t kTimeout = 2000000000ull;

struct Probe2Args {
    int mode, c, swap;
    const __nv_bfloat16* P;   // mode 3: [64][64]
    float* D;                 // mode 3: [128][64]; mode 4: [64][16]
    int* err;
};

__global__ void __launch_bounds__(128) umma_probe2_kernel(Probe2Args a, const __grid_constant__ CUtensorMap mA,
                                                          const __grid_constant__ CUtensorMap mB)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // mode 3: As = V (2 slabs, 16 KB), Bs = P blocks (8 KB). mode 4: 8 KB pad, Q (32 KB), K (32 KB)
    uint8_t* As = base + 8192;
    uint8_t* Bs = base + 8192 + 32768;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + 8192 + 65536);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + 8192 + 65536 + 64);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (warp == 0) tmem_alloc(tmem_holder, 128);
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    if (a.mode == 3) {
        // P into the four no-swizzle blocks, one 16-byte core-matrix row per thread step
        for (int i = threadIdx.x; i < 64 * 8; i += 128) {
            const int r = i / 8, g = i % 8, s = g * 8, kk = s / 16, sc = s % 16;
            const uint4 v = *reinterpret_cast<const uint4*>(a.P + (size_t)r * 64 + s);
            *reinterpret_cast<uint4*>(Bs + kk * 2048 + (r >> 3) * 256 + (sc >> 3) * 128 + (r & 7) * 16) = v;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (threadIdx.x == 0) {
        const uint32_t bytes = a.mode == 3 ? 2 * 8192 : 8 * 8192;
        mbar_arrive_expect_tx(&bars[0], bytes);
        if (a.mode == 3) {
            tma_load_2d(As, &mA, &bars[0], 0, 0);
            tma_load_2d(As + 8192, &mA, &bars[0], 64, 0);
        } else {
            for (int i = 0; i < 4; ++i) {
                tma_load_2d(As + i * 8192, &mA, &bars[0], i * 64, 0);
                tma_load_2d(Bs + i * 8192, &mB, &bars[0], i * 64, 0);
            }
        }
        if (mbar_wait(&bars[0], 0, kTimeout)) {
            tc_fence_after();
            if (a.mode == 3) {
                const uint32_t id = idesc_bf16(128, 64, true, false);
                const uint32_t lbo = a.swap ? 256 : 128, sbo = a.swap ? 128 : 256;
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem, sdesc(smem_u32(As) + kk * 2048, 8192, 1024, kSwizzle128),
                           sdesc(smem_u32(Bs) + kk * 2048, lbo, sbo, kNoSwizzle), id, kk > 0);
            } else {
                const uint32_t id = idesc_bf16(128, 16, false, false);
                for (int kk = 0; kk < 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                    mma_ss(tmem, sdesc(smem_u32(As) + off - 8192, 16, 1024, kSwizzle128),
                           sdesc(smem_u32(Bs) + off + a.c * 16 * 128, 16, 1024, kSwizzle128), id, kk > 0);
                }
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
            const uint32_t lq = (uint32_t)(warp * 32) << 16;
            if (a.mode == 3) {
                for (int c = 0; c < 2; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lq + c * 32, r);
                    tmem_wait_ld();
                    for (int i = 0; i < 32; ++i) a.D[(size_t)m * 64 + c * 32 + i] = __uint_as_float(r[i]);
                }
            } else if (warp >= 2) {
                uint32_t r[16];
                tmem_ld16(tmem + lq, r);
                tmem_wait_ld();
                for (int i = 0; i < 16; ++i) a.D[(size_t)(m - 64) * 16 + i] = __uint_as_float(r[i]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

// mode 3: A = V [64][128], P = [64][64] (device, bf16), D = [128][64] fp32.
// mode 4: A = Q [64][256], B = K [64][256] (device, bf16), c in 0..3, D = [64][16] fp32.
// Returns 0 on success.
extern "C" int umma_probe2(int mode, int c, int swap, const void* A, const void* B, float* D)
{
    CUtensorMap mA, mB;
    memset(&mA, 0, sizeof(mA));
    memset(&mB, 0, sizeof(mB));
    uint32_t box[2] = {64, 64};
    if (mode == 3) {
        uint64_t dims[2] = {128, 64}, str[1] = {128 * 2};
        if (!make_tmap(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return 10;
    } else {
        uint64_t dims[2] = {256, 64}, str[1] = {256 * 2};
        if (!make_tmap(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return 10;
        if (!make_tmap(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return 11;
    }
    int* err = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return 12;
    cudaMemset(err, 0, sizeof(int));
    Probe2Args a{mode, c, swap, static_cast<const __nv_bfloat16*>(B), D, err};
    const int smem = 8192 + 65536 + 1024 + 1024;
    cudaFuncSetAttribute(umma_probe2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    umma_probe2_kernel<<<1, 128, smem>>>(a, mA, mB);
    cudaError_t e = cudaDeviceSynchronize();
    int h = 0;
    cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(err);
    if (e != cudaSuccess) {
        fprintf(stderr, "umma_probe2: %s\n", cudaGetErrorString(e));
        return 20;
    }
    return h;
}
