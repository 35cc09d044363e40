// Self-test of the tensor-core operand conventions the attention kernels rely
// on: 128-byte-swizzled shared-memory tiles described by tcgen05 matrix
// descriptors, K-major and MN-major, bf16 in, fp32 accumulate in tensor
// memory, read back with tcgen05.ld. One CTA, one 128x128x64 product.
// Mode 3 takes A from tensor memory instead (written by the threads with
// tcgen05.st, row i in lane i, two bf16 per column) and B MN-major.
// Mode 4 issues nothing: the wait for the MMA's completion can never succeed,
// so it must give up after its bound, record kErrWaitTimeout, free the tensor
// memory and return -- the failure path every kernel's waits take.
//
// Operands are staged into shared memory by the threads (the same byte
// layout a 128-byte-swizzle TMA load produces), inside a 200 KB dynamic
// allocation so that any descriptor offset the host passes (each at most
// 16 KB) stays within the CTA's shared memory.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace pkv {
namespace {

constexpr int kSmem = 200 * 1024;

// Writes rows x 64 bf16 (row-major source with row stride `ld` elements,
// starting at column c0) into a 128-byte-swizzled tile at dst.
__device__ void stage_sw128(uint8_t* dst, const __nv_bfloat16* src, int rows, int ld, int c0) {
    for (int i = threadIdx.x; i < rows * 8; i += blockDim.x) {
        const int r = i / 8, ch = i % 8;
        const uint4 v = *reinterpret_cast<const uint4*>(src + (size_t)r * ld + c0 + ch * 8);
        *reinterpret_cast<uint4*>(dst + tc::sw128_offset(r, ch)) = v;
    }
}

__global__ void __launch_bounds__(128) umma_selftest_kernel(int mode, const __nv_bfloat16* a,
        const __nv_bfloat16* b, float* d, int lbo, int sbo, int* err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;                 // 16 KB
    uint8_t* sB = smem + 16384;         // 16 KB
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x / 32;

    // Stage operands.
    if (mode == 4) {
        // nothing to stage
    } else if (mode == 2) {                    // A stored [K=64][M=128]: two 64-wide M halves
        stage_sw128(sA, a, 64, 128, 0);
        stage_sw128(sA + 8192, a, 64, 128, 64);
    } else if (mode != 3) {             // A stored [M=128][K=64]
        stage_sw128(sA, a, 128, 64, 0);
    }
    if (mode == 4) {
        // nothing to stage
    } else if (mode >= 1) {             // B stored [K=64][N=128]
        stage_sw128(sB, b, 64, 128, 0);
        stage_sw128(sB + 8192, b, 64, 128, 64);
    } else {                            // B stored [N=128][K=64]
        stage_sw128(sB, b, 128, 64, 0);
    }
    tc::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 256);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t t_A = tmem + 128;    // mode 3: A in columns [128, 160)
    if (mode == 3) {
        // Thread i owns row i (lane i): 64 bf16 -> 32 columns, lower k in the low half.
        const int row = threadIdx.x;
        uint32_t w[32];
        for (int c = 0; c < 32; ++c) {
            const uint32_t lo = __bfloat16_as_ushort(a[(size_t)row * 64 + 2 * c]);
            const uint32_t hi = __bfloat16_as_ushort(a[(size_t)row * 64 + 2 * c + 1]);
            w[c] = lo | (hi << 16);
        }
        tc::tmem_st32(t_A + ((uint32_t)(warp * 32) << 16), w);
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
    }

    const uint32_t mn_lbo = lbo ? (uint32_t)lbo : 8192u;
    const uint32_t mn_sbo = sbo ? (uint32_t)sbo : 1024u;
    if (threadIdx.x == 0 && mode != 4) {
        const uint32_t idesc = tc::idesc_bf16(128, 128, mode == 2, mode >= 1);
        const uint32_t a0 = tc::smem_u32(sA), b0 = tc::smem_u32(sB);
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = mode == 2 ? tc::sdesc(a0 + kk * 2048, mn_lbo, mn_sbo)
                                          : tc::sdesc(a0 + kk * 32, 16, 1024);
            const uint64_t bd = mode >= 1 ? tc::sdesc(b0 + kk * 2048, mn_lbo, mn_sbo)
                                          : tc::sdesc(b0 + kk * 32, 16, 1024);
            if (mode == 3)
                tc::mma_bf16_ts(tmem, t_A + kk * 8, bd, idesc, kk > 0);
            else
                tc::mma_bf16(tmem, ad, bd, idesc, kk > 0);
        }
        tc::mma_commit(&bar);
    }
    __syncwarp();
    const bool ok = tc::mbar_wait(&bar, 0, err);
    tc::tc_fence_after();
    if (ok) {
        const int row = warp * 32 + (threadIdx.x & 31);
        for (int c = 0; c < 128; c += 32) {
            uint32_t r[32];
            tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c, r);
            tc::tmem_wait_ld(r);
            for (int j = 0; j < 32; ++j) d[row * 128 + c + j] = __uint_as_float(r[j]);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t run_selftest_umma(int mode, const void* a, const void* b, float* d, int lbo, int sbo,
                              int* d_err) {
    if (lbo < 0 || lbo > 16384 || sbo < 0 || sbo > 16384 || (lbo & 15) || (sbo & 15))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(umma_selftest_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    umma_selftest_kernel<<<1, 128, kSmem>>>(mode, static_cast<const __nv_bfloat16*>(a),
                                            static_cast<const __nv_bfloat16*>(b), d, lbo, sbo,
                                            d_err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return cudaDeviceSynchronize();
}

}  // namespace pkv
