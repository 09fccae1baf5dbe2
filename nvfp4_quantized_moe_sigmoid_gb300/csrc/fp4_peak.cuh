// fp4_peak.cuh - measures this GPU's dense FP4 tensor-pipe throughput, the
// denominator of the FP4 roofline fraction the benchmark reports for the
// grouped (prefill / high-concurrency) path. Not an operation of the pages.
//
// One CTA per SM, each issuing `iters` block-scaled MMAs
//   tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X
// of shape M = 128, N = n, K = 64 (the shape and kind the grouped GEMM uses)
// from one thread, back to back, into `chains` accumulators in tensor memory,
// on operands resident in shared memory (K-major, 128-byte swizzle, arbitrary
// E2M1 bytes) with unit E4M3 scales. The host times the launch with CUDA
// events: flops = 2 M N K iters CTAs over the elapsed time.
#pragma once

#include "moe_grouped_tc.cuh"

namespace nvfp4moe {

constexpr int kPeakThreads = 128;
constexpr int kPeakSmemA = 16384;  // 128 rows x 128 bytes
constexpr int kPeakSmemB = 32768;  // up to 256 rows x 128 bytes

__global__ void __launch_bounds__(kPeakThreads, 1) k_fp4_peak(int n, int chains, int iters) {
    extern __shared__ __align__(1024) uint8_t pk_smem[];
    uint8_t* const sa = pk_smem + ((1024u - (smem_u32(pk_smem) & 1023u)) & 1023u);
    uint8_t* const sb = sa + kPeakSmemA;
    __shared__ uint32_t tmem_s;
    __shared__ __align__(8) uint64_t done;
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kPeakSmemA + kPeakSmemB; i += kPeakThreads)
        sa[i] = static_cast<uint8_t>((i * 37u + blockIdx.x * 11u) >> 1);
    if (tid == 0) {
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    if (warp == 0) tc_alloc(&tmem_s, kTcCols);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the operand bytes, for the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;
    // unit scales (E4M3 1.0 = 0x38) in columns 448..511 of every lane
    {
        const uint32_t ad = tmem + (static_cast<uint32_t>(32 * warp) << 16) + 448;
#pragma unroll 1
        for (int col = 0; col < 64; ++col) tc_st_x1(ad + col, 0x38383838u);
        tc_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const uint64_t ad = umma_desc_sw128(smem_u32(sa)), bd = umma_desc_sw128(smem_u32(sb));
        const uint32_t idesc = umma_idesc_mxf4(n);
#pragma unroll 1
        for (int i = 0; i < iters; ++i) {
            const int ch = i % chains, ks = i & 3;
            tc_mma_mxf4(tmem + static_cast<uint32_t>(ch * n), ad + static_cast<uint64_t>(2 * ks),
                        bd + static_cast<uint64_t>(2 * ks), idesc, tmem + 448 + 4 * ks, tmem + 480 + 4 * ks,
                        i >= chains);
        }
        tc_commit(&done);
        if (!mbar_wait_bounded(&done, 0)) set_dev_error(kErrWaitDrain);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, kTcCols);
    }
}

}  // namespace nvfp4moe
