// quantize.cuh - nvfp4_quantize: NVFP4 quantisation of a row-major matrix
// ("Let's optimize Nemotron 3.5 Lightning - a worklog", Step 1: 4-bit values
// with one scale per 16 elements; Step 3: dynamic per-row activations).
//
// HBM-bound elementwise work: one thread per 16-element block, 16-byte loads,
// 8-byte code stores; PER_TENSOR adds a grid-wide amax pass (atomicMax on the
// float bits, which order like unsigned integers for non-negative values).
#pragma once

#include "common.cuh"

namespace nvfp4moe {

template <bool BF16>
__device__ __forceinline__ void load_block16(const void* x, int64_t blk, float (&v)[16]) {
    if (BF16) {
        const uint4* p = reinterpret_cast<const uint4*>(x) + 2 * blk;
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(x) + 4 * blk;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 f = __ldg(p + i);
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
    }
}

// amax over all elements -> atomicMax into *amax_bits (float bits)
template <bool BF16>
__global__ void __launch_bounds__(256) k_amax(const void* x, int64_t nblocks, unsigned int* amax_bits) {
    float m = 0.0f;
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        float v[16];
        load_block16<BF16>(x, b, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    m = warp_max(m);
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        float r = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        r = warp_max(r);
        if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(r));
    }
}

// Blocks quantised with one global. gsrc_is_amax: *gsrc holds amax bits
// (PER_TENSOR), else *gsrc is the global itself (GIVEN).
template <bool BF16>
__global__ void __launch_bounds__(256) k_quantize_global(const void* x, int64_t nblocks,
                                                         const float* gsrc, int gsrc_is_amax,
                                                         uint8_t* codes, uint8_t* scales) {
    const float g = gsrc_is_amax ? __fdiv_rn(__uint_as_float(*reinterpret_cast<const unsigned int*>(gsrc)), 2688.0f)
                                 : *gsrc;
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        float v[16];
        load_block16<BF16>(x, b, v);
        const QBlock q = quantize_block16(v, g);
        reinterpret_cast<uint2*>(codes)[b] = make_uint2(q.lo, q.hi);
        scales[b] = static_cast<uint8_t>(q.scale);
    }
}

__global__ void k_finalize_global(float* g) {
    g[0] = __fdiv_rn(__uint_as_float(*reinterpret_cast<unsigned int*>(g)), 2688.0f);
}

// One warp per row: row amax, g = amax / 2688, then the row's blocks.
template <bool BF16>
__global__ void __launch_bounds__(256) k_quantize_rows(const void* x, int64_t rows, int64_t cols,
                                                       float* gout, uint8_t* codes, uint8_t* scales) {
    const int lane = threadIdx.x & 31;
    const int64_t nb = cols / 16;
    for (int64_t r = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; r < rows;
         r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        float m = 0.0f;
        for (int64_t b = lane; b < nb; b += 32) {
            float v[16];
            load_block16<BF16>(x, r * nb + b, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
        }
        m = warp_max(m);
        const float g = __fdiv_rn(m, 2688.0f);
        if (lane == 0) gout[r] = g;
        for (int64_t b = lane; b < nb; b += 32) {
            float v[16];
            load_block16<BF16>(x, r * nb + b, v);
            const QBlock q = quantize_block16(v, g);
            reinterpret_cast<uint2*>(codes)[r * nb + b] = make_uint2(q.lo, q.hi);
            scales[r * nb + b] = static_cast<uint8_t>(q.scale);
        }
    }
}

}  // namespace nvfp4moe
