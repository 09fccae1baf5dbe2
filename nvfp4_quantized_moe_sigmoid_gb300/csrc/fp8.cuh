// fp8.cuh - the shared expert in FP8 (E4M3) per-tensor W8A8 ("nemotron35-
// w4a4-v13" card, precision table: shared experts FP8 per-tensor W8A8; "Let's
// optimize Nemotron 3.5 Lightning - a worklog", Step 3: the quant config puts
// the shared experts at "num_bits: e4m3") and the E4M3 quantiser behind it.
//
//   x_q = E4M3(x / g_x), g_x = amax(x row) / 448         per token
//   u   = g_up g_x (W_up . x_q),   a = bf16(relu(u)^2)
//   a_q = E4M3(a / g_a), g_a = amax(a row) / 448         per token
//   y   = g_dn g_a (W_dn . a_q),   out = bf16(y + residual)
//
// E4M3 x E4M3 products are exact, so mma.sync m16n8k32 (e4m3 in, FP32
// accumulate) takes the weight bytes straight from memory: nothing is
// decoded. A CTA owns one 16-row tile of W; its eight warps split the
// reduction by 64-k steps (warp w takes steps w, w + 8, ...) and their
// accumulators are added in warp order. In a step, lane (g, q) loads 16
// contiguous weight bytes of rows g and g + 8 and the same 16 bytes of the
// activation row of token g, so the reduction index is permuted alike for
// both operands. Up to 8 tokens are the MMA's columns.
#pragma once

#include "quantize.cuh"

namespace nvfp4moe {

constexpr int kF8MaxT = 8;
constexpr int kF8Warps = 8;
constexpr int kF8Threads = 32 * kF8Warps;

// E4M3 bytes of lo, hi (round to nearest even, saturating at 448; the sign of
// a value that rounds to 0 is kept) as {lo, hi}.
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 16 values -> 16 E4M3 bytes of v / g, one binary32 division each; g = 0
// (an all-zero row or tensor) gives codes 0 with the sign kept.
__device__ __forceinline__ uint4 fp8_block16(const float (&v)[16], float g) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x = v[4 * j + i];
            q[i] = g == 0.0f ? (signbit(x) ? -0.0f : 0.0f) : __fdiv_rn(x, g);
        }
        w[j] = e4m3x2_rn(q[0], q[1]) | (e4m3x2_rn(q[2], q[3]) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Blocks of 16 with one scale: *gsrc holds amax bits (per tensor: the scale
// is amax / 448) or the scale itself (given).
template <bool BF16>
__global__ void __launch_bounds__(256) k_fp8_quantize_global(const void* x, int64_t nblocks, const float* gsrc,
                                                             int gsrc_is_amax, uint8_t* q) {
    const float g = gsrc_is_amax ? __fdiv_rn(__uint_as_float(*reinterpret_cast<const unsigned int*>(gsrc)), 448.0f)
                                 : *gsrc;
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        float v[16];
        load_block16<BF16>(x, b, v);
        reinterpret_cast<uint4*>(q)[b] = fp8_block16(v, g);
    }
}

__global__ void k_fp8_finalize_global(float* g) {
    g[0] = __fdiv_rn(__uint_as_float(*reinterpret_cast<unsigned int*>(g)), 448.0f);
}

// One warp per row: row amax, g = amax / 448, then the row's blocks.
template <bool BF16>
__global__ void __launch_bounds__(256) k_fp8_quantize_rows(const void* x, int64_t rows, int64_t cols, float* gout,
                                                           uint8_t* q) {
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
        const float g = __fdiv_rn(m, 448.0f);
        if (lane == 0) gout[r] = g;
        for (int64_t b = lane; b < nb; b += 32) {
            float v[16];
            load_block16<BF16>(x, r * nb + b, v);
            reinterpret_cast<uint4*>(q)[r * nb + b] = fp8_block16(v, g);
        }
    }
}

// One warp per token row: the unit-weight RMS norm of the pre-normed block
// (the same arithmetic as the other kernels' norm) into dst.
__global__ void __launch_bounds__(256) k_fp8_rmsnorm_rows(const uint16_t* src, int T, int K, float eps,
                                                          uint16_t* dst) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp < T) warp_rmsnorm_row(src + (size_t)warp * K, dst + (size_t)warp * K, K, eps);
}

// D += A(16 x 32, e4m3, row) * B(32 x 8, e4m3, col), FP32 accumulate.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct Fp8GemvArgs {
    const uint8_t* w;      // [n][K] E4M3
    const float* gw;       // [1] per-tensor scale
    int n, K;              // K % 64 == 0
    const uint8_t* xq;     // [T][K] E4M3 activation rows
    const float* gx;       // [T] their scales
    int T;                 // <= 8
    // up: act[t][r] = bf16(relu(u)^2), amax[t] (float bits of the bf16 values)
    uint16_t* act;
    // down: out[t][r] = bf16(y + residual[t][r]) (residual may be null)
    const uint16_t* residual;
    uint16_t* out;
};

template <int KIND>
__global__ void __launch_bounds__(kF8Threads) k_fp8_gemv(const Fp8GemvArgs a) {
    extern __shared__ __align__(16) uint8_t f8_smem[];  // [T][K] activation bytes
    __shared__ float4 part[kF8Warps][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int K = a.K, T = a.T;
    for (int i = threadIdx.x; i < T * K / 16; i += kF8Threads)
        reinterpret_cast<uint4*>(f8_smem)[i] = __ldg(reinterpret_cast<const uint4*>(a.xq) + i);
    __syncthreads();
    const int r0 = 16 * blockIdx.x;
    const uint8_t* wa = a.w + (size_t)(r0 + g) * K + 16 * q;
    const uint8_t* wb = a.w + (size_t)(r0 + g + 8) * K + 16 * q;
    const uint8_t* xb = g < T ? f8_smem + (size_t)g * K + 16 * q : nullptr;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int steps = K >> 6;
#pragma unroll 2
    for (int s = warp; s < steps; s += kF8Warps) {
        const uint4 ua = __ldg(reinterpret_cast<const uint4*>(wa + 64 * s));
        const uint4 ub = __ldg(reinterpret_cast<const uint4*>(wb + 64 * s));
        const uint4 bx = xb ? *reinterpret_cast<const uint4*>(xb + 64 * s) : make_uint4(0, 0, 0, 0);
        mma_e4m3_16832(acc, ua.x, ub.x, ua.y, ub.y, bx.x, bx.y);
        mma_e4m3_16832(acc, ua.z, ub.z, ua.w, ub.w, bx.z, bx.w);
    }
    part[warp][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    __syncthreads();
    if (warp != 0) return;
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < kF8Warps; ++w) {  // in warp order
        const float4 p = part[w][lane];
        d[0] = __fadd_rn(d[0], p.x);
        d[1] = __fadd_rn(d[1], p.y);
        d[2] = __fadd_rn(d[2], p.z);
        d[3] = __fadd_rn(d[3], p.w);
    }
    const float gw = __ldg(a.gw);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int t = 2 * q + (v & 1), r = r0 + g + 8 * (v >> 1);
        if (t >= T) continue;
        const float y = __fmul_rn(__fmul_rn(d[v], gw), __ldg(a.gx + t));
        if (KIND == kGroupedUp) {
            const float rl = fmaxf(y, 0.0f);
            const __nv_bfloat16 b = __float2bfloat16_rn(__fmul_rn(rl, rl));
            a.act[(size_t)t * a.n + r] = *reinterpret_cast<const uint16_t*>(&b);
        } else {
            const float res = a.residual ? __uint_as_float(static_cast<uint32_t>(a.residual[(size_t)t * a.n + r]) << 16)
                                         : 0.0f;
            const __nv_bfloat16 b = __float2bfloat16_rn(__fadd_rn(y, res));
            a.out[(size_t)t * a.n + r] = *reinterpret_cast<const uint16_t*>(&b);
        }
    }
}

}  // namespace nvfp4moe
