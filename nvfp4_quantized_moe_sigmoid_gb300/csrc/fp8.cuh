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
// decoded. Two launches per 8 tokens (up, then down). Each CTA first
// quantises the token rows its GEMV needs into shared memory (warp t: row t,
// after the RMS norm for the up projection), then owns one 16-row tile of W;
// its eight warps split the reduction by 64-k steps (warp w takes steps w,
// w + 8, ...) and their accumulators are added in warp order. In a step,
// lane (g, q) loads 16 contiguous weight bytes of rows g and g + 8 and the
// same 16 bytes of the activation row of token g, so the reduction index is
// permuted alike for both operands. Up to 8 tokens are the MMA's columns.
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
    const uint16_t* src;   // [T][K] bf16 activation rows, quantised per row in the prologue
    float rms_eps;         // > 0: RMS-normalise the rows first
    int T;                 // <= 8
    // up: act[t][r] = bf16(relu(u)^2)
    uint16_t* act;
    // down: out[t][r] = bf16(y + residual[t][r]) (residual may be null)
    const uint16_t* residual;
    uint16_t* out;
};

// 16 bf16 values from shared or global memory (16-byte aligned)
__device__ __forceinline__ void bf16x16(const uint16_t* p, float (&v)[16]) {
    const uint4 x = reinterpret_cast<const uint4*>(p)[0], y = reinterpret_cast<const uint4*>(p)[1];
    const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// A warp's weight steps held in registers at once (K <= 64 * 8 * kF8Steps in
// one pass; longer rows take several passes).
constexpr int kF8Steps = 8;

// dynamic shared memory: [T][K] E4M3 rows
template <int KIND>
__global__ void __launch_bounds__(kF8Threads) k_fp8_gemv(const Fp8GemvArgs a) {
    extern __shared__ __align__(16) uint8_t f8_smem[];
    __shared__ float4 part[kF8Warps][32];
    __shared__ float gx_s[kF8MaxT], inv_s[kF8MaxT];
    __shared__ float red[2][kF8Warps][kF8MaxT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int K = a.K, T = a.T;
    const int r0 = 16 * blockIdx.x;
    const uint8_t* wa = a.w + (size_t)(r0 + g) * K + 16 * q;
    const uint8_t* wb = a.w + (size_t)(r0 + g + 8) * K + 16 * q;
    const int steps = K >> 6;
    // the first pass of weight loads is issued before the activation rows are
    // prepared: the weights do not depend on them
    uint4 ua[kF8Steps], ub[kF8Steps];
#pragma unroll
    for (int i = 0; i < kF8Steps; ++i) {
        const int s = warp + kF8Warps * i;
        if (s < steps) {
            ua[i] = __ldg(reinterpret_cast<const uint4*>(wa + 64 * s));
            ub[i] = __ldg(reinterpret_cast<const uint4*>(wb + 64 * s));
        }
    }
    // the rows (and, for the down projection, the up kernel's output) are an
    // earlier kernel's: with programmatic dependent launch this kernel may
    // start, and its weight loads run, while that kernel finishes
    pdl_trigger();
    pdl_wait();
    // token rows -> E4M3 in shared memory, all threads on all rows at once:
    // per row the sum of squares and the amax (in warp order), then (the RMS
    // norm: y = bf16(x inv), whose amax is bf16(amax(x) inv) as rounding is
    // monotonic) the row scale and the codes
    const bool norm = a.rms_eps > 0.0f;
    const int nb = K / 16;
    {
        float ss[kF8MaxT], mx[kF8MaxT];
#pragma unroll
        for (int t = 0; t < kF8MaxT; ++t) ss[t] = mx[t] = 0.0f;
        for (int b = threadIdx.x; b < nb; b += kF8Threads) {
#pragma unroll
            for (int t = 0; t < kF8MaxT; ++t) {
                if (t >= T) break;
                float v[16];
                bf16x16(a.src + (size_t)t * K + 16 * b, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    ss[t] = __fmaf_rn(v[i], v[i], ss[t]);
                    mx[t] = fmaxf(mx[t], fabsf(v[i]));
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kF8MaxT; ++t) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ss[t] = __fadd_rn(ss[t], __shfl_xor_sync(0xffffffffu, ss[t], o));
                mx[t] = fmaxf(mx[t], __shfl_xor_sync(0xffffffffu, mx[t], o));
            }
            if (lane == 0) {
                red[0][warp][t] = ss[t];
                red[1][warp][t] = mx[t];
            }
        }
    }
    __syncthreads();
    if (threadIdx.x < T) {
        const int t = threadIdx.x;
        float ss = 0.0f, m = 0.0f;
        for (int w = 0; w < kF8Warps; ++w) {  // in warp order
            ss = __fadd_rn(ss, red[0][w][t]);
            m = fmaxf(m, red[1][w][t]);
        }
        const float inv = norm ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), a.rms_eps)))
                               : 1.0f;
        const float amax = norm ? __bfloat162float(__float2bfloat16_rn(__fmul_rn(m, inv))) : m;
        inv_s[t] = inv;
        gx_s[t] = __fdiv_rn(amax, 448.0f);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += kF8Threads) {
#pragma unroll
        for (int t = 0; t < kF8MaxT; ++t) {
            if (t >= T) break;
            float v[16];
            bf16x16(a.src + (size_t)t * K + 16 * b, v);
            if (norm) {
                const float inv = inv_s[t];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(v[i], inv)));
            }
            reinterpret_cast<uint4*>(f8_smem + (size_t)t * K)[b] = fp8_block16(v, gx_s[t]);
        }
    }
    __syncthreads();
    const uint8_t* xb = g < T ? f8_smem + (size_t)g * K + 16 * q : nullptr;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int p0 = 0; p0 < steps; p0 += kF8Warps * kF8Steps) {
        if (p0 > 0) {  // the next pass of weight loads
#pragma unroll
            for (int i = 0; i < kF8Steps; ++i) {
                const int s = p0 + warp + kF8Warps * i;
                if (s < steps) {
                    ua[i] = __ldg(reinterpret_cast<const uint4*>(wa + 64 * s));
                    ub[i] = __ldg(reinterpret_cast<const uint4*>(wb + 64 * s));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kF8Steps; ++i) {
            const int s = p0 + warp + kF8Warps * i;
            if (s < steps) {
                const uint4 bx = xb ? *reinterpret_cast<const uint4*>(xb + 64 * s) : make_uint4(0, 0, 0, 0);
                mma_e4m3_16832(acc, ua[i].x, ub[i].x, ua[i].y, ub[i].y, bx.x, bx.y);
                mma_e4m3_16832(acc, ua[i].z, ub[i].z, ua[i].w, ub[i].w, bx.z, bx.w);
            }
        }
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
        const float y = __fmul_rn(__fmul_rn(d[v], gw), gx_s[t]);
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
