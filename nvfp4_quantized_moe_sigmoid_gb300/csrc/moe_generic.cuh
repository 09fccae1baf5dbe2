// moe_generic.cuh - moe_expert_forward for layer shapes whose hidden,
// intermediate or shared width is a multiple of 16 but not of 64 (the NVFP4
// block is 16 elements: "Let's optimize Nemotron 3.5 Lightning - a worklog",
// Step 1; the fast kernels walk 64-k steps). The same arithmetic as the fast
// paths, written plainly for any such width: correct rather than fast.
//
// Per (token t, slot j) - slot k is the shared expert - one CTA:
//   x   = the token's bf16 row (RMS-normalised first when asked)
//   W4A4: x is quantised per row (g = amax / 2688, blocks of 16) and used
//         as its exact E2M1 x E4M3 values times g; W4A16: x as it is
//   u_r = (g_up g_x) sum_k W_up[r][k] x[k]                        (FP32)
//   a_r = bf16(relu(u_r)^2)                  -> act / act_sh (workspace)
// then, once every row of the token's intermediates is written, one CTA per
// (token, slot) again:
//   a'  = a quantised per row as x was (W4A4), or a (W4A16)
//   y_h = (g_dn g_a) sum_r W_dn[h][r] a'[r]   (times the gate for a routed slot)
// and one thread per (token, h):
//   out = bf16(y_shared + sum_j y_j (in slot order) [+ residual])
// Weights are dequantised exactly (E2M1 x E4M3 in FP32) and each product is
// exact; a lane adds its products over whole blocks in k order and the lanes'
// sums meet in an xor-shuffle tree.
#pragma once

#include "common.cuh"

namespace nvfp4moe {

constexpr int kGenThreads = 256;

struct GenArgs {
    const uint8_t* codes;   // routed matrices [E][n][K/2] (up: n = I, K = H; down: n = H, K = I)
    const uint8_t* scales;  // [E][n][K/16]
    const float* global;    // [E]
    const uint8_t* sh_codes;  // shared expert's matrix [n_sh][K_sh/2]
    const uint8_t* sh_scales;
    const float* sh_global;
    int E, n, K, n_sh, K_sh;
    const uint16_t* src;     // up: hidden [T][H]; down: act [T][k][I]
    const uint16_t* src_sh;  // down: act_sh [T][S]
    float rms_eps;           // up only: > 0 normalises the hidden row
    const int32_t* topk_idx;  // [T][k]
    const float* topk_w;      // [T][k]
    int T, k;
    bool w4a4;
    uint16_t* act;      // up: [T][k][I] bf16
    uint16_t* act_sh;   // up: [T][S] bf16
    float* ypart;       // down: [T][k][H], gate included
    float* ysh;         // down: [T][H]
};

// E2M1 code (bit 3 sign, bits 2-1 exponent, bit 0 mantissa) -> value:
// 0 or 0.5 for exponent 0, else (1 + m / 2) 2^(e - 1)
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float v = e == 0 ? 0.5f * static_cast<float>(m) : __uint_as_float(((126u + e) << 23) | (m << 22));
    return (c & 8u) ? -v : v;
}

// One weight row against the activation values xs (shared memory), one warp:
// lane l takes blocks l, l + 32, ...
__device__ __forceinline__ float gen_row_dot(const uint8_t* codes, const uint8_t* scales, const float* xs, int K) {
    const int lane = threadIdx.x & 31;
    float acc = 0.0f;
    for (int b = lane; b < (K >> 4); b += 32) {
        const float s = e4m3_to_float(scales[b]);
        const uint2 c = *reinterpret_cast<const uint2*>(codes + 8 * b);  // 16 codes, low nibble first
        const uint32_t w[2] = {c.x, c.y};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc = __fmaf_rn(__fmul_rn(e2m1_to_float((w[h] >> (4 * i)) & 15u), s), xs[16 * b + 8 * h + i], acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    return acc;
}

// The activation values of a bf16 row (shared memory, K elements) into xs:
// W4A4 quantises the row (returns its global g); W4A16 copies it (returns 1).
__device__ float gen_activation(const uint16_t* row, int K, bool w4a4, float* xs, unsigned int* amax_s) {
    const int tid = threadIdx.x;
    if (!w4a4) {
        for (int i = tid; i < K; i += kGenThreads) xs[i] = bf16_bits_to_float(row[i]);
        __syncthreads();
        return 1.0f;
    }
    if (tid == 0) *amax_s = 0u;
    __syncthreads();
    float m = 0.0f;
    for (int i = tid; i < K; i += kGenThreads) m = fmaxf(m, fabsf(bf16_bits_to_float(row[i])));
    atomicMax(amax_s, __float_as_uint(m));
    __syncthreads();
    const float g = __fdiv_rn(__uint_as_float(*amax_s), 2688.0f);
    for (int b = tid; b < (K >> 4); b += kGenThreads) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = bf16_bits_to_float(row[16 * b + i]);
        const QBlock q = quantize_block16(v, g);
        const float s = e4m3_to_float(q.scale);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t c = ((i < 8 ? q.lo : q.hi) >> (4 * (i & 7))) & 15u;
            xs[16 * b + i] = __fmul_rn(e2m1_to_float(c), s);
        }
    }
    __syncthreads();
    return g;
}

// The expert of slot j of token t (-1: out of range, flagged), or the shared
// expert (slot k).
__device__ __forceinline__ int gen_expert(const GenArgs& a, int t, int j) {
    if (j == a.k) return -2;
    const int e = __ldg(a.topk_idx + (size_t)t * a.k + j);
    if (e < 0 || e >= a.E) {
        if (threadIdx.x == 0) set_dev_error(kErrBadInput);
        return -1;
    }
    return e;
}

// Up: CTA per (t, j); dynamic shared memory: [H] bf16 row, then [H] floats.
__global__ void __launch_bounds__(kGenThreads) k_gen_up(const GenArgs a) {
    extern __shared__ __align__(16) uint8_t gsm[];
    __shared__ unsigned int amax_s;
    const int t = blockIdx.x / (a.k + 1), j = blockIdx.x % (a.k + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = gen_expert(a, t, j);
    if (e == -1) return;
    const int H = a.K;
    uint16_t* row = reinterpret_cast<uint16_t*>(gsm);
    float* xs = reinterpret_cast<float*>(gsm + ((2 * (size_t)H + 15) & ~size_t(15)));
    if (warp == 0) {
        if (a.rms_eps > 0.0f)
            warp_rmsnorm_row(a.src + (size_t)t * H, row, H, a.rms_eps);
        else
            warp_copy_row(a.src + (size_t)t * H, row, H);
    }
    __syncthreads();
    const float gx = gen_activation(row, H, a.w4a4, xs, &amax_s);
    const bool sh = e == -2;
    const int n = sh ? a.n_sh : a.n;
    const float gw = sh ? __ldg(a.sh_global) : __ldg(a.global + e);
    const float f = __fmul_rn(gw, gx);
    for (int r = warp; r < n; r += kGenThreads / 32) {
        const size_t wr = sh ? (size_t)r : (size_t)e * a.n + r;
        const float u = __fmul_rn(gen_row_dot((sh ? a.sh_codes : a.codes) + wr * (H >> 1),
                                              (sh ? a.sh_scales : a.scales) + wr * (H >> 4), xs, H),
                                  f);
        if (lane == 0) {
            const float rl = fmaxf(u, 0.0f);
            const __nv_bfloat16 bv = __float2bfloat16_rn(__fmul_rn(rl, rl));
            const uint16_t bits = *reinterpret_cast<const uint16_t*>(&bv);
            if (sh)
                a.act_sh[(size_t)t * a.n_sh + r] = bits;
            else
                a.act[((size_t)t * a.k + j) * a.n + r] = bits;
        }
    }
}

// Down: CTA per (t, j); dynamic shared memory: [K] floats (K = I, or S for
// the shared expert).
__global__ void __launch_bounds__(kGenThreads) k_gen_down(const GenArgs a) {
    extern __shared__ __align__(16) uint8_t gsm[];
    __shared__ unsigned int amax_s;
    const int t = blockIdx.x / (a.k + 1), j = blockIdx.x % (a.k + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = gen_expert(a, t, j);
    if (e == -1) return;
    const bool sh = e == -2;
    const int K = sh ? a.K_sh : a.K, H = a.n;
    const uint16_t* row = sh ? a.src_sh + (size_t)t * K : a.src + ((size_t)t * a.k + j) * K;
    float* xs = reinterpret_cast<float*>(gsm);
    const float ga = gen_activation(row, K, a.w4a4, xs, &amax_s);
    const float gw = sh ? __ldg(a.sh_global) : __ldg(a.global + e);
    const float f = __fmul_rn(gw, ga);
    const float gate = sh ? 1.0f : __ldg(a.topk_w + (size_t)t * a.k + j);
    for (int h = warp; h < H; h += kGenThreads / 32) {
        const size_t wr = sh ? (size_t)h : (size_t)e * H + h;
        const float y = __fmul_rn(gen_row_dot((sh ? a.sh_codes : a.codes) + wr * (K >> 1),
                                              (sh ? a.sh_scales : a.scales) + wr * (K >> 4), xs, K),
                                  f);
        if (lane == 0) {
            if (sh)
                a.ysh[(size_t)t * H + h] = y;
            else
                a.ypart[((size_t)t * a.k + j) * H + h] = __fmul_rn(gate, y);
        }
    }
}

// out[t][h] = bf16(ysh + ypart[slot 0] + ... + ypart[slot k - 1] [+ residual])
__global__ void __launch_bounds__(kGenThreads) k_gen_combine(const float* __restrict__ ypart,
                                                             const float* __restrict__ ysh, int T, int k, int H,
                                                             const uint16_t* residual, uint16_t* out) {
    const int i = blockIdx.x * kGenThreads + threadIdx.x;
    if (i >= T * H) return;
    const int t = i / H, h = i - t * H;
    float acc = ysh[i];
    for (int j = 0; j < k; ++j) acc = __fadd_rn(acc, ypart[((size_t)t * k + j) * H + h]);
    if (residual) acc = __fadd_rn(acc, bf16_bits_to_float(residual[i]));
    const __nv_bfloat16 ob = __float2bfloat16_rn(acc);
    out[i] = *reinterpret_cast<const uint16_t*>(&ob);
}

// The lm_head (weight-only NVFP4, bf16 activations) for a hidden width that
// is a multiple of 16 but not of 64: logits[t][v] = g_w sum_k W[v][k] x_t[k]
// (x_t RMS-normalised first when asked). Grid (V / 64 rows, T / 8 tokens):
// a CTA holds up to 8 token rows as FP32 in shared memory, a warp takes
// vocabulary rows and decodes each weight block once for all its tokens.
constexpr int kGenLmTok = 8, kGenLmRows = 64;

__global__ void __launch_bounds__(kGenThreads) k_gen_lm_head(const uint8_t* __restrict__ codes,
                                                             const uint8_t* __restrict__ scales,
                                                             const float* __restrict__ global, int V, int H,
                                                             const uint16_t* __restrict__ hidden, int T,
                                                             float rms_eps, float* __restrict__ logits,
                                                             int64_t ld) {
    extern __shared__ __align__(16) uint8_t gsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * kGenLmTok, nt = min(kGenLmTok, T - t0);
    uint16_t* rows = reinterpret_cast<uint16_t*>(gsm);                               // [8][H] bf16
    float* xs = reinterpret_cast<float*>(gsm + (size_t)kGenLmTok * H * 2);           // [8][H]
    if (warp < nt) {
        if (rms_eps > 0.0f)
            warp_rmsnorm_row(hidden + (size_t)(t0 + warp) * H, rows + (size_t)warp * H, H, rms_eps);
        else
            warp_copy_row(hidden + (size_t)(t0 + warp) * H, rows + (size_t)warp * H, H);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nt * H; i += kGenThreads) xs[i] = bf16_bits_to_float(rows[i]);
    __syncthreads();
    const float gw = __ldg(global);
    const int v1 = min(V, (blockIdx.x + 1) * kGenLmRows);
    for (int v = blockIdx.x * kGenLmRows + warp; v < v1; v += kGenThreads / 32) {
        const uint8_t* cr = codes + (size_t)v * (H >> 1);
        const uint8_t* sr = scales + (size_t)v * (H >> 4);
        float acc[kGenLmTok];
#pragma unroll
        for (int t = 0; t < kGenLmTok; ++t) acc[t] = 0.0f;
        for (int b = lane; b < (H >> 4); b += 32) {
            const float s = e4m3_to_float(sr[b]);
            const uint2 c = *reinterpret_cast<const uint2*>(cr + 8 * b);
            const uint32_t w2[2] = {c.x, c.y};
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float wv = __fmul_rn(e2m1_to_float((w2[i >> 3] >> (4 * (i & 7))) & 15u), s);
#pragma unroll
                for (int t = 0; t < kGenLmTok; ++t)
                    if (t < nt) acc[t] = __fmaf_rn(wv, xs[(size_t)t * H + 16 * b + i], acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < kGenLmTok; ++t) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xffffffffu, acc[t], o));
            if (lane == 0 && t < nt) logits[(size_t)(t0 + t) * ld + v] = __fmul_rn(acc[t], gw);
        }
    }
}

}  // namespace nvfp4moe
