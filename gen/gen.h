/*
 * gen.h - seeded synthetic inputs for the NVFP4 MoE decode path.
 *
 * This module is input generation only: it holds none of the method's
 * arithmetic (no quantisation, routing or GEMV). It is compiled twice, once by
 * gcc for the host (gen_host.c) and once by nvcc for the device (gen_cuda.cu),
 * and both builds must produce bit-identical values, so that the CPU oracle and
 * the CUDA path can be fed the same tensors without copying them.
 *
 * Generator: Philox4x32-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11),
 * written from its published definition (two 32x32->64 multiplies per round,
 * Weyl key schedule, ten rounds).
 *
 * Normal variates: Marsaglia's polar method on pairs of Philox outputs. Every
 * floating-point step is a single IEEE-754 binary32 operation (+, -, *, /,
 * sqrt, int->float conversion), each correctly rounded, with no fused
 * multiply-add; the logarithm is computed here from those operations alone
 * (exponent split + atanh series), never from a math library, so that the host
 * and the device agree to the last bit. Builds must disable FMA contraction
 * (gcc: -ffp-contract=off; nvcc: -fmad=false).
 *
 * Tensor identity: each synthetic tensor is addressed by (seed, tensor_id)
 * which becomes the Philox key; element i is a pure function of
 * (seed, tensor_id, i), so any slice can be regenerated on either side.
 */
#ifndef NVFP4MOE_GEN_H
#define NVFP4MOE_GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define GEN_FN static __host__ __device__ __forceinline__
#else
#define GEN_FN static inline
#endif

/* ---- tensor ids: kind in bits 28..31, layer in 20..27, index in 0..19 ---- */
enum {
    GEN_KIND_ROUTER_W = 1,  /* router gate [E][H], BF16-valued, held as FP32 */
    GEN_KIND_ROUTER_B = 2,  /* e_score_correction_bias [E], FP32 uniform      */
    GEN_KIND_UP = 3,        /* routed up_proj master [I][H] of expert idx     */
    GEN_KIND_DOWN = 4,      /* routed down_proj master [H][I] of expert idx   */
    GEN_KIND_SH_UP = 5,     /* shared expert up_proj master [S][H]            */
    GEN_KIND_SH_DOWN = 6,   /* shared expert down_proj master [H][S]          */
    GEN_KIND_LM_HEAD = 7,   /* lm_head master [V][H]                          */
    GEN_KIND_HIDDEN = 8     /* hidden-state draw z_idx [H]                    */
};

GEN_FN uint32_t gen_tensor_id(uint32_t kind, uint32_t layer, uint32_t index) {
    return (kind << 28) | ((layer & 0xFFu) << 20) | (index & 0xFFFFFu);
}

/* ---- Philox4x32-10 ---- */
GEN_FN void gen_mulhilo32(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

GEN_FN void gen_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                              uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint32_t hi0, lo0, hi1, lo1;
        gen_mulhilo32(0xD2511F53u, c0, &hi0, &lo0);
        gen_mulhilo32(0xCD9E8D57u, c2, &hi1, &lo1);
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* ---- exact float helpers ---- */
GEN_FN uint32_t gen_f2u(float f) {
    union { float f; uint32_t u; } v; v.f = f; return v.u;
}
GEN_FN float gen_u2f(uint32_t u) {
    union { float f; uint32_t u; } v; v.u = u; return v.f;
}

/* Natural log of x in (0, 1], from +,-,*,/ only: x = m * 2^e with
 * m in [sqrt(1/2), sqrt(2)); ln m = 2 atanh(s), s = (m-1)/(m+1), |s| < 0.172,
 * series to s^13 (truncation < 1e-11, well below binary32 resolution). */
GEN_FN float gen_logf(float x) {
    uint32_t b = gen_f2u(x);
    int e = (int)((b >> 23) & 0xFFu) - 127;
    float m = gen_u2f((b & 0x007FFFFFu) | 0x3F800000u); /* [1, 2) */
    if (m > 1.41421356f) { m = m * 0.5f; e = e + 1; }
    float s = (m - 1.0f) / (m + 1.0f);
    float s2 = s * s;
    float p = 1.0f / 13.0f;
    p = p * s2; p = p + 1.0f / 11.0f;
    p = p * s2; p = p + 1.0f / 9.0f;
    p = p * s2; p = p + 1.0f / 7.0f;
    p = p * s2; p = p + 1.0f / 5.0f;
    p = p * s2; p = p + 1.0f / 3.0f;
    p = p * s2; p = p + 1.0f;
    float lm = (s + s) * p;
    float ef = (float)e;
    return ef * 0.693147182f + lm;
}

/* Two standard normal variates for pair index p of tensor (seed, tid).
 * Polar method: candidate (u, v) uniform in [-1, 1)^2, accepted when
 * 0 < s = u^2 + v^2 < 1; then n = (u, v) * sqrt(-2 ln s / s). Up to 16
 * candidates (8 Philox blocks) are tried in a fixed order; the chance that
 * all fail is 2e-11 per pair, and then (0, 0) is returned. */
GEN_FN void gen_normal_pair(uint32_t seed, uint32_t tid, uint64_t p, float* n0, float* n1) {
    const uint32_t key[2] = {seed, tid};
    for (uint32_t a = 0; a < 8; ++a) {
        uint32_t ctr[4] = {(uint32_t)p, (uint32_t)(p >> 32), a, 0x6E6F726Du};
        uint32_t r[4];
        gen_philox4x32_10(ctr, key, r);
        for (int j = 0; j < 2; ++j) {
            float u = (float)(int32_t)r[2 * j] * 4.656612873077392578125e-10f;     /* 2^-31 */
            float v = (float)(int32_t)r[2 * j + 1] * 4.656612873077392578125e-10f;
            float s = u * u + v * v;
            if (s > 0.0f && s < 1.0f) {
                float lg = gen_logf(s);
                float t = (-2.0f * lg) / s;
#if defined(__CUDA_ARCH__)
                float f = __fsqrt_rn(t);
#else
                float f = __builtin_sqrtf(t);
#endif
                *n0 = u * f;
                *n1 = v * f;
                return;
            }
        }
    }
    *n0 = 0.0f;
    *n1 = 0.0f;
}

GEN_FN float gen_normal(uint32_t seed, uint32_t tid, uint64_t i) {
    float a, b;
    gen_normal_pair(seed, tid, i >> 1, &a, &b);
    return (i & 1) ? b : a;
}

/* Uniform in [0, 1) with 24 random bits (exact in binary32). */
GEN_FN float gen_uniform01(uint32_t seed, uint32_t tid, uint64_t i) {
    const uint32_t key[2] = {seed, tid};
    uint64_t blk = i >> 2;
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0x756E6966u, 0u};
    uint32_t r[4];
    gen_philox4x32_10(ctr, key, r);
    return (float)(r[i & 3] >> 8) * 5.9604644775390625e-8f; /* 2^-24 */
}

/* binary32 -> bfloat16 bits, round to nearest even (inputs are finite). */
GEN_FN uint16_t gen_f32_to_bf16(float f) {
    uint32_t u = gen_f2u(f);
    uint32_t rounding = 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)((u + rounding) >> 16);
}

/* sigma * N(0,1), rounded to bf16. */
GEN_FN uint16_t gen_normal_bf16(uint32_t seed, uint32_t tid, uint64_t i, float sigma) {
    return gen_f32_to_bf16(gen_normal(seed, tid, i) * sigma);
}

/* lo + (hi - lo) * U[0,1) in binary32. */
GEN_FN float gen_uniform_f32(uint32_t seed, uint32_t tid, uint64_t i, float lo, float hi) {
    float w = hi - lo;
    return lo + w * gen_uniform01(seed, tid, i);
}

/* Hidden state of token t with pairwise correlation rho between tokens:
 * h_t = sqrt(rho) z_0 + sqrt(1 - rho) z_{t+1}; rho = 0 gives h_t = z_{t+1}.
 * z_j is the normal tensor GEN_KIND_HIDDEN with index j. */
GEN_FN uint16_t gen_hidden_bf16(uint32_t seed, uint32_t layer, uint32_t t, uint64_t i,
                                float sqrt_rho, float sqrt_1m_rho) {
    float zt = gen_normal(seed, gen_tensor_id(GEN_KIND_HIDDEN, layer, t + 1), i);
    if (sqrt_rho == 0.0f) return gen_f32_to_bf16(zt);
    float z0 = gen_normal(seed, gen_tensor_id(GEN_KIND_HIDDEN, layer, 0), i);
    float a = sqrt_rho * z0;
    float b = sqrt_1m_rho * zt;
    return gen_f32_to_bf16(a + b);
}

#endif /* NVFP4MOE_GEN_H */
