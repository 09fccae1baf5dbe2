/*
 * gen_host.c - host build of the synthetic-input generator (see gen.h).
 * Fills caller-owned host buffers; OpenMP splits the index range only, so the
 * values do not depend on the thread count.
 */
#include "gen.h"

#include <stddef.h>

void gen_fill_normal_bf16(uint16_t* out, int64_t n, uint32_t seed, uint32_t tid, float sigma) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < (n + 1) / 2; ++p) {
        float a, b;
        gen_normal_pair(seed, tid, (uint64_t)p, &a, &b);
        out[2 * p] = gen_f32_to_bf16(a * sigma);
        if (2 * p + 1 < n) out[2 * p + 1] = gen_f32_to_bf16(b * sigma);
    }
}

/* elements [i0, i0+n) of the same tensor, for regenerating a slice. */
void gen_fill_normal_bf16_range(uint16_t* out, int64_t i0, int64_t n, uint32_t seed, uint32_t tid,
                                float sigma) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = gen_normal_bf16(seed, tid, (uint64_t)(i0 + j), sigma);
}

void gen_fill_normal_f32(float* out, int64_t n, uint32_t seed, uint32_t tid) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = gen_normal(seed, tid, (uint64_t)i);
}

void gen_fill_uniform_f32(float* out, int64_t n, uint32_t seed, uint32_t tid, float lo, float hi) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = gen_uniform_f32(seed, tid, (uint64_t)i, lo, hi);
}

/* rows [t0, t0+nt) of the hidden-state matrix [T][H] (bf16). */
void gen_fill_hidden_bf16(uint16_t* out, int32_t t0, int32_t nt, int64_t H, uint32_t seed,
                          uint32_t layer, float sqrt_rho, float sqrt_1m_rho) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < (int64_t)nt * H; ++j) {
        int64_t t = j / H, i = j % H;
        out[j] = gen_hidden_bf16(seed, layer, (uint32_t)(t0 + t), (uint64_t)i, sqrt_rho, sqrt_1m_rho);
    }
}

void gen_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    gen_philox4x32_10(ctr, key, out);
}

float gen_log_test(float x) { return gen_logf(x); }

uint32_t gen_tid(uint32_t kind, uint32_t layer, uint32_t index) {
    return gen_tensor_id(kind, layer, index);
}
