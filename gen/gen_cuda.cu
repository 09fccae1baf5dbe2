/*
 * gen_cuda.cu - device build of the synthetic-input generator (see gen.h).
 * Compiled with -fmad=false so that every binary32 step matches the host
 * build bit for bit. Grid-stride kernels; the launchers are stream-ordered and
 * return cudaError_t as int.
 */
#include <cuda_runtime.h>

#include "gen.h"

namespace {

__global__ void k_normal_bf16(uint16_t* out, int64_t n, uint32_t seed, uint32_t tid, float sigma) {
    int64_t np = (n + 1) / 2;
    for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < np;
         p += (int64_t)gridDim.x * blockDim.x) {
        float a, b;
        gen_normal_pair(seed, tid, (uint64_t)p, &a, &b);
        out[2 * p] = gen_f32_to_bf16(a * sigma);
        if (2 * p + 1 < n) out[2 * p + 1] = gen_f32_to_bf16(b * sigma);
    }
}

__global__ void k_bf16_to_f32(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = gen_u2f((uint32_t)in[i] << 16);
}

__global__ void k_uniform_f32(float* out, int64_t n, uint32_t seed, uint32_t tid, float lo, float hi) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = gen_uniform_f32(seed, tid, (uint64_t)i, lo, hi);
}

__global__ void k_hidden_bf16(uint16_t* out, int32_t t0, int32_t nt, int64_t H, uint32_t seed,
                              uint32_t layer, float sr, float s1r) {
    int64_t n = (int64_t)nt * H;
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        int64_t t = j / H, i = j % H;
        out[j] = gen_hidden_bf16(seed, layer, (uint32_t)(t0 + t), (uint64_t)i, sr, s1r);
    }
}

int grid_for(int64_t n) {
    int64_t g = (n + 255) / 256;
    if (g > 152 * 32) g = 152 * 32;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace

extern "C" {

int gen_dev_normal_bf16(uint16_t* out, int64_t n, uint32_t seed, uint32_t tid, float sigma,
                        cudaStream_t s) {
    if (n <= 0) return 0;
    k_normal_bf16<<<grid_for((n + 1) / 2), 256, 0, s>>>(out, n, seed, tid, sigma);
    return (int)cudaGetLastError();
}

/* BF16-valued FP32 tensor: sigma*N(0,1) rounded to bf16, then widened. `tmp`
 * holds n bf16 values of scratch supplied by the caller. */
int gen_dev_normal_bf16_as_f32(float* out, uint16_t* tmp, int64_t n, uint32_t seed, uint32_t tid,
                               float sigma, cudaStream_t s) {
    if (n <= 0) return 0;
    k_normal_bf16<<<grid_for((n + 1) / 2), 256, 0, s>>>(tmp, n, seed, tid, sigma);
    k_bf16_to_f32<<<grid_for(n), 256, 0, s>>>(tmp, out, n);
    return (int)cudaGetLastError();
}

int gen_dev_uniform_f32(float* out, int64_t n, uint32_t seed, uint32_t tid, float lo, float hi,
                        cudaStream_t s) {
    if (n <= 0) return 0;
    k_uniform_f32<<<grid_for(n), 256, 0, s>>>(out, n, seed, tid, lo, hi);
    return (int)cudaGetLastError();
}

int gen_dev_hidden_bf16(uint16_t* out, int32_t t0, int32_t nt, int64_t H, uint32_t seed,
                        uint32_t layer, float sqrt_rho, float sqrt_1m_rho, cudaStream_t s) {
    int64_t n = (int64_t)nt * H;
    if (n <= 0) return 0;
    k_hidden_bf16<<<grid_for(n), 256, 0, s>>>(out, t0, nt, H, seed, layer, sqrt_rho, sqrt_1m_rho);
    return (int)cudaGetLastError();
}

}  // extern "C"
