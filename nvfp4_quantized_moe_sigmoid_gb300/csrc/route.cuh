// route.cuh - moe_route_topk: sigmoid router with correction bias
// ("NVIDIA-Nemotron-3.5-Lightning-30B-A3B-W4A16" card, "Left at bfloat16":
// the .gate and its fp32 e_score_correction_bias; "Quantization (PTQ + QAD)",
// Precision Recipes: router compute FP32).
//
// Design: one thread-block cluster of 8 CTAs per tile of TT tokens. The gate
// matrix (E x H fp32, 1.38 MB at the pages' shape) is split by expert across
// the 8 CTAs, one warp per expert, so the logits of a token come from 8 SMs
// streaming the gate rows in parallel. Each CTA leaves its logits in shared
// memory; after a hardware cluster barrier, CTA rank 0 reads all of them
// through distributed shared memory and runs the top-k per token in one warp.
// No global scratch and no spin-waits.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace nvfp4moe {

namespace cg = cooperative_groups;

constexpr int kRouteCluster = 8;
constexpr int kRouteWarps = 16;
constexpr int kRouteMaxExpertsPerCta = 32;  // E <= 256

template <int TT>
__global__ void __cluster_dims__(kRouteCluster, 1, 1) __launch_bounds__(kRouteWarps * 32)
    k_route(const uint16_t* __restrict__ hidden, const float* __restrict__ Wg,
            const float* __restrict__ bias, int T, int H, int E, int k, float rms_eps,
            int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t* hs = reinterpret_cast<uint16_t*>(smem_raw);  // [TT][H] bf16
    __shared__ float zs[TT][kRouteMaxExpertsPerCta];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tile = blockIdx.x / kRouteCluster;
    const int t0 = tile * TT;
    const int nt = min(TT, T - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // stage the token tile's hidden rows (bf16) in shared memory, RMS-normalised
    // when rms_eps > 0 (the same warp routine as the expert kernels use)
    if (rms_eps > 0.0f) {
        for (int t = warp; t < nt; t += kRouteWarps)
            warp_rmsnorm_row(hidden + (int64_t)(t0 + t) * H, hs + t * H, H, rms_eps);
    } else {
        const int n16 = nt * H / 8;  // uint4 count (H % 16 == 0)
        const uint4* src = reinterpret_cast<const uint4*>(hidden + (int64_t)t0 * H);
        uint4* dst = reinterpret_cast<uint4*>(hs);
        for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldg(src + i);
    }
    __syncthreads();

    // logits: this CTA owns experts e = rank + 8 * j; warp w takes j = w, w + 16
    for (int j = warp; j * kRouteCluster + rank < E; j += kRouteWarps) {
        const int e = j * kRouteCluster + rank;
        const float4* wr = reinterpret_cast<const float4*>(Wg + (int64_t)e * H);
        float acc[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
        // issue eight 16-byte gate loads per lane before using any of them
        for (int i0 = lane; i0 < H / 4; i0 += 32 * 8) {
            float4 w4[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + 32 * u;
                w4[u] = i < H / 4 ? __ldg(wr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + 32 * u;
                if (i >= H / 4) break;
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    if (t < nt) {
                        const uint2 hv = *reinterpret_cast<const uint2*>(hs + t * H + 4 * i);
                        acc[t] = fmaf(w4[u].x, __uint_as_float(hv.x << 16), acc[t]);
                        acc[t] = fmaf(w4[u].y, __uint_as_float(hv.x & 0xFFFF0000u), acc[t]);
                        acc[t] = fmaf(w4[u].z, __uint_as_float(hv.y << 16), acc[t]);
                        acc[t] = fmaf(w4[u].w, __uint_as_float(hv.y & 0xFFFF0000u), acc[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) zs[t][j] = v;
        }
    }
    cluster.sync();

    if (rank == 0) {
        // top-k: one warp per token; lane l holds experts l, l + 32, ...
        for (int t = warp; t < nt; t += kRouteWarps) {
            constexpr int kPer = 8;  // E <= 256
            float c[kPer], sg[kPer];
            bool taken[kPer];
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const int e = lane + 32 * q;
                taken[q] = true;
                c[q] = -INFINITY;
                sg[q] = 0.0f;
                if (e < E) {
                    const float* zr = cluster.map_shared_rank(&zs[0][0], e % kRouteCluster);
                    const float z = zr[t * kRouteMaxExpertsPerCta + e / kRouteCluster];
                    sg[q] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
                    c[q] = __fadd_rn(sg[q], __ldg(bias + e));
                    taken[q] = false;
                }
            }
            float ssum = 0.0f;
            float selsig = 0.0f;
            int selidx = 0;
            for (int j = 0; j < k; ++j) {
                // lane-local best: larger c, then lower index
                float bc = -INFINITY;
                int be = 0x7FFFFFFF;
                float bs = 0.0f;
#pragma unroll
                for (int q = 0; q < kPer; ++q) {
                    const int e = lane + 32 * q;
                    if (!taken[q] && (c[q] > bc || (c[q] == bc && e < be))) {
                        bc = c[q];
                        be = e;
                        bs = sg[q];
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float oc = __shfl_xor_sync(0xffffffffu, bc, o);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    const float os = __shfl_xor_sync(0xffffffffu, bs, o);
                    if (oc > bc || (oc == bc && oe < be)) {
                        bc = oc;
                        be = oe;
                        bs = os;
                    }
                }
#pragma unroll
                for (int q = 0; q < kPer; ++q)
                    if (lane + 32 * q == be) taken[q] = true;
                ssum = __fadd_rn(ssum, bs);
                if (lane == j) {
                    selidx = be;
                    selsig = bs;
                }
            }
            if (lane < k) {
                topk_idx[(int64_t)(t0 + t) * k + lane] = selidx;
                topk_w[(int64_t)(t0 + t) * k + lane] = __fdiv_rn(selsig, ssum);
            }
        }
    }
    // keep every CTA's shared memory alive until rank 0 has read it
    cluster.sync();
}

}  // namespace nvfp4moe
