// route.cuh - moe_route_topk: sigmoid router with correction bias
// ("NVIDIA-Nemotron-3.5-Lightning-30B-A3B-W4A16" card, "Left at bfloat16":
// the .gate and its fp32 e_score_correction_bias; "Quantization (PTQ + QAD)",
// Precision Recipes: router compute FP32).
//
// Design: one thread-block cluster of 8 CTAs per tile of TT tokens. The gate
// matrix (E x H fp32, 1.38 MB at the pages' shape) is split by expert across
// the 8 CTAs, one warp per expert. The gate rows are constant, so each CTA
// stages its rows into shared memory with bulk TMA copies before it waits on
// the kernel that produced the hidden state (programmatic dependent launch);
// when they do not fit, they are read from global memory instead. Each CTA
// leaves its logits in shared memory; after a hardware cluster barrier, CTA
// rank 0 reads all of them through distributed shared memory and runs the
// top-k per token in one warp. No global scratch.
#pragma once

#include <cooperative_groups.h>

#include "moe_decode.cuh"

namespace nvfp4moe {

namespace cg = cooperative_groups;

constexpr int kRouteCluster = 8;
constexpr int kRouteWarps = kConsumerWarps;
constexpr int kRouteMaxExpertsPerCta = 32;  // E <= 256
constexpr int kRouteTile = 8;               // tokens per cluster

// kRouteWarps * 32 threads == kConsumerThreads, so the consumer-barrier
// helpers of the expert kernels serve this kernel's whole CTA too.
static_assert(kRouteWarps * 32 == kConsumerThreads, "route CTA size must match the consumer barrier");

template <int TT>
__global__ void __cluster_dims__(kRouteCluster, 1, 1) __launch_bounds__(kRouteWarps * 32)
    k_route(const uint16_t* __restrict__ hidden, const float* __restrict__ Wg,
            const float* __restrict__ bias, int T, int H, int E, int k, float rms_eps,
            int stage_w, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
            DecodePlan* __restrict__ plan_out, __half* __restrict__ xq_out, float* __restrict__ gx_out,
            int w4a4) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t* hs = reinterpret_cast<uint16_t*>(smem_raw);             // [TT][H] bf16
    float* wsm = reinterpret_cast<float*>(smem_raw + (size_t)TT * H * 2);  // [nj][H] gate rows
    __shared__ float zs[TT][kRouteMaxExpertsPerCta];
    __shared__ __align__(8) uint64_t wbar;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tile = blockIdx.x / kRouteCluster;
    const int t0 = tile * TT;
    const int nt = min(TT, T - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nj = (E - rank + kRouteCluster - 1) / kRouteCluster;  // experts of this CTA

    if (threadIdx.x == 0) {
        mbar_init(&wbar, 1);
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < TT * kRouteMaxExpertsPerCta; i += blockDim.x) (&zs[0][0])[i] = 0.0f;
    pdl_trigger();
    __syncthreads();
    if (stage_w && threadIdx.x == 0) {
        mbar_arrive_expect_tx(&wbar, (uint32_t)(nj * H * 4));
        for (int j = 0; j < nj; ++j)
            bulk_g2s(wsm + (size_t)j * H, Wg + (int64_t)(j * kRouteCluster + rank) * H, (uint32_t)(H * 4), &wbar);
    }
    pdl_wait();

    // stage the token tile's hidden rows (bf16) in shared memory, RMS-normalised
    // when rms_eps > 0 (the same warp routine as the expert kernels use)
    for (int t = warp; t < nt; t += kRouteWarps) {
        if (rms_eps > 0.0f)
            warp_rmsnorm_row(hidden + (int64_t)(t0 + t) * H, hs + t * H, H, rms_eps);
        else
            warp_copy_row(hidden + (int64_t)(t0 + t) * H, hs + t * H, H);
    }
    __syncthreads();
    bool wok = true;
    if (stage_w) {
        wok = __all_sync(0xffffffffu, mbar_wait_bounded(&wbar, 0));
        if (!wok && lane == 0) set_dev_error(kErrWaitFull);
    }

    // logits: this CTA owns experts e = rank + 8 * j; warp w takes j = w, w + 16
    for (int j = warp; j * kRouteCluster + rank < E && wok; j += kRouteWarps) {
        const int e = j * kRouteCluster + rank;
        const float4* wr = stage_w ? reinterpret_cast<const float4*>(wsm + (size_t)j * H)
                                   : reinterpret_cast<const float4*>(Wg + (int64_t)e * H);
        float acc[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
        // issue eight 16-byte gate loads per lane before using any of them
        for (int i0 = lane; i0 < H / 4; i0 += 32 * 8) {
            float4 w4[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + 32 * u;
                w4[u] = i < H / 4 ? (stage_w ? wr[i] : __ldg(wr + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
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
                    c[q] = __fadd_rn(sg[q], __ldg(bias + e));  // constant weights
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
        if (plan_out != nullptr) {
            // planning mode (one cluster holds every token): the step plan and
            // the up kernel's B rows, prepared once for all of its CTAs
            __shared__ DecodePlan plan;
            __shared__ unsigned int red[kRouteTile];
            __shared__ const uint16_t* srcs[kRouteTile];
            __threadfence();
            __syncthreads();
            build_plan(plan, topk_idx, topk_w, T, k, E);
            {
                const uint32_t* src = reinterpret_cast<const uint32_t*>(&plan);
                uint32_t* dst = reinterpret_cast<uint32_t*>(plan_out);
                for (int i = threadIdx.x; i < (int)(sizeof(DecodePlan) / 4); i += blockDim.x) dst[i] = src[i];
            }
            if (threadIdx.x < nt) srcs[threadIdx.x] = hs + threadIdx.x * H;
            __syncthreads();
            if (w4a4) prepare_b_rows<true, false>(srcs, nt, H, xq_out, gx_out, red);
            else prepare_b_rows<false, false>(srcs, nt, H, xq_out, gx_out, red);
        }
    }
    // keep every CTA's shared memory alive until rank 0 has read it, and do not
    // exit while a gate-row copy could still be landing
    cluster.sync();
    if (stage_w && !wok && threadIdx.x == 0 && !mbar_wait_bounded(&wbar, 0)) set_dev_error(kErrWaitDrain);
}

// ---------------------------------------------------------------- many tokens
// The router for prefill and many concurrent tokens: one CTA per 8 tokens and
// every expert, in one wave of T / 8 CTAs. The gate matrix (1.4 MB at the
// pages' shape) stays in L2 after the first CTAs have read it, and every CTA
// streams it from there; each warp takes two experts at a time so that every
// hidden value it loads from shared memory serves two dot products. Logits,
// sigmoid, biased top-k and the renormalised gates as in k_route (every
// summation order agrees with the oracle within the binary32 bound).
constexpr int kRouteRowsTile = 8;

__global__ void __launch_bounds__(kConsumerThreads) k_route_rows(
    const uint16_t* __restrict__ hidden, const float* __restrict__ Wg, const float* __restrict__ bias, int T, int H,
    int E, int k, float rms_eps, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
    extern __shared__ __align__(16) unsigned char rr_smem[];
    uint16_t* hs = reinterpret_cast<uint16_t*>(rr_smem);  // [8][H] bf16 (normalised)
    __shared__ float zs[kRouteRowsTile][256];
    const int t0 = blockIdx.x * kRouteRowsTile;
    const int nt = min(kRouteRowsTile, T - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    for (int t = warp; t < nt; t += kConsumerWarps) {
        if (rms_eps > 0.0f)
            warp_rmsnorm_row(hidden + (int64_t)(t0 + t) * H, hs + (size_t)t * H, H, rms_eps);
        else
            warp_copy_row(hidden + (int64_t)(t0 + t) * H, hs + (size_t)t * H, H);
    }
    __syncthreads();
    const int H4 = H >> 2;
    for (int e0 = 2 * warp; e0 < E; e0 += 2 * kConsumerWarps) {
        const bool two = e0 + 1 < E;
        const float4* w0 = reinterpret_cast<const float4*>(Wg + (int64_t)e0 * H);
        const float4* w1 = reinterpret_cast<const float4*>(Wg + (int64_t)(two ? e0 + 1 : e0) * H);
        float a0[kRouteRowsTile], a1[kRouteRowsTile];
#pragma unroll
        for (int t = 0; t < kRouteRowsTile; ++t) a0[t] = a1[t] = 0.0f;
        for (int i0 = lane; i0 < H4; i0 += 32 * 4) {
            float4 x0[4], x1[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + 32 * u;
                x0[u] = i < H4 ? __ldg(w0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                x1[u] = i < H4 ? __ldg(w1 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + 32 * u;
                if (i >= H4) break;
#pragma unroll
                for (int t = 0; t < kRouteRowsTile; ++t) {
                    if (t < nt) {
                        const uint2 hv = *reinterpret_cast<const uint2*>(hs + (size_t)t * H + 4 * i);
                        const float h0 = __uint_as_float(hv.x << 16), h1 = __uint_as_float(hv.x & 0xFFFF0000u);
                        const float h2 = __uint_as_float(hv.y << 16), h3 = __uint_as_float(hv.y & 0xFFFF0000u);
                        a0[t] = fmaf(x0[u].x, h0, a0[t]);
                        a0[t] = fmaf(x0[u].y, h1, a0[t]);
                        a0[t] = fmaf(x0[u].z, h2, a0[t]);
                        a0[t] = fmaf(x0[u].w, h3, a0[t]);
                        a1[t] = fmaf(x1[u].x, h0, a1[t]);
                        a1[t] = fmaf(x1[u].y, h1, a1[t]);
                        a1[t] = fmaf(x1[u].z, h2, a1[t]);
                        a1[t] = fmaf(x1[u].w, h3, a1[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kRouteRowsTile; ++t) {
            float v0 = a0[t], v1 = a1[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                v1 += __shfl_xor_sync(0xffffffffu, v1, o);
            }
            if (lane == 0 && t < nt) {
                zs[t][e0] = v0;
                if (two) zs[t][e0 + 1] = v1;
            }
        }
    }
    __syncthreads();
    // top-k: one warp per token; lane l holds experts l, l + 32, ...
    for (int t = warp; t < nt; t += kConsumerWarps) {
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
                sg[q] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-zs[t][e])));
                c[q] = __fadd_rn(sg[q], __ldg(bias + e));
                taken[q] = false;
            }
        }
        float ssum = 0.0f, selsig = 0.0f;
        int selidx = 0;
        for (int j = 0; j < k; ++j) {
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

}  // namespace nvfp4moe
