// lm_head.cuh - lm_head_gemv: NVFP4 weight-only lm_head ("Let's optimize
// Nemotron 3.5 Lightning - a worklog", Step 4: the 131072 x 2688 vocabulary
// matrix read once per step; "nemotron35-w4a4-v13" card, precision table:
// lm_head NVFP4 weight-only W4A16).
//
// A pure HBM stream of the weight matrix: persistent CTAs (two per SM when
// half an SM's shared memory holds three stages besides the token rows: one
// or two tokens at the pages' width) each take a contiguous range of 16-row
// tiles; one producer thread stages them with bulk TMA copies (the first
// ring-full before waiting on the previous kernel), the twelve consumer warps
// run the tensor-core tile with up to 8 token columns (bf16 activations,
// RMS-normalised when asked, converted once per CTA to f16). The FP4 -> f16
// conversion, not the copy, sets the pace, so two CTAs per SM give it more
// warps.
#pragma once

#include "gemv_tile.cuh"

namespace nvfp4moe {

constexpr int kLmMaxT = 8;
constexpr int kLmStaticSmem = 12288;  // the kernel's static shared memory, rounded up

struct LmArgs {
    const uint8_t* codes;   // [V][H/2]
    const uint8_t* scales;  // [V][H/16]
    const float* global;    // [1]
    int64_t V;
    int H;
    const uint16_t* hidden;  // [T][H]
    float rms_eps;           // > 0: logits of RMSNorm(hidden)
    int T;                   // <= 8 per launch
    float* logits;           // [T][ld]
    int64_t ld;
    int ring_bytes;          // shared memory for the staging ring; B rows follow it
    int groups;              // consumer warp groups (a divisor of the stage count)
};

__global__ void __launch_bounds__(kThreads, 2) k_lm_head(const LmArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Ring ring;
    __shared__ const uint16_t* srcs[kLmMaxT];
    __shared__ float gx[kLmMaxT];            // per token: the W4A16 row prescale 2^e
    __shared__ unsigned int red[kLmMaxT];    // per token: the row amax

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stage_bytes = 9 * a.H;
    const int nst = min(kMaxStages, a.ring_bytes / stage_bytes);
    const int ngr = a.groups >= 1 && nst % a.groups == 0 ? a.groups : nst;
    ring_init(ring, nst, ngr);
    pdl_trigger();
    __syncthreads();

    const int64_t N = a.V >> 4;
    const int64_t ib = N * blockIdx.x / gridDim.x, ie = N * (blockIdx.x + 1) / gridDim.x;
    const int n = static_cast<int>(ie - ib);
    uint8_t* ring_base = smem;
    __half* xb = reinterpret_cast<__half*>(smem + a.ring_bytes);             // [T][H] f16
    uint16_t* xn = reinterpret_cast<uint16_t*>(xb + (size_t)a.T * a.H);  // [T][H] bf16

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            // the weights do not depend on the previous kernel: a ring-full is
            // issued before waiting on it
            const uint32_t cbytes = 16u * (uint32_t)(a.H >> 1), sbytes = 16u * (uint32_t)(a.H >> 4);
            const uint8_t* cw = a.codes + 16 * ib * (a.H >> 1);
            const uint8_t* sw = a.scales + 16 * ib * (a.H >> 4);
            FillCursor f = fill_cursor(0, nst);
            for (int li = 0; li < n; ++li) {
                if (li == nst) pdl_wait();
                if (!ring_fill(ring, ring_base, stage_bytes, nst, f, cw, sw, a.H)) break;
                cw += cbytes;
                sw += sbytes;
            }
        }
        pdl_wait();
    } else {
        pdl_wait();
        if (warp < a.T) {
            if (a.rms_eps > 0.0f)
                warp_rmsnorm_row(a.hidden + (size_t)warp * a.H, xn + (size_t)warp * a.H, a.H, a.rms_eps);
            else
                warp_copy_row(a.hidden + (size_t)warp * a.H, xn + (size_t)warp * a.H, a.H);
        }
        if (threadIdx.x < a.T) srcs[threadIdx.x] = xn + (size_t)threadIdx.x * a.H;
        consumer_bar();
        prepare_b_rows<false, false>(srcs, a.T, a.H, xb, gx, red);
        const float gw = __ldg(a.global);
        const int g = lane >> 2, q = lane & 3;
        const __half* bcol = g < a.T ? xb + (size_t)g * a.H : nullptr;
        GroupCursor cur = group_cursor(nst, ngr, a.H, a.H);
        for (; cur.li < n; cursor_next(cur)) {
            float acc[4];
            bool ok;
            const bool lead = group_tile(ring, cur, ring_base, stage_bytes, a.H, bcol, acc, ok);
            if (!ok) break;
            if (!lead) continue;
            const int64_t row0 = 16 * (ib + cur.li);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int t = 2 * q + (v & 1);
                if (t < a.T) a.logits[(size_t)t * a.ld + row0 + g + 8 * (v >> 1)] = __fmul_rn(acc[v], __fmul_rn(gw, gx[t]));
            }
        }
    }
    __syncthreads();
    ring_drain(ring, nst);
}

}  // namespace nvfp4moe
