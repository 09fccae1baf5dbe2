// moe_decode.cuh - moe_expert_forward for 1..4 tokens (batch-1 decode and the
// 4-token speculative verify of "Let's optimize Nemotron 3.5 Lightning - a
// worklog", Step 5). At this size the layer is a stream of NVFP4 weights
// (worklog, Interlude), so both kernels are persistent HBM streams:
//
//   up kernel   : items = 16-row tiles of every selected expert's up_proj and
//                 of the shared expert's up_proj. Epilogue: relu^2 -> bf16
//                 intermediate rows in the workspace.
//   down kernel : items = 16-row tiles of every selected expert's down_proj
//                 and of the shared expert's down_proj. Epilogue: gate-weighted
//                 FP32 partial rows; the warp that completes a 16-row output
//                 tile (per-tile counter) sums the partials in a fixed order,
//                 adds the residual and writes bf16.
//
// Each CTA takes a contiguous, cost-balanced range of items; one producer
// thread streams the range through a ring of shared-memory stages with bulk
// TMA copies, eight consumer warps run the tensor-core tile (gemv_tile.cuh).
// Experts chosen by several tokens are read once per step: items are per
// unique expert, and the MMA's columns are the tokens.
#pragma once

#include "gemv_tile.cuh"

namespace nvfp4moe {

constexpr int kDecodeMaxT = 4;
constexpr int kDecodeMaxK = 16;
constexpr int kDecodeMaxU = kDecodeMaxT * kDecodeMaxK;

struct DecodePlan {
    int U;                                 // unique experts this step
    int expert[kDecodeMaxU];               // ascending expert ids
    int8_t choice[kDecodeMaxU][kDecodeMaxT];  // j with topk_idx[t][j] == expert, else -1
    float gate[kDecodeMaxU][kDecodeMaxT];  // topk_w[t][j] or 0
    unsigned int bits[8];                  // E <= 256 bitmap
};

// Every CTA builds the same plan from topk_idx (T*k <= 64 entries).
// Expert ids outside [0, E) are dropped (and flagged in the error word).
__device__ __forceinline__ void build_plan(DecodePlan& p, const int32_t* __restrict__ topk_idx,
                                           const float* __restrict__ topk_w, int T, int k, int E) {
    const int tid = threadIdx.x;
    if (tid < 8) p.bits[tid] = 0u;
    for (int i = tid; i < kDecodeMaxU * kDecodeMaxT; i += blockDim.x) {
        (&p.choice[0][0])[i] = -1;
        (&p.gate[0][0])[i] = 0.0f;
    }
    __syncthreads();
    const int P = T * k;
    int e = -1;
    if (tid < P) {
        e = __ldg(topk_idx + tid);
        if (e < 0 || e >= E) {
            if (blockIdx.x == 0) set_dev_error(kErrBadInput);
            e = -1;
        } else {
            atomicOr(&p.bits[e >> 5], 1u << (e & 31));
        }
    }
    __syncthreads();
    if (tid < P && e >= 0) {
        int slot = __popc(p.bits[e >> 5] & ((1u << (e & 31)) - 1u));
        for (int w = 0; w < (e >> 5); ++w) slot += __popc(p.bits[w]);
        p.expert[slot] = e;
        p.choice[slot][tid / k] = static_cast<int8_t>(tid % k);
        p.gate[slot][tid / k] = __ldg(topk_w + tid);
    }
    if (tid == 0) {
        int u = 0;
        for (int w = 0; w < 8; ++w) u += __popc(p.bits[w]);
        p.U = u;
    }
    __syncthreads();
}

struct UpArgs {
    const uint8_t* codes;   // routed up [E][I][H/2]
    const uint8_t* scales;  // [E][I][H/16]
    const float* global;    // [E]
    const uint8_t* sh_codes;
    const uint8_t* sh_scales;
    const float* sh_global;
    int E, H, I, S;
    const uint16_t* hidden;  // [T][H] bf16
    float rms_eps;           // > 0: experts see RMSNorm(hidden)
    const int32_t* topk_idx;
    const float* topk_w;
    int T, k;
    uint16_t* act;     // [T*k][I] bf16
    uint16_t* act_sh;  // [T][S] bf16
    int ring_bytes;    // shared memory for the staging ring; B rows follow it
};

template <bool W4A4>
__global__ void __launch_bounds__(kThreads, 1) k_moe_up_decode(const UpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Ring ring;
    __shared__ DecodePlan plan;
    __shared__ float gx[kDecodeMaxT];
    __shared__ unsigned int red[kDecodeMaxT];
    __shared__ const uint16_t* srcs[kDecodeMaxT];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stage_bytes = 9 * a.H;  // 16 rows x (H/2 code bytes + H/16 scale bytes)
    const int nst = min(kMaxStages, a.ring_bytes / stage_bytes);
    ring_init(ring, nst);
    build_plan(plan, a.topk_idx, a.topk_w, a.T, a.k, a.E);  // contains __syncthreads

    const int RI = a.I >> 4, RS = a.S >> 4;
    const int U = plan.U;
    const int64_t N = (int64_t)U * RI + RS;
    const int64_t ib = N * blockIdx.x / gridDim.x, ie = N * (blockIdx.x + 1) / gridDim.x;
    const int n = static_cast<int>(ie - ib);
    uint8_t* ring_base = smem;
    __half* xb = reinterpret_cast<__half*>(smem + a.ring_bytes);  // [T][H] f16 B operand
    uint16_t* xn = reinterpret_cast<uint16_t*>(xb + (size_t)a.T * a.H);  // [T][H] normalised bf16

    auto item = [&](int64_t i, const uint8_t*& c, const uint8_t*& s) {
        if (i < (int64_t)U * RI) {
            const int u = static_cast<int>(i / RI), r = static_cast<int>(i % RI);
            const int64_t row = (int64_t)plan.expert[u] * a.I + 16 * r;
            c = a.codes + row * (a.H >> 1);
            s = a.scales + row * (a.H >> 4);
        } else {
            const int64_t row = 16 * (i - (int64_t)U * RI);
            c = a.sh_codes + row * (a.H >> 1);
            s = a.sh_scales + row * (a.H >> 4);
        }
    };

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int li = 0; li < n; ++li) {
                const uint8_t *c, *s;
                item(ib + li, c, s);
                if (!ring_fill(ring, ring_base, stage_bytes, nst, li, c, s, a.H)) break;
            }
        }
    } else {
        if (a.rms_eps > 0.0f) {
            if (warp < a.T) warp_rmsnorm_row(a.hidden + (size_t)warp * a.H, xn + (size_t)warp * a.H, a.H, a.rms_eps);
            if (threadIdx.x < a.T) srcs[threadIdx.x] = xn + (size_t)threadIdx.x * a.H;
        } else {
            if (threadIdx.x < a.T) srcs[threadIdx.x] = a.hidden + (size_t)threadIdx.x * a.H;
        }
        consumer_bar();
        prepare_b_rows<W4A4>(srcs, a.T, a.H, xb, gx, red);
        const int g = lane >> 2, q = lane & 3;
        const __half* bcol = g < a.T ? xb + (size_t)g * a.H : nullptr;
        for (int li = warp; warp < nst && li < n; li += nst) {
            if (!ring_acquire(ring, nst, li)) break;
            const uint8_t* st = ring_base + (size_t)(li % nst) * stage_bytes;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            tile_mma_16x8(st, st + 16 * (a.H >> 1), a.H, bcol, acc);
            ring_release(ring, nst, li);
            const int64_t i = ib + li;
            const bool routed = i < (int64_t)U * RI;
            const int u = routed ? static_cast<int>(i / RI) : 0;
            const int r = routed ? static_cast<int>(i % RI) : static_cast<int>(i - (int64_t)U * RI);
            const float gw = routed ? __ldg(a.global + plan.expert[u]) : __ldg(a.sh_global);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int t = 2 * q + (v & 1);
                const int row = 16 * r + g + 8 * (v >> 1);
                if (t >= a.T) continue;
                const float gs = W4A4 ? __fmul_rn(gw, gx[t]) : gw;
                const float uval = __fmul_rn(acc[v], gs);
                const float rl = fmaxf(uval, 0.0f);
                const __nv_bfloat16 bv = __float2bfloat16_rn(__fmul_rn(rl, rl));
                const uint16_t bits = *reinterpret_cast<const uint16_t*>(&bv);
                if (routed) {
                    const int j = plan.choice[u][t];
                    if (j >= 0) a.act[((size_t)t * a.k + j) * a.I + row] = bits;
                } else {
                    a.act_sh[(size_t)t * a.S + row] = bits;
                }
            }
        }
    }
    __syncthreads();
    ring_drain(ring, nst);
}

struct DownArgs {
    const uint8_t* codes;   // routed down [E][H][I/2]
    const uint8_t* scales;  // [E][H][I/16]
    const float* global;    // [E]
    const uint8_t* sh_codes;  // [H][S/2]
    const uint8_t* sh_scales;
    const float* sh_global;
    int E, H, I, S;
    const int32_t* topk_idx;
    const float* topk_w;
    int T, k;
    const uint16_t* act;     // [T*k][I]
    const uint16_t* act_sh;  // [T][S]
    const uint16_t* residual;  // [T][H] or null
    uint16_t* out;             // [T][H]
    float* ypart;              // [T*k][H]
    float* ysh;                // [T][H]
    int* tilecnt;              // [H/16], zero on entry, zero on exit
    int ring_bytes;            // shared memory for the staging ring; B rows follow it
};

template <bool W4A4>
__global__ void __launch_bounds__(kThreads, 1) k_moe_down_decode(const DownArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Ring ring;
    __shared__ DecodePlan plan;
    __shared__ float gbf[3 * kDecodeMaxT];      // row globals of the B slots, [slot * T + t]
    __shared__ unsigned int red[3 * kDecodeMaxT];
    __shared__ const uint16_t* srcs[3 * kDecodeMaxT];
    __shared__ int slot_u[2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    build_plan(plan, a.topk_idx, a.topk_w, a.T, a.k, a.E);

    const int RH = a.H >> 4;
    const int U = plan.U;
    const int64_t cI = a.I >> 6, cS = a.S >> 6;  // item costs (K / 64)
    const int64_t NR = (int64_t)U * RH;
    const int64_t C = NR * cI + (int64_t)RH * cS;
    auto first_item = [&](int64_t c0) -> int64_t {  // first item whose start cost >= c0
        if (c0 <= NR * cI) return (c0 + cI - 1) / cI;
        return NR + (c0 - NR * cI + cS - 1) / cS;
    };
    const int64_t ib = first_item(C * blockIdx.x / gridDim.x);
    const int64_t ie = first_item(C * (blockIdx.x + 1) / gridDim.x);
    const int n = static_cast<int>(ie - ib);
    // stage size from the widest item this CTA owns (routed K = I, shared K = S)
    const bool has_routed = n > 0 && ib < NR, has_shared = n > 0 && ie > NR;
    const int kmax = max(has_routed ? a.I : 0, has_shared ? a.S : 0);
    const int stage_bytes = 9 * max(kmax, 64);
    const int nst = min(kMaxStages, a.ring_bytes / stage_bytes);
    ring_init(ring, nst);
    __syncthreads();

    uint8_t* ring_base = smem;
    __half* bsm = reinterpret_cast<__half*>(smem + a.ring_bytes);
    // B slots: two routed experts [T][I] each, then the shared expert [T][S]
    __half* bslot[3] = {bsm, bsm + (size_t)a.T * a.I, bsm + (size_t)2 * a.T * a.I};

    auto item_k = [&](int64_t i) { return i < NR ? a.I : a.S; };
    auto item = [&](int64_t i, const uint8_t*& c, const uint8_t*& s) {
        if (i < NR) {
            const int u = static_cast<int>(i / RH), r = static_cast<int>(i % RH);
            const int64_t row = (int64_t)plan.expert[u] * a.H + 16 * r;
            c = a.codes + row * (a.I >> 1);
            s = a.scales + row * (a.I >> 4);
        } else {
            const int64_t row = 16 * (i - NR);
            c = a.sh_codes + row * (a.S >> 1);
            s = a.sh_scales + row * (a.S >> 4);
        }
    };

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int li = 0; li < n; ++li) {
                const uint8_t *c, *s;
                item(ib + li, c, s);
                if (!ring_fill(ring, ring_base, stage_bytes, nst, li, c, s, item_k(ib + li))) break;
            }
        }
    } else {
        // B operands of the experts this CTA touches (at most two routed + shared)
        if (threadIdx.x == 0) {
            slot_u[0] = slot_u[1] = -1;
            if (n > 0 && ib < NR) slot_u[0] = static_cast<int>(ib / RH);
            if (n > 0 && ib < NR) {
                const int64_t last_routed = min(ie, NR) - 1;
                const int u1 = static_cast<int>(last_routed / RH);
                if (u1 != slot_u[0]) slot_u[1] = u1;
            }
        }
        consumer_bar();
        const bool need_sh = n > 0 && ie > NR;
        if (threadIdx.x < 3 * a.T) {
            const int sl = threadIdx.x / a.T, t = threadIdx.x % a.T;
            const uint16_t* p = nullptr;
            if (sl < 2 && slot_u[sl] >= 0) {
                const int j = plan.choice[slot_u[sl]][t];
                if (j >= 0) p = a.act + ((size_t)t * a.k + j) * a.I;
            }
            srcs[threadIdx.x] = p;
        }
        consumer_bar();
        prepare_b_rows<W4A4>(srcs, 2 * a.T, a.I, bsm, gbf, red);
        if (need_sh) {
            if (threadIdx.x < a.T) srcs[threadIdx.x] = a.act_sh + (size_t)threadIdx.x * a.S;
            consumer_bar();
            prepare_b_rows<W4A4>(srcs, a.T, a.S, bslot[2], gbf + 2 * a.T, red);
        }

        const int g = lane >> 2, q = lane & 3;
        for (int li = warp; warp < nst && li < n; li += nst) {
            const int64_t i = ib + li;
            const bool routed = i < NR;
            const int u = routed ? static_cast<int>(i / RH) : -1;
            const int r = routed ? static_cast<int>(i % RH) : static_cast<int>(i - NR);
            const int sl = routed ? (u == slot_u[0] ? 0 : (u == slot_u[1] ? 1 : -1)) : 2;
            if (sl < 0) {  // the launch guarantees at most two routed experts per CTA
                if (lane == 0) set_dev_error(kErrBadInput);
                continue;
            }
            const int K = routed ? a.I : a.S;
            const __half* bcol = nullptr;
            if (g < a.T && (!routed || plan.choice[u][g] >= 0)) bcol = bslot[sl] + (size_t)g * K;
            if (!ring_acquire(ring, nst, li)) break;
            const uint8_t* st = ring_base + (size_t)(li % nst) * stage_bytes;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            tile_mma_16x8(st, st + 16 * (K >> 1), K, bcol, acc);
            ring_release(ring, nst, li);
            const float gw = routed ? __ldg(a.global + plan.expert[u]) : __ldg(a.sh_global);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int t = 2 * q + (v & 1);
                const int row = 16 * r + g + 8 * (v >> 1);
                if (t >= a.T) continue;
                const float gs = W4A4 ? __fmul_rn(gw, gbf[sl * a.T + t]) : gw;
                const float y = __fmul_rn(acc[v], gs);
                if (routed) {
                    const int j = plan.choice[u][t];
                    if (j >= 0) a.ypart[((size_t)t * a.k + j) * a.H + row] = __fmul_rn(plan.gate[u][t], y);
                } else {
                    a.ysh[(size_t)t * a.H + row] = y;
                }
            }
            // publish, then count this contribution to output tile r
            __threadfence();
            __syncwarp();
            int prev = 0;
            if (lane == 0) prev = atomicAdd(a.tilecnt + r, 1);
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if (prev == U) {  // U routed + 1 shared contributions: this warp is last
                __threadfence();
                for (int o = lane; o < 16 * a.T; o += 32) {
                    const int t = o >> 4, row = 16 * r + (o & 15);
                    float acc2 = __ldcg(a.ysh + (size_t)t * a.H + row);
                    for (int j = 0; j < a.k; ++j)
                        acc2 = __fadd_rn(acc2, __ldcg(a.ypart + ((size_t)t * a.k + j) * a.H + row));
                    if (a.residual)
                        acc2 = __fadd_rn(acc2, bf16_bits_to_float(a.residual[(size_t)t * a.H + row]));
                    const __nv_bfloat16 ob = __float2bfloat16_rn(acc2);
                    a.out[(size_t)t * a.H + row] = *reinterpret_cast<const uint16_t*>(&ob);
                }
                if (lane == 0) a.tilecnt[r] = 0;
            }
        }
    }
    __syncthreads();
    ring_drain(ring, nst);
}

}  // namespace nvfp4moe
