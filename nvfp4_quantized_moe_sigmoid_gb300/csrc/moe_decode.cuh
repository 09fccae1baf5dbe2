// moe_decode.cuh - moe_expert_forward for 1..4 tokens (batch-1 decode and the
// 4-token speculative verify of "Let's optimize Nemotron 3.5 Lightning - a
// worklog", Step 5). At this size the layer is a stream of NVFP4 weights
// (worklog, Interlude), so both kernels are persistent HBM streams:
//
//   up kernel   : items = 16-row tiles of the shared expert's up_proj and of
//                 every selected expert's up_proj. Epilogue: relu^2 -> bf16
//                 intermediate rows in the workspace.
//   down kernel : items = 16-row tiles of the shared expert's down_proj and of
//                 every selected expert's down_proj. Epilogue: gate-weighted
//                 FP32 partial rows; the warp that completes a 16-row output
//                 tile (per-tile counter) sums the partials in a fixed order,
//                 adds the residual and writes bf16.
//
// Each CTA takes an even share of the shared-expert tiles and an even share of
// the routed tiles. The shared-expert tiles do not depend on the routing, so
// their bulk copies are issued before the kernel waits on the previous one
// (programmatic dependent launch); the routed ones follow once the plan is
// built. One producer thread streams the tiles through the staging ring,
// sixteen consumer warps (eight pairs) run the tensor-core tile. Experts
// chosen by several tokens are read once per step: items are per unique
// expert and the MMA's columns are the tokens.
#pragma once

#include "gemv_tile.cuh"

namespace nvfp4moe {

constexpr int kDecodeMaxT = 4;
constexpr int kDecodeMaxK = 16;
constexpr int kDecodeMaxU = kDecodeMaxT * kDecodeMaxK;

struct DecodePlan {
    int U;                                    // unique experts this step
    int expert[kDecodeMaxU];                  // ascending expert ids
    int8_t choice[kDecodeMaxU][kDecodeMaxT];  // j with topk_idx[t][j] == expert, else -1
    float gate[kDecodeMaxU][kDecodeMaxT];     // topk_w[t][j] or 0
    unsigned int bits[8];                     // E <= 256 bitmap
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
        e = __ldcg(topk_idx + tid);
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
        p.gate[slot][tid / k] = __ldcg(topk_w + tid);
    }
    if (tid == 0) {
        int u = 0;
        for (int w = 0; w < 8; ++w) u += __popc(p.bits[w]);
        p.U = u;
    }
    __syncthreads();
}

__device__ __forceinline__ int64_t share_begin(int64_t n, int b, int G) { return n * b / G; }

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
    ring_init(ring, nst, nst);
    pdl_trigger();
    __syncthreads();

    const int G = gridDim.x, b = blockIdx.x;
    const int RI = a.I >> 4, RS = a.S >> 4;
    const int64_t sb = share_begin(RS, b, G), se = share_begin(RS, b + 1, G);
    const int n_sh = static_cast<int>(se - sb);
    uint8_t* ring_base = smem;
    __half* xb = reinterpret_cast<__half*>(smem + a.ring_bytes);             // [T][H] f16 B operand
    uint16_t* xn = reinterpret_cast<uint16_t*>(xb + (size_t)a.T * a.H);      // [T][H] normalised bf16

    auto sh_tile = [&](int64_t r, const uint8_t*& c, const uint8_t*& s) {
        c = a.sh_codes + 16 * r * (a.H >> 1);
        s = a.sh_scales + 16 * r * (a.H >> 4);
    };
    // shared-expert weights do not depend on the previous kernel: stage them first
    const int pre = min(n_sh, nst);
    FillCursor fc = fill_cursor(0, nst);  // the producer's next item
    if (warp == kConsumerWarps && lane == 0) {
        for (int li = 0; li < pre; ++li) {
            const uint8_t *c, *s;
            sh_tile(sb + li, c, s);
            ring_fill(ring, ring_base, stage_bytes, nst, fc, c, s, a.H);
        }
    }
    pdl_wait();
    build_plan(plan, a.topk_idx, a.topk_w, a.T, a.k, a.E);  // contains __syncthreads

    const int U = plan.U;
    const int64_t NR = (int64_t)U * RI;
    const int64_t rb = share_begin(NR, b, G), re = share_begin(NR, b + 1, G);
    const int n = n_sh + static_cast<int>(re - rb);
    auto item = [&](int li, const uint8_t*& c, const uint8_t*& s) {
        if (li < n_sh) {
            sh_tile(sb + li, c, s);
        } else {
            const int i = static_cast<int>(rb) + (li - n_sh);  // U x rows < 2^31
            const int u = static_cast<int>(i / RI), r = static_cast<int>(i % RI);
            const int64_t row = (int64_t)plan.expert[u] * a.I + 16 * r;
            c = a.codes + row * (a.H >> 1);
            s = a.scales + row * (a.H >> 4);
        }
    };

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int li = pre; li < n; ++li) {
                const uint8_t *c, *s;
                item(li, c, s);
                if (!ring_fill(ring, ring_base, stage_bytes, nst, fc, c, s, a.H)) break;
            }
        }
    } else {
        if (warp < a.T) {
            if (a.rms_eps > 0.0f)
                warp_rmsnorm_row(a.hidden + (size_t)warp * a.H, xn + (size_t)warp * a.H, a.H, a.rms_eps);
            else
                warp_copy_row(a.hidden + (size_t)warp * a.H, xn + (size_t)warp * a.H, a.H);
        }
        if (threadIdx.x < a.T) srcs[threadIdx.x] = xn + (size_t)threadIdx.x * a.H;
        consumer_bar();
        prepare_b_rows<W4A4, false>(srcs, a.T, a.H, xb, gx, red);
        const int g = lane >> 2, q = lane & 3;
        const __half* bcol = g < a.T ? xb + (size_t)g * a.H : nullptr;
        GroupCursor cur = group_cursor(nst, nst, a.H, a.H);
        for (; cur.li < n; cursor_next(cur)) {
            const int li = cur.li;
            float acc[4];
            bool ok;
            const bool mine = group_tile(ring, cur, ring_base, stage_bytes, a.H, bcol, acc, ok);
            if (!ok) break;
            if (!mine) continue;
            const bool routed = li >= n_sh;
            int u = 0, r;
            if (routed) {
                const int i = static_cast<int>(rb) + (li - n_sh);  // U x rows < 2^31
                u = static_cast<int>(i / RI);
                r = static_cast<int>(i % RI);
            } else {
                r = static_cast<int>(sb + li);
            }
            const float gw = routed ? __ldg(a.global + plan.expert[u]) : __ldg(a.sh_global);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int t = 2 * q + (v & 1);
                const int row = 16 * r + g + 8 * (v >> 1);
                if (t >= a.T) continue;
                const float gs = __fmul_rn(gw, gx[t]);  // gx: W4A4 row global, W4A16 row prescale
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
    const uint16_t* act;       // [T*k][I]
    const uint16_t* act_sh;    // [T][S]
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
    __shared__ float gbf[3 * kDecodeMaxT];  // row globals of the B slots, [slot * T + t]
    __shared__ unsigned int red[3 * kDecodeMaxT];
    __shared__ const uint16_t* srcs[3 * kDecodeMaxT];
    __shared__ int slot_u[2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int RH = a.H >> 4;
    const int64_t sb = share_begin(RH, b, G), se = share_begin(RH, b + 1, G);
    const int n_sh = static_cast<int>(se - sb);
    // stage size from the widest item this CTA can own (routed K = I, shared K = S)
    const int kmax = n_sh > 0 ? max(a.I, a.S) : a.I;
    const int stage_bytes = 9 * kmax;
    const int nst = min(kMaxStages, a.ring_bytes / stage_bytes);
    ring_init(ring, nst, nst);
    pdl_trigger();
    __syncthreads();

    uint8_t* ring_base = smem;
    __half* bsm = reinterpret_cast<__half*>(smem + a.ring_bytes);
    // B slots: two routed experts [T][I] each, then the shared expert [T][S]
    __half* const bslot0 = bsm;
    __half* const bslot1 = bsm + (size_t)a.T * a.I;
    __half* const bslot2 = bsm + (size_t)2 * a.T * a.I;

    auto sh_tile = [&](int64_t r, const uint8_t*& c, const uint8_t*& s) {
        c = a.sh_codes + 16 * r * (a.S >> 1);
        s = a.sh_scales + 16 * r * (a.S >> 4);
    };
    const int pre = min(n_sh, nst);
    FillCursor fc = fill_cursor(0, nst);  // the producer's next item
    if (warp == kConsumerWarps && lane == 0) {
        for (int li = 0; li < pre; ++li) {
            const uint8_t *c, *s;
            sh_tile(sb + li, c, s);
            ring_fill(ring, ring_base, stage_bytes, nst, fc, c, s, a.S);
        }
    }
    pdl_wait();
    build_plan(plan, a.topk_idx, a.topk_w, a.T, a.k, a.E);

    const int U = plan.U;
    const int64_t NR = (int64_t)U * RH;
    const int64_t rb = share_begin(NR, b, G), re = share_begin(NR, b + 1, G);
    const int n = n_sh + static_cast<int>(re - rb);
    auto item = [&](int li, const uint8_t*& c, const uint8_t*& s, int& K) {
        if (li < n_sh) {
            sh_tile(sb + li, c, s);
            K = a.S;
        } else {
            const int i = static_cast<int>(rb) + (li - n_sh);  // U x rows < 2^31
            const int u = static_cast<int>(i / RH), r = static_cast<int>(i % RH);
            const int64_t row = (int64_t)plan.expert[u] * a.H + 16 * r;
            c = a.codes + row * (a.I >> 1);
            s = a.scales + row * (a.I >> 4);
            K = a.I;
        }
    };

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int li = pre; li < n; ++li) {
                const uint8_t *c, *s;
                int K;
                item(li, c, s, K);
                if (!ring_fill(ring, ring_base, stage_bytes, nst, fc, c, s, K)) break;
            }
        }
    } else {
        // B operands of the experts this CTA touches (at most two routed + shared)
        if (threadIdx.x == 0) {
            slot_u[0] = slot_u[1] = -1;
            if (re > rb) {
                slot_u[0] = static_cast<int>(rb / RH);
                const int u1 = static_cast<int>((re - 1) / RH);
                if (u1 != slot_u[0]) slot_u[1] = u1;
            }
        }
        consumer_bar();
        if (threadIdx.x < 2 * a.T) {
            const int sl = threadIdx.x / a.T, t = threadIdx.x % a.T;
            const uint16_t* p = nullptr;
            if (slot_u[sl] >= 0) {
                const int j = plan.choice[slot_u[sl]][t];
                if (j >= 0) p = a.act + ((size_t)t * a.k + j) * a.I;
            }
            srcs[threadIdx.x] = p;
        }
        consumer_bar();
        prepare_b_rows<W4A4, true>(srcs, 2 * a.T, a.I, bsm, gbf, red);
        if (n_sh > 0) {
            if (threadIdx.x < a.T) srcs[threadIdx.x] = a.act_sh + (size_t)threadIdx.x * a.S;
            consumer_bar();
            prepare_b_rows<W4A4, true>(srcs, a.T, a.S, bslot2, gbf + 2 * a.T, red);
        }

        const int g = lane >> 2, q = lane & 3;
        GroupCursor cur = group_cursor(nst, nst, a.I, a.S);
        for (; cur.li < n; cursor_next(cur)) {
            const int li = cur.li;
            const bool routed = li >= n_sh;
            int u = -1, r, sl, K;
            if (routed) {
                const int i = static_cast<int>(rb) + (li - n_sh);  // U x rows < 2^31
                u = static_cast<int>(i / RH);
                r = static_cast<int>(i % RH);
                sl = u == slot_u[0] ? 0 : (u == slot_u[1] ? 1 : -1);
                K = a.I;
            } else {
                r = static_cast<int>(sb + li);
                sl = 2;
                K = a.S;
            }
            // the launch guarantees at most two routed experts per CTA
            if (sl < 0 && lane == 0) set_dev_error(kErrBadInput);
            __half* const bs = sl == 0 ? bslot0 : (sl == 1 ? bslot1 : bslot2);
            const __half* bcol = nullptr;
            if (sl >= 0 && g < a.T && (!routed || plan.choice[u][g] >= 0)) bcol = bs + (size_t)g * K;
            float acc[4];
            bool ok;
            const bool mine = group_tile(ring, cur, ring_base, stage_bytes, K, bcol, acc, ok);
            if (!ok) break;
            if (!mine) continue;
            const float gw = routed ? __ldg(a.global + plan.expert[u]) : __ldg(a.sh_global);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int t = 2 * q + (v & 1);
                const int row = 16 * r + g + 8 * (v >> 1);
                if (t >= a.T || sl < 0) continue;
                const float gs = __fmul_rn(gw, gbf[sl * a.T + t]);
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
                    // all loads of this output first, then the fixed-order sum
                    float yv[kDecodeMaxK];
#pragma unroll
                    for (int j = 0; j < kDecodeMaxK; ++j)
                        yv[j] = j < a.k ? __ldcg(a.ypart + ((size_t)t * a.k + j) * a.H + row) : 0.0f;
                    float acc2 = __ldcg(a.ysh + (size_t)t * a.H + row);
                    const float res = a.residual ? bf16_bits_to_float(__ldcg(a.residual + (size_t)t * a.H + row)) : 0.0f;
#pragma unroll
                    for (int j = 0; j < kDecodeMaxK; ++j)
                        if (j < a.k) acc2 = __fadd_rn(acc2, yv[j]);
                    if (a.residual) acc2 = __fadd_rn(acc2, res);
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
