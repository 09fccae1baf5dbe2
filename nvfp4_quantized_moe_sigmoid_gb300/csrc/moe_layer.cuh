// moe_layer.cuh - moe_layer_forward for 1..4 tokens: the router, the routed
// and shared experts and the combine of one MoE layer as three kernels chained
// by programmatic dependent launch, handing prepared operands to each other
// through the workspace so that no CTA repeats another's work:
//
//   route kernel (route.cuh, planning mode): RMS norm of the hidden rows,
//     gate logits, sigmoid + bias top-k; CTA rank 0 also writes the step
//     plan (unique experts, choices, gates) and the up kernel's B operand
//     (the normalised rows, NVFP4-quantised in W4A4, as exact f16 values).
//   up kernel: shared-expert tiles are staged before the wait; after it the
//     plan and B rows are loaded (bulk copies), the routed tiles streamed, and
//     relu^2 -> bf16 rows written. The last CTA to finish an expert's tiles
//     (per-expert counter) quantises that expert's intermediate rows once and
//     writes them as the down kernel's B operand.
//   down kernel: shared-expert tiles staged before the wait; plan and B rows
//     loaded; routed tiles streamed; gate-weighted partial rows written; the
//     CTA that completes a 16-row output tile sums its partials in a fixed
//     order, adds the residual and writes bf16.
// The arithmetic is that of moe_route_topk + moe_expert_forward.
#pragma once

#include "moe_decode.cuh"

namespace nvfp4moe {

// Workspace regions of moe_layer_forward (offsets computed on the host).
struct LayerWs {
    DecodePlan* plan;
    __half* xq;      // [T][H] up-B rows (exact f16)
    float* gx;       // [T] row globals of xq (W4A4), else unused
    uint16_t* act;   // [T*k][I] bf16 relu^2 rows
    uint16_t* act_sh;  // [T][S]
    __half* aq;      // [T*k][I] down-B rows
    float* ga;       // [T*k]
    __half* aq_sh;   // [T][S]
    float* gsh;      // [T]
    float* ypart;    // [T*k][H]
    float* ysh;      // [T][H]
    int* ecnt;       // [kDecodeMaxU + 1] completed up tiles per unique expert (+ shared), zero on exit
    int* tilecnt;    // [H/16] completed contributions per output tile, zero on exit
};

// Quantise (W4A4) or convert (W4A16) one bf16 row of length K held in global
// memory (written by other CTAs of this kernel, read through L2) into f16 B
// values in global memory; the whole CTA's consumer threads work on it.
template <bool W4A4>
__device__ __forceinline__ void cta_prepare_row_global(const uint16_t* src, int K, __half* dst, float* gout,
                                                       unsigned int* red_slot) {
    const int ctid = threadIdx.x;
    const int nb = K >> 4;
    uint4 u[kBRegBlocks][2];
#pragma unroll
    for (int m = 0; m < kBRegBlocks; ++m) {
        const int b = ctid + m * kConsumerThreads;
        u[m][0] = u[m][1] = make_uint4(0, 0, 0, 0);
        if (b < nb) {
            u[m][0] = __ldcg(reinterpret_cast<const uint4*>(src + 16 * b));
            u[m][1] = __ldcg(reinterpret_cast<const uint4*>(src + 16 * b + 8));
        }
    }
    float g = 0.0f;
    {
        if (ctid == 0) *red_slot = 0u;
        consumer_bar();
        float mx = 0.0f;
#pragma unroll
        for (int m = 0; m < kBRegBlocks; ++m) {
            const uint32_t w[8] = {u[m][0].x, u[m][0].y, u[m][0].z, u[m][0].w,
                                   u[m][1].x, u[m][1].y, u[m][1].z, u[m][1].w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] << 16)));
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
            }
        }
        mx = warp_max(mx);
        if ((ctid & 31) == 0) atomicMax(red_slot, __float_as_uint(mx));
        consumer_bar();
        const float amax = __uint_as_float(*red_slot);
        g = W4A4 ? __fdiv_rn(amax, 2688.0f) : w4a16_row_inv_scale(amax);
        if (ctid == 0) *gout = W4A4 ? g : w4a16_row_scale(amax);  // the epilogue's row factor
    }
#pragma unroll
    for (int m = 0; m < kBRegBlocks; ++m) {
        const int b = ctid + m * kConsumerThreads;
        if (b < nb) b_block_store<W4A4>(u[m][0], u[m][1], g, reinterpret_cast<uint4*>(dst + 16 * b));
    }
    consumer_bar();  // red_slot is reused by the next row
}

struct LayerUpArgs {
    const uint8_t* codes;   // routed up [E][I][H/2]
    const uint8_t* scales;  // [E][I][H/16]
    const float* global;    // [E]
    const uint8_t* sh_codes;
    const uint8_t* sh_scales;
    const float* sh_global;
    int E, H, I, S, T, k;
    LayerWs ws;
    int ring_bytes;
};

template <bool W4A4>
__global__ void __launch_bounds__(kThreads, 1) k_layer_up(const LayerUpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Ring ring;
    __shared__ DecodePlan plan;
    __shared__ float gx[kDecodeMaxT];
    __shared__ unsigned int red1;
    __shared__ __align__(8) uint64_t bbar;
    __shared__ int finish[3];  // expert slots this CTA completes (-1 none; 64 = shared)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stage_bytes = 9 * a.H;
    const int nst = min(kMaxStages, a.ring_bytes / stage_bytes);
    ring_init(ring, nst, nst);
    if (threadIdx.x == 0) mbar_init(&bbar, 1);
    pdl_trigger();
    __syncthreads();

    const int G = gridDim.x, b = blockIdx.x;
    const int RI = a.I >> 4, RS = a.S >> 4;
    const int64_t sb = share_begin(RS, b, G), se = share_begin(RS, b + 1, G);
    const int n_sh = static_cast<int>(se - sb);
    uint8_t* ring_base = smem;
    __half* xb = reinterpret_cast<__half*>(smem + a.ring_bytes);  // [T][H] f16 B operand

    auto sh_tile = [&](int64_t r, const uint8_t*& c, const uint8_t*& s) {
        c = a.sh_codes + 16 * r * (a.H >> 1);
        s = a.sh_scales + 16 * r * (a.H >> 4);
    };
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
    if (threadIdx.x == 0) {  // B rows prepared by the route kernel
        mbar_arrive_expect_tx(&bbar, (uint32_t)(a.T * a.H * 2));
        bulk_g2s(xb, a.ws.xq, (uint32_t)(a.T * a.H * 2), &bbar);
    }
    {  // the plan written by the route kernel
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.ws.plan);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&plan);
        for (int i = threadIdx.x; i < (int)(sizeof(DecodePlan) / 4); i += blockDim.x) dst[i] = __ldcg(src + i);
        if (threadIdx.x < a.T) gx[threadIdx.x] = __ldcg(a.ws.gx + threadIdx.x);
    }
    __syncthreads();

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
        const bool bok = __all_sync(0xffffffffu, mbar_wait_bounded(&bbar, 0));
        if (!bok && lane == 0) set_dev_error(kErrWaitFull);
        const int g = lane >> 2, q = lane & 3;
        const __half* bcol = (bok && g < a.T) ? xb + (size_t)g * a.H : nullptr;
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
                    if (j >= 0) a.ws.act[((size_t)t * a.k + j) * a.I + row] = bits;
                } else {
                    a.ws.act_sh[(size_t)t * a.S + row] = bits;
                }
            }
        }
    }
    __threadfence();  // publish this thread's rows before the CTA counts them
    __syncthreads();

    // count this CTA's finished tiles per expert; the CTA that completes an
    // expert prepares its intermediate rows for the down kernel
    if (threadIdx.x == 0) {
        finish[0] = finish[1] = finish[2] = -1;
        __threadfence();
        if (n_sh > 0 && atomicAdd(a.ws.ecnt + kDecodeMaxU, n_sh) + n_sh == RS) finish[2] = kDecodeMaxU;
        if (re > rb) {
            const int u0 = static_cast<int>(rb / RI), u1 = static_cast<int>((re - 1) / RI);
            for (int u = u0, f = 0; u <= u1 && f < 2; ++u, ++f) {
                const int64_t lo = max(rb, (int64_t)u * RI), hi = min(re, (int64_t)(u + 1) * RI);
                const int cnt = static_cast<int>(hi - lo);
                if (atomicAdd(a.ws.ecnt + u, cnt) + cnt == RI) finish[f] = u;
            }
        }
        __threadfence();
    }
    __syncthreads();
    if (warp < kConsumerWarps) {
        for (int f = 0; f < 3; ++f) {
            const int u = finish[f];
            if (u < 0) continue;
            if (u == kDecodeMaxU) {
                for (int t = 0; t < a.T; ++t)
                    cta_prepare_row_global<W4A4>(a.ws.act_sh + (size_t)t * a.S, a.S,
                                                 a.ws.aq_sh + (size_t)t * a.S, a.ws.gsh + t, &red1);
            } else {
                for (int t = 0; t < a.T; ++t) {
                    const int j = plan.choice[u][t];
                    if (j < 0) continue;
                    const size_t p = (size_t)t * a.k + j;
                    cta_prepare_row_global<W4A4>(a.ws.act + p * a.I, a.I, a.ws.aq + p * a.I, a.ws.ga + p, &red1);
                }
            }
            if (threadIdx.x == 0) a.ws.ecnt[u] = 0;
        }
    }
    __syncthreads();
    ring_drain(ring, nst);
}

struct LayerDownArgs {
    const uint8_t* codes;   // routed down [E][H][I/2]
    const uint8_t* scales;  // [E][H][I/16]
    const float* global;    // [E]
    const uint8_t* sh_codes;  // [H][S/2]
    const uint8_t* sh_scales;
    const float* sh_global;
    int E, H, I, S, T, k;
    LayerWs ws;
    const uint16_t* residual;  // [T][H] or null
    uint16_t* out;             // [T][H]
    int ring_bytes;
};

template <bool W4A4>
__global__ void __launch_bounds__(kThreads, 1) k_layer_down(const LayerDownArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Ring ring;
    __shared__ DecodePlan plan;
    __shared__ float gbf[3 * kDecodeMaxT];  // row globals of the B slots, [slot * T + t]
    __shared__ int slot_u[2];
    __shared__ __align__(8) uint64_t bbar;
    __shared__ int tdone[32];  // output tiles this CTA completes
    __shared__ int ntdone;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int RH = a.H >> 4;
    const int64_t sb = share_begin(RH, b, G), se = share_begin(RH, b + 1, G);
    const int n_sh = static_cast<int>(se - sb);
    const int kmax = n_sh > 0 ? max(a.I, a.S) : a.I;
    const int stage_bytes = 9 * kmax;
    const int nst = min(kMaxStages, a.ring_bytes / stage_bytes);
    ring_init(ring, nst, nst);
    if (threadIdx.x == 0) mbar_init(&bbar, 1);
    pdl_trigger();
    __syncthreads();

    uint8_t* ring_base = smem;
    __half* bsm = reinterpret_cast<__half*>(smem + a.ring_bytes);
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
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.ws.plan);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&plan);
        for (int i = threadIdx.x; i < (int)(sizeof(DecodePlan) / 4); i += blockDim.x) dst[i] = __ldcg(src + i);
    }
    __syncthreads();

    const int U = plan.U;
    const int64_t NR = (int64_t)U * RH;
    const int64_t rb = share_begin(NR, b, G), re = share_begin(NR, b + 1, G);
    const int n = n_sh + static_cast<int>(re - rb);
    if (threadIdx.x == 0) {
        slot_u[0] = slot_u[1] = -1;
        if (re > rb) {
            slot_u[0] = static_cast<int>(rb / RH);
            const int u1 = static_cast<int>((re - 1) / RH);
            if (u1 != slot_u[0]) slot_u[1] = u1;
        }
        // B rows of the experts this CTA touches, prepared by the up kernel
        uint32_t bytes = 0;
        for (int sl = 0; sl < 2; ++sl) {
            if (slot_u[sl] < 0) continue;
            for (int t = 0; t < a.T; ++t) {
                const int j = plan.choice[slot_u[sl]][t];
                if (j < 0) continue;
                const size_t p = (size_t)t * a.k + j;
                bytes += (uint32_t)(a.I * 2);
                gbf[sl * a.T + t] = __ldcg(a.ws.ga + p);
            }
        }
        if (n_sh > 0) {
            bytes += (uint32_t)(a.T * a.S * 2);
            for (int t = 0; t < a.T; ++t) gbf[2 * a.T + t] = __ldcg(a.ws.gsh + t);
        }
        mbar_arrive_expect_tx(&bbar, bytes);
        for (int sl = 0; sl < 2; ++sl) {
            if (slot_u[sl] < 0) continue;
            for (int t = 0; t < a.T; ++t) {
                const int j = plan.choice[slot_u[sl]][t];
                if (j < 0) continue;
                const size_t p = (size_t)t * a.k + j;
                bulk_g2s((sl ? bslot1 : bslot0) + (size_t)t * a.I, a.ws.aq + p * a.I, (uint32_t)(a.I * 2), &bbar);
            }
        }
        if (n_sh > 0) bulk_g2s(bslot2, a.ws.aq_sh, (uint32_t)(a.T * a.S * 2), &bbar);
    }
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
    __syncthreads();

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
        const bool bok = __all_sync(0xffffffffu, mbar_wait_bounded(&bbar, 0));
        if (!bok && lane == 0) set_dev_error(kErrWaitFull);
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
            if (sl < 0 && lane == 0) set_dev_error(kErrBadInput);
            __half* const bs = sl == 0 ? bslot0 : (sl == 1 ? bslot1 : bslot2);
            const __half* bcol = nullptr;
            if (bok && sl >= 0 && g < a.T && (!routed || plan.choice[u][g] >= 0)) bcol = bs + (size_t)g * K;
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
                    if (j >= 0) a.ws.ypart[((size_t)t * a.k + j) * a.H + row] = __fmul_rn(plan.gate[u][t], y);
                } else {
                    a.ws.ysh[(size_t)t * a.H + row] = y;
                }
            }
        }
    }
    __threadfence();  // publish this thread's partial rows before the CTA counts them
    __syncthreads();

    // count this CTA's contributions per output tile (once per CTA); the CTA
    // that completes a tile (U routed + 1 shared contributions) combines it.
    // Routed items cover fewer than RH consecutive (u, r), so a tile r occurs
    // at most once among them, plus at most once among the shared items.
    if (threadIdx.x == 0) {
        int nd = 0;
        auto count = [&](int r, int c) {
            if (atomicAdd(a.ws.tilecnt + r, c) + c == U + 1 && nd < 32) tdone[nd++] = r;
        };
        for (int64_t r = sb; r < se; ++r) {
            int c = 1;
            for (int64_t i = rb; i < re; ++i)
                if (i % RH == r) ++c;
            count(static_cast<int>(r), c);
        }
        for (int64_t i = rb; i < re; ++i) {
            const int64_t r = i % RH;
            if (r >= sb && r < se) continue;  // counted with the shared tile
            count(static_cast<int>(r), 1);
        }
        ntdone = nd;
        __threadfence();
    }
    __syncthreads();
    if (warp < kConsumerWarps) {
        const int nd = ntdone;
        for (int o = threadIdx.x; o < nd * 16 * a.T; o += kConsumerThreads) {
            const int d = o / (16 * a.T), rem = o % (16 * a.T);
            const int t = rem >> 4, row = 16 * tdone[d] + (rem & 15);
            float yv[kDecodeMaxK];
#pragma unroll
            for (int j = 0; j < kDecodeMaxK; ++j)
                yv[j] = j < a.k ? __ldcg(a.ws.ypart + ((size_t)t * a.k + j) * a.H + row) : 0.0f;
            float acc2 = __ldcg(a.ws.ysh + (size_t)t * a.H + row);
            const float res = a.residual ? bf16_bits_to_float(__ldcg(a.residual + (size_t)t * a.H + row)) : 0.0f;
#pragma unroll
            for (int j = 0; j < kDecodeMaxK; ++j)
                if (j < a.k) acc2 = __fadd_rn(acc2, yv[j]);
            if (a.residual) acc2 = __fadd_rn(acc2, res);
            const __nv_bfloat16 ob = __float2bfloat16_rn(acc2);
            a.out[(size_t)t * a.H + row] = *reinterpret_cast<const uint16_t*>(&ob);
        }
        if (threadIdx.x < nd) a.ws.tilecnt[tdone[threadIdx.x]] = 0;
    }
    __syncthreads();
    ring_drain(ring, nst);
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bbar, 0)) set_dev_error(kErrWaitDrain);
}

}  // namespace nvfp4moe
