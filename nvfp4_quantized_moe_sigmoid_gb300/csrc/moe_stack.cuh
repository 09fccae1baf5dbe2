// moe_stack.cuh - moe_stack_forward: L consecutive MoE decode layers (1..4
// tokens, pre-norm residual chain h_{l+1} = h_l + moe_l(norm(h_l))) in one
// persistent cooperative kernel, one CTA per SM.
//
// Decode at this size is a stream of NVFP4 weights ("Let's optimize Nemotron
// 3.5 Lightning - a worklog", Interlude), and between layers it is a chain of
// small dependent steps (router, top-k, experts, combine). Separate kernels
// pay a drain and a fill at every step; here every CTA runs the whole chain
// and the steps meet through per-layer counters in the workspace:
//
//   per layer l, every CTA:
//     1. wait until every 16-row tile of h_l is final (counter); load h_l;
//     2. x = RMSNorm(h_l); B operand of the up tiles (NVFP4 in W4A4);
//     3. router logits of this CTA's experts (gate rows staged in shared
//        memory during the previous layer) -> workspace, count them;
//     4. wait for all E logits; sigmoid + bias top-k (rank per expert, every
//        CTA computes the same selection), the step plan (unique experts);
//        from here the producer streams the routed tiles;
//     5. its share of the shared expert's up tiles (staged during the
//        previous layer, computed while the routed tiles are in flight):
//        relu^2 -> bf16 rows + row amax (W4A4);
//     6. its share of the routed up tiles (per-expert done counters);
//     7. wait for the experts whose down tiles it owns; quantise their
//        intermediate rows with the now final row amax (W4A4) as its B operand;
//     8. its share of the shared and routed down tiles -> gate-weighted FP32
//        partial rows; each tile counts its contribution to its 16 output
//        rows, and the warp that brings the last one (U routed + 1 shared)
//        combines them: h_{l+1} = bf16(shared + sum_j gate_j y_j + h_l).
//
// One producer thread streams every tile the CTA owns through the staging
// ring in consumption order, and fills the next layer's constant tiles
// (router rows, shared-expert up tiles) as soon as stages free up, so they
// land while the current layer is still waiting on its dependencies.
// Every wait is bounded; a CTA that gives up sets the workspace abort flag,
// which ends every other CTA's waits, and the last CTA to leave resets the
// counters for the next call.
//
// The steps are out-of-line functions sharing one per-CTA context in shared
// memory, which keeps the code a layer runs small enough for the SM's
// instruction cache to hold from one layer to the next.
#pragma once

#include "moe_decode.cuh"

namespace nvfp4moe {

constexpr int kStackMaxLayers = 32;

struct StackLayer {
    const uint8_t* up_codes;  // [E][I][H/2]
    const uint8_t* up_scales;
    const float* up_global;   // [E]
    const uint8_t* down_codes;  // [E][H][I/2]
    const uint8_t* down_scales;
    const float* down_global;
    const uint8_t* shu_codes;  // [S][H/2]
    const uint8_t* shu_scales;
    const float* shu_global;
    const uint8_t* shd_codes;  // [H][S/2]
    const uint8_t* shd_scales;
    const float* shd_global;
    const float* router_w;  // [E][H]
    const float* router_b;  // [E]
};

// Per-layer counters: fixed slots, then one per unique expert, then one per
// 16-row output tile.
constexpr int kCntLogits = 0;  // router logits written (target E)
constexpr int kCntShUp = 1;    // shared-expert up tiles done (target S/16)
constexpr int kCntHDone = 2;   // output tiles of h_{l+1} final (target H/16)
constexpr int kCntUp = 3;      // + u: up tiles of unique expert u done (target I/16)
constexpr int kCntTile = kCntUp + kDecodeMaxU;  // + r: contributions to output tile r (target U + 1)
__host__ __device__ constexpr int stack_cnt_per_layer(int H) { return kCntTile + H / 16; }

struct StackWs {
    int* cnt;            // [L][stack_cnt_per_layer], then the exit count and the abort flag
    float* z;            // [L][T][E] router logits
    uint16_t* act;       // [T*k][I] bf16 relu^2 rows of the routed experts
    uint16_t* act_sh;    // [T][S] of the shared expert
    unsigned int* amax;  // [2][T*k + T] row amax bits of act, then act_sh, by layer parity
    float* ypart;        // [T*k][H] gate-weighted down rows
    float* ysh;          // [T][H] shared-expert down rows
};

struct StackArgs {
    StackLayer layer[kStackMaxLayers];
    int L, E, H, I, S, T, k;
    float rms_eps;
    const uint16_t* hidden_in;  // [T][H] h_0
    uint16_t* hidden_out;       // [L][T][H] h_1 .. h_L
    int32_t* topk_idx;          // [L][T][k]
    float* topk_w;              // [L][T][k]
    StackWs ws;
    int ring_cap;                   // staging ring bytes at the start of dynamic shared memory
    int off_gate, off_uni, off_tk;  // dynamic shared-memory regions after the ring
};

// Counter updates that publish data: the warp's (or CTA's) earlier writes,
// ordered before the executing thread by a warp or CTA barrier, are visible
// to whoever acquires the counter (no separate full fence).
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_add(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *p >= target. False if the wait expired (flags the error word and
// the abort flag) or another CTA raised the abort flag.
__device__ __noinline__ bool wait_geq(const int* p, int target, int* abort_g) {
    if (ld_acquire_gpu(p) >= target) return true;  // no timer read when nothing to wait for
    const unsigned long long t0 = globaltimer();
    for (int it = 0;; ++it) {
        if (ld_acquire_gpu(p) >= target) return true;
        __nanosleep(64);  // leave the issue slots to the computing warps
        if ((it & 15) == 15) {
            if (ld_acquire_gpu(abort_g)) return false;
            if (globaltimer() - t0 > kWaitTimeoutNs) {
                set_dev_error(kErrWaitPeer);
                atomicExch(abort_g, 1);
                return false;
            }
        }
    }
}

__device__ __noinline__ bool mbar_wait_abortable(uint64_t* b, uint32_t parity, volatile int* abort_s,
                                                unsigned int err = kErrWaitFull) {
    if (mbar_try_wait(b, parity)) return true;  // no timer read and no suspension when the phase is done
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(b, parity)) return true;
        if (*abort_s) return false;
        if (globaltimer() - t0 > kWaitTimeoutNs) {
            set_dev_error(err);
            return false;
        }
    }
}

// ---------------------------------------------------------------- staging ring
// A byte ring over the CTA's free shared memory. 16-row tiles of any K
// (9 K bytes: codes [16][K/2], then scales [16][K/16]) are placed one after
// another in issue order (an item that would cross the end starts again at
// offset 0), so that as many tiles are in flight as fit, whatever their K.
// Item li completes on full[li % kSlots] and is computed by warp group
// li % kGroups (the consumer warps w with w % kGroups == li % kGroups), whose
// kGroupWarps warps each take a contiguous share of its 128-k chunks and
// release it on empty[li % kSlots]. kSlots is a multiple of kGroups, so the
// same warps wait on every use of a slot, in order (a parity wait can only
// tell the current phase of an mbarrier from the one before it). The
// producer reclaims space in issue order: before placing an item it waits
// until the item that last used the slot, and every older item whose bytes
// the new one would overwrite, have been released.
constexpr int kGroups = 4;
constexpr int kGroupWarps = kConsumerWarps / kGroups;
constexpr int kSlots = 16;
static_assert(kConsumerWarps % kGroups == 0 && kSlots % kGroups == 0, "ring groups");
static_assert((kSlots & (kSlots - 1)) == 0, "slot index by mask");

struct BRing {
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    uint32_t off[kSlots];  // byte offset of the slot's current item
    int vs[kSlots];        // its virtual start (producer side)
    int uses[kSlots];      // fills of the slot (producer side)
    // partial tiles handed from ranks 1.. of a group to its rank 0, double
    // buffered by the group's item parity; warp w >= kGroups uses w - kGroups
    float4 xred[kConsumerWarps - kGroups][2][32];
};

constexpr int kNormMaxChunks = 64;  // H <= 16384

// Per-CTA state of the stack kernel, in shared memory.
struct StackCta {
    BRing br;
    DecodePlan plan;
    uint64_t gbar;  // router rows landed (one phase per layer)
    uint64_t pbar;  // plan ready for the producer (one phase per layer)
    uint64_t qbar;  // producer done reading the plan (one phase per layer)
    int gate_issued;
    int abort_s;
    int last_cta;  // this CTA is the last to leave (resets the workspace)
    // geometry
    int G, b, ring_cap, ng, amax_stride;
    int su_b, su_e, sd_b, sd_e;  // shared-expert up / down tile ranges of this CTA
    uint8_t* ring_base;
    float* gsm;      // [ng][H] router rows
    uint16_t* X;     // [T][H] h_l, then x_l
    __half* xq;      // [T][H] up B operand
    __half* bslot;   // down B: routed [T][I], [T][I], shared [T][S] (aliases X, xq)
    float* tk_c;     // [T][E] biased scores
    float* tk_s;     // [T][E] sigmoids
    // step scratch
    float norm_part[kDecodeMaxT][kNormMaxChunks];
    float norm_inv[kDecodeMaxT];
    float gx[kDecodeMaxT];
    unsigned int red[kDecodeMaxT];
    float gbf[3 * kDecodeMaxT];
    int sel_idx[kDecodeMaxT][kDecodeMaxK];
    float sel_sig[kDecodeMaxT][kDecodeMaxK];
    float sel_w[kDecodeMaxT][kDecodeMaxK];
    float zred[kConsumerWarps][kDecodeMaxT];
    int slot_u[2];
    // per-tensor globals of this layer's unique experts and shared expert
    float up_g[kDecodeMaxU], down_g[kDecodeMaxU];
    float shu_g, shd_g;
    // router correction bias and the routed experts' per-tensor globals of
    // the current layer, staged with its router rows
    __align__(16) float bias_s[256];
    __align__(16) float upg_s[256];
    __align__(16) float dng_s[256];
};

__device__ __forceinline__ bool cta_abort(StackCta& c) { return *static_cast<volatile int*>(&c.abort_s) != 0; }
__device__ __forceinline__ void set_cta_abort(StackCta& c) { *static_cast<volatile int*>(&c.abort_s) = 1; }

// Consumers: item li by its warp group (see the ring above); the group's
// rank-0 warp gets lead = 1 and the finished 16 x 8 tile, ok = 0 in every
// warp of the group if any of them timed out.
__device__ __noinline__ TileOut bgroup_tile_core(StackCta* cp, int li, int K, const __half* bcol) {
    BRing& r = cp->br;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp % kGroups, rank = warp / kGroups;
    const int s = li % kSlots;
    const bool waited = mbar_wait_bounded(&r.full[s], static_cast<uint32_t>((li / kSlots) & 1));
    const bool got = __all_sync(0xffffffffu, waited);
    if (!got && lane == 0) set_dev_error(kErrWaitFull);
    const int nc = (K + 127) >> 7;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (got) {
        const uint8_t* st = cp->ring_base + r.off[s];
        tile_mma_16x8(st, st + 8 * K, K, bcol, nc * rank / kGroupWarps, nc * (rank + 1) / kGroupWarps, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&r.empty[s]);
    TileOut o;
    o.acc = make_float4(acc[0], acc[1], acc[2], acc[3]);
    const int u = (li / kGroups) & 1;
    if (rank) r.xred[warp - kGroups][u][lane] = o.acc;
    o.ok = group_bar_and(g, kGroupWarps, got);
    o.lead = 0;
    if (rank || !o.ok) return o;
#pragma unroll
    for (int p = 1; p < kGroupWarps; ++p) {
        const float4 x = r.xred[g + (p - 1) * kGroups][u][lane];
        o.acc.x += x.x;
        o.acc.y += x.y;
        o.acc.z += x.z;
        o.acc.w += x.w;
    }
    o.lead = 1;
    return o;
}

__device__ __forceinline__ bool bgroup_tile(StackCta& c, int li, int K, const __half* bcol, float (&acc)[4],
                                            bool& ok) {
    const TileOut o = bgroup_tile_core(&c, li, K, bcol);
    acc[0] = o.acc.x;
    acc[1] = o.acc.y;
    acc[2] = o.acc.z;
    acc[3] = o.acc.w;
    ok = o.ok != 0;
    return o.lead != 0;
}

__device__ __forceinline__ int* layer_cnt(const StackArgs& a, int l) {
    return a.ws.cnt + (size_t)l * stack_cnt_per_layer(a.H);
}
__device__ __forceinline__ int* abort_flag(const StackArgs& a) {
    return a.ws.cnt + (size_t)a.L * stack_cnt_per_layer(a.H) + 1;
}

// Even share of n items: CTA b of G takes [n b / G, n (b + 1) / G) (n G < 2^31).
__device__ __forceinline__ int share_begin32(int n, int b, int G) { return n * b / G; }

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    const __nv_bfloat16 x = __float2bfloat16_rn(lo), y = __float2bfloat16_rn(hi);
    return static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&x)) |
           (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&y)) << 16);
}

// ---------------------------------------------------------------- steps 1-2
// h_l (global, final) -> X; x_l = RMSNorm(h_l) in place (or h_l); the up
// tiles' B operand from x_l. RMS norm: inv = 1/sqrt(sum x^2 / H + eps),
// y = bf16(x * inv); chunk c = elements [256c, 256c + 256), lane l sums its
// eight elements 256c + 8l .. + 7 in order (fused multiply-add), an
// xor-shuffle tree gives the chunk sum, chunk sums are added in chunk order.
template <bool W4A4>
__device__ __noinline__ void st_input(const StackArgs& a, StackCta& c, const uint16_t* h, int l) {
    const int ctid = threadIdx.x, warp = ctid >> 5, lane = ctid & 31;
    const int T = a.T, H = a.H;
    uint16_t* X = c.X;
    if (ctid == kConsumerThreads - 1) {  // used by the epilogues later in the layer
        c.shu_g = __ldg(a.layer[l].shu_global);
        c.shd_g = __ldg(a.layer[l].shd_global);
    }
#pragma unroll 1
    for (int i = 8 * ctid; i < T * H; i += 8 * kConsumerThreads)
        *reinterpret_cast<uint4*>(X + i) = __ldcg(reinterpret_cast<const uint4*>(h + i));
    consumer_bar();
    if (a.rms_eps > 0.0f) {
        const int nch = (H + 255) >> 8;
#pragma unroll 1
        for (int item = warp; item < T * nch; item += kConsumerWarps) {
            const int r = item / nch, ch = item % nch;
            const int i = 256 * ch + 8 * lane;
            float ss = 0.0f;
            if (i < H) {
                const uint4 v = *reinterpret_cast<const uint4*>(X + (size_t)r * H + i);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x0 = __uint_as_float(w[j] << 16), x1 = __uint_as_float(w[j] & 0xFFFF0000u);
                    ss = __fmaf_rn(x0, x0, ss);
                    ss = __fmaf_rn(x1, x1, ss);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
            if (lane == 0) c.norm_part[r][ch] = ss;
        }
        consumer_bar();
        if (ctid < T) {
            float sum = 0.0f;
#pragma unroll 1
            for (int ch0 = 0; ch0 < nch; ch0 += 8) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = ch0 + j < nch ? c.norm_part[ctid][ch0 + j] : 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (ch0 + j < nch) sum = __fadd_rn(sum, v[j]);
            }
            c.norm_inv[ctid] =
                __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, static_cast<float>(H)), a.rms_eps)));
        }
        consumer_bar();
#pragma unroll 1
        for (int i = 8 * ctid; i < T * H; i += 8 * kConsumerThreads) {
            const float inv = c.norm_inv[i / H];
            const uint4 v = *reinterpret_cast<const uint4*>(X + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o[j] = bf16x2_rn(__fmul_rn(__uint_as_float(w[j] << 16), inv),
                                 __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), inv));
            *reinterpret_cast<uint4*>(X + i) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    // B operand: per-row global = amax / 2688 (W4A4), then each 16-block
    const int nb = H >> 4;
    if (W4A4) {
        if (ctid < T) c.red[ctid] = 0u;
        consumer_bar();
#pragma unroll 1
        for (int i = ctid; i < T * nb; i += kConsumerThreads) {
            const uint16_t* p = X + (size_t)(i / nb) * H + 16 * (i % nb);
            const uint4 u0 = *reinterpret_cast<const uint4*>(p), u1 = *reinterpret_cast<const uint4*>(p + 8);
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            float mx = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
            atomicMax(&c.red[i / nb], __float_as_uint(mx));
        }
    }
    consumer_bar();
    if (W4A4 && ctid < T) c.gx[ctid] = __fdiv_rn(__uint_as_float(c.red[ctid]), 2688.0f);
#pragma unroll 1
    for (int i = ctid; i < T * nb; i += kConsumerThreads) {
        const int r = i / nb;
        const uint16_t* p = X + (size_t)r * H + 16 * (i % nb);
        const float g = W4A4 ? __fdiv_rn(__uint_as_float(c.red[r]), 2688.0f) : 0.0f;
        b_block_store<W4A4>(*reinterpret_cast<const uint4*>(p), *reinterpret_cast<const uint4*>(p + 8), g,
                            reinterpret_cast<uint4*>(c.xq + (size_t)r * H + 16 * (i % nb)));
    }
    consumer_bar();
}

// ---------------------------------------------------------------- step 3
// z[t][e] = sum_i x[t][i] Wg[e][i] (FP32) for this CTA's experts e = b + j G.
// Returns false if the router rows never landed.
__device__ __noinline__ bool st_router(const StackArgs& a, StackCta& c, int l) {
    const int ctid = threadIdx.x, warp = ctid >> 5, lane = ctid & 31;
    const int T = a.T, H = a.H, E = a.E;
    const bool ok = mbar_wait_bounded(&c.gbar, static_cast<uint32_t>(l & 1));
    if (consumer_bar_or(!ok || cta_abort(c))) {
        if (ctid == 0 && !ok) set_dev_error(kErrWaitFull);
        return false;
    }
    float* z = a.ws.z + (size_t)l * T * E;
#pragma unroll 1
    for (int j = 0; j < c.ng; ++j) {
        const float4* w4 = reinterpret_cast<const float4*>(c.gsm + (size_t)j * H);
        float acc[kDecodeMaxT] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
        for (int i4 = ctid; i4 < H / 4; i4 += kConsumerThreads) {
            const float4 w = w4[i4];
#pragma unroll
            for (int t = 0; t < kDecodeMaxT; ++t) {
                if (t < T) {
                    const uint2 hv = *reinterpret_cast<const uint2*>(c.X + (size_t)t * H + 4 * i4);
                    acc[t] = fmaf(w.x, __uint_as_float(hv.x << 16), acc[t]);
                    acc[t] = fmaf(w.y, __uint_as_float(hv.x & 0xFFFF0000u), acc[t]);
                    acc[t] = fmaf(w.z, __uint_as_float(hv.y << 16), acc[t]);
                    acc[t] = fmaf(w.w, __uint_as_float(hv.y & 0xFFFF0000u), acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kDecodeMaxT; ++t) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) c.zred[warp][t] = v;
        }
        consumer_bar();
        if (ctid < T) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) s = __fadd_rn(s, c.zred[w][ctid]);
            z[(size_t)ctid * E + c.b + j * c.G] = s;
        }
        consumer_bar();
    }
    if (ctid == 0 && c.ng > 0) red_release_add(layer_cnt(a, l) + kCntLogits, c.ng);
    return true;
}

// ---------------------------------------------------------------- step 4
// Top-k by (sigma + bias desc, index asc) for every token, its gates
// sigma / sum(sigma), and the step plan. Every CTA computes the same result.
// One warp per token: lane l holds experts l, l + 32, ... as order-preserving
// 32-bit keys of sigma + bias; each of the k picks is a warp max of the key
// followed by a warp min of the index among the lanes that hold that key.
constexpr int kTopkPerLane = 8;  // E <= 256

__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // > 0 for every non-NaN value
}

__device__ __noinline__ void st_topk_plan(const StackArgs& a, StackCta& c, int l) {
    const int ctid = threadIdx.x, warp = ctid >> 5, lane = ctid & 31;
    const int T = a.T, E = a.E, k = a.k;
    if (ctid < 8) c.plan.bits[ctid] = 0u;
#pragma unroll 1
    for (int i = ctid; i < kDecodeMaxU * kDecodeMaxT; i += kConsumerThreads) {
        (&c.plan.choice[0][0])[i] = -1;
        (&c.plan.gate[0][0])[i] = 0.0f;
    }
    // sigma = 1 / (1 + exp(-z)) and the order key of sigma + bias, one
    // (token, expert) per thread
    uint32_t* const keys = reinterpret_cast<uint32_t*>(c.tk_c);
    const float* const z = a.ws.z + (size_t)l * T * E;
#pragma unroll 1
    for (int i = ctid; i < T * E; i += kConsumerThreads) {
        const float s = __frcp_rn(__fadd_rn(1.0f, expf(-__ldcg(z + i))));
        float v = __fadd_rn(s, c.bias_s[i % E]);
        if (v != v) v = -INFINITY;
        c.tk_s[i] = s;
        keys[i] = order_key(__fadd_rn(v, 0.0f));  // -0 and +0 compare equal
    }
    consumer_bar();
    if (warp < T) {
        const int t = warp;
        uint32_t key[kTopkPerLane];
        float sg[kTopkPerLane];
#pragma unroll
        for (int q = 0; q < kTopkPerLane; ++q) {
            const int e = lane + 32 * q;
            key[q] = e < E ? keys[t * E + e] : 0u;
            sg[q] = e < E ? c.tk_s[t * E + e] : 0.0f;
        }
        float ssum = 0.0f;
        for (int j = 0; j < k; ++j) {
            // this lane's best: largest key, then smallest index (smaller q)
            uint32_t bk = 0u;
            int bq = 0;
#pragma unroll
            for (int q = 0; q < kTopkPerLane; ++q)
                if (key[q] > bk) {
                    bk = key[q];
                    bq = q;
                }
            const uint32_t km = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t cand = (bk == km && bk != 0u) ? static_cast<uint32_t>(lane + 32 * bq) : 0xFFFFFFFFu;
            const int es = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
            const int qs = es >> 5;
            float mine = 0.0f;
#pragma unroll
            for (int q = 0; q < kTopkPerLane; ++q)
                if (q == qs) {
                    mine = sg[q];
                    if (lane == (es & 31)) key[q] = 0u;  // taken
                }
            const float sj = __shfl_sync(0xffffffffu, mine, es & 31);
            ssum = __fadd_rn(ssum, sj);
            if (lane == 0) {
                c.sel_idx[t][j] = es;
                c.sel_sig[t][j] = sj;
            }
        }
        __syncwarp();
        if (lane < k) {
            const float w = __fdiv_rn(c.sel_sig[t][lane], ssum);
            c.sel_w[t][lane] = w;
            if (c.b == 0) {
                a.topk_idx[((size_t)l * T + t) * k + lane] = c.sel_idx[t][lane];
                a.topk_w[((size_t)l * T + t) * k + lane] = w;
            }
        }
    }
    consumer_bar();
    if (ctid < T * k) {
        const int e = c.sel_idx[ctid / k][ctid % k];
        atomicOr(&c.plan.bits[e >> 5], 1u << (e & 31));
    }
    consumer_bar();
    if (ctid < T * k) {
        const int t = ctid / k, j = ctid % k;
        const int e = c.sel_idx[t][j];
        int slot = __popc(c.plan.bits[e >> 5] & ((1u << (e & 31)) - 1u));
#pragma unroll 1
        for (int w = 0; w < (e >> 5); ++w) slot += __popc(c.plan.bits[w]);
        c.plan.expert[slot] = e;
        c.plan.choice[slot][t] = static_cast<int8_t>(j);
        c.plan.gate[slot][t] = c.sel_w[t][j];
    }
    if (ctid == 0) {
        int u = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) u += __popc(c.plan.bits[w]);
        c.plan.U = u;
    }
    consumer_bar();
}

// The per-tensor globals of the layer's unique experts, from the staged
// arrays (before the producer may restage them for the next layer).
__device__ __noinline__ void st_layer_globals(StackCta& c) {
    const int ctid = threadIdx.x;
    if (ctid < c.plan.U) {
        c.up_g[ctid] = c.upg_s[c.plan.expert[ctid]];
        c.down_g[ctid] = c.dng_s[c.plan.expert[ctid]];
    }
    consumer_bar();
}

// ---------------------------------------------------------------- steps 5, 6
// Up tiles [base, base + n): shared (routed == false, tiles su_b + i) or
// routed (tiles i of the U x I/16 list from ru_b). relu^2 -> bf16 rows, row
// amax (W4A4), one count per finished tile. Returns false on a timeout.
template <bool W4A4>
__device__ __noinline__ bool st_up_tiles(const StackArgs& a, StackCta& c, int l, int base, int n, bool routed,
                                         int ru_b) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = a.T, k = a.k, H = a.H, I = a.I, S = a.S, RI = I >> 4;
    unsigned int* const amax = a.ws.amax + (size_t)(l & 1) * c.amax_stride;
    int* const cnt = layer_cnt(a, l);
    const __half* bcol = g < T ? c.xq + (size_t)g * H : nullptr;
    const int end = base + n;
#pragma unroll 1
    for (int li = first_item(base, warp % kGroups, kGroups); li < end; li += kGroups) {
        float acc[4];
        bool ok;
        const bool lead = bgroup_tile(c, li, H, bcol, acc, ok);
        if (!ok) return false;
        if (!lead) continue;
        int u = 0, r;
        if (routed) {
            const int i = ru_b + (li - base);
            u = i / RI;
            r = i % RI;
        } else {
            r = c.su_b + (li - base);
        }
        const float gw = routed ? c.up_g[u] : c.shu_g;
        float m[2] = {0.0f, 0.0f};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int t = 2 * q + (v & 1);
            if (t >= T) continue;
            const int j = routed ? c.plan.choice[u][t] : 0;
            if (j < 0) continue;
            const float gs = W4A4 ? __fmul_rn(gw, c.gx[t]) : gw;
            const float rl = fmaxf(__fmul_rn(acc[v], gs), 0.0f);
            const __nv_bfloat16 bv = __float2bfloat16_rn(__fmul_rn(rl, rl));
            const int row = 16 * r + g + 8 * (v >> 1);
            uint16_t* dst = routed ? a.ws.act + ((size_t)t * k + j) * I : a.ws.act_sh + (size_t)t * S;
            dst[row] = *reinterpret_cast<const uint16_t*>(&bv);
            m[v & 1] = fmaxf(m[v & 1], __bfloat162float(bv));
        }
        if (W4A4) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], o));
                m[1] = fmaxf(m[1], __shfl_xor_sync(0xffffffffu, m[1], o));
            }
            if (g == 0) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int t = 2 * q + p;
                    if (t >= T) continue;
                    if (routed) {
                        const int j = c.plan.choice[u][t];
                        if (j >= 0) atomicMax(amax + t * k + j, __float_as_uint(m[p]));
                    } else {
                        atomicMax(amax + T * k + t, __float_as_uint(m[p]));
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) red_release_add(cnt + (routed ? kCntUp + u : kCntShUp), 1);
    }
    return true;
}

// ---------------------------------------------------------------- step 7
// B operands of this CTA's down tiles: routed experts slot_u[0..1] ([T][I]
// each) and the shared expert ([T][S]), from the finished bf16 rows and their
// final row amax. Returns false if a wait failed.
template <bool W4A4>
__device__ __noinline__ bool st_down_operands(const StackArgs& a, StackCta& c, int l, int rd_b, int rd_e) {
    const int ctid = threadIdx.x;
    const int T = a.T, k = a.k, I = a.I, S = a.S, RI = I >> 4, RS = S >> 4, RH = a.H >> 4;
    const bool has_sd = c.sd_e > c.sd_b;
    int* const cnt = layer_cnt(a, l);
    const unsigned int* amax = a.ws.amax + (size_t)(l & 1) * c.amax_stride;
    if (ctid == 0) {
        c.slot_u[0] = c.slot_u[1] = -1;
        if (rd_e > rd_b) {
            c.slot_u[0] = rd_b / RH;
            const int u1 = (rd_e - 1) / RH;
            if (u1 != c.slot_u[0]) c.slot_u[1] = u1;
        }
    }
    consumer_bar();  // also: every up tile of this CTA is done, X / xq may be overwritten
    bool ok = true;
    if (ctid == 0 && has_sd) ok = wait_geq(cnt + kCntShUp, RS, abort_flag(a));
    if (ctid == 32 && c.slot_u[0] >= 0) ok = wait_geq(cnt + kCntUp + c.slot_u[0], RI, abort_flag(a));
    if (ctid == 64 && c.slot_u[1] >= 0) ok = wait_geq(cnt + kCntUp + c.slot_u[1], RI, abort_flag(a));
    if (consumer_bar_or(!ok || cta_abort(c))) return false;
    // one pass over the blocks of all rows: routed rows r = sl * T + t (slot
    // sl of this CTA, token t; [I] each), then the shared rows ([S] each).
    // Every thread reads its row's amax itself (no staging barrier) and keeps
    // up to kBRegBlocks blocks' loads in flight before quantising any.
    const int nbr = I >> 4, nbs = S >> 4;
    const int nr = 2 * T * nbr, total = nr + (has_sd ? T * nbs : 0);
    auto locate = [&](int i, const uint16_t*& src, const unsigned int*& am, __half*& dst, int& r, int& bb) {
        src = nullptr;
        am = nullptr;
        if (i < nr) {
            r = i / nbr;
            bb = i - r * nbr;
            const int sl = r / T, t = r - sl * T;
            dst = c.bslot + (size_t)r * I + 16 * bb;
            const int u = c.slot_u[sl];
            const int j = u >= 0 ? c.plan.choice[u][t] : -1;
            if (j >= 0) {
                src = a.ws.act + ((size_t)t * k + j) * I + 16 * bb;
                am = amax + t * k + j;
            }
        } else {
            const int i2 = i - nr, t = i2 / nbs;
            bb = i2 - t * nbs;
            r = 2 * T + t;
            dst = c.bslot + (size_t)2 * T * I + (size_t)t * S + 16 * bb;
            src = a.ws.act_sh + (size_t)t * S + 16 * bb;
            am = amax + T * k + t;
        }
    };
#pragma unroll 1
    for (int i0 = ctid; i0 < total; i0 += kBRegBlocks * kConsumerThreads) {
        uint4 u[kBRegBlocks][2];
        unsigned int mb[kBRegBlocks];
#pragma unroll
        for (int q = 0; q < kBRegBlocks; ++q) {
            const int i = i0 + q * kConsumerThreads;
            u[q][0] = u[q][1] = make_uint4(0, 0, 0, 0);
            mb[q] = 0u;
            if (i < total) {
                const uint16_t* src;
                const unsigned int* am;
                __half* dst;
                int r, bb;
                locate(i, src, am, dst, r, bb);
                if (src) {
                    u[q][0] = __ldcg(reinterpret_cast<const uint4*>(src));
                    u[q][1] = __ldcg(reinterpret_cast<const uint4*>(src) + 1);
                    if (W4A4) mb[q] = __ldcg(am);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kBRegBlocks; ++q) {
            const int i = i0 + q * kConsumerThreads;
            if (i >= total) break;
            const uint16_t* src;
            const unsigned int* am;
            __half* dst;
            int r, bb;
            locate(i, src, am, dst, r, bb);
            const float g = W4A4 ? __fdiv_rn(__uint_as_float(mb[q]), 2688.0f) : 0.0f;
            b_block_store<W4A4>(u[q][0], u[q][1], g, reinterpret_cast<uint4*>(dst));
            if (bb == 0) c.gbf[r] = g;  // the row's first block records its global
        }
    }
    consumer_bar();
    return true;
}

// The warp that completes output tile r of layer l: its 16 rows of
// h_{l+1} = bf16(((ysh + y_0) + y_1) + ... + y_{k-1} + h_l), FP32 in this order.
__device__ __noinline__ void combine_tile(const StackArgs& a, StackCta& c, int l, int r) {
    const int lane = threadIdx.x & 31;
    const int T = a.T, k = a.k, H = a.H;
    const uint16_t* res = l == 0 ? a.hidden_in : a.hidden_out + (size_t)(l - 1) * T * H;
    uint16_t* out = a.hidden_out + (size_t)l * T * H;
    // the next layer's row amax buffer starts at zero: its last readers (layer
    // l - 1) are done, and its first writers wait until every tile is final
    unsigned int* am = a.ws.amax + (size_t)((l + 1) & 1) * c.amax_stride;
#pragma unroll 1
    for (int i = lane; i < c.amax_stride; i += 32) am[i] = 0u;
#pragma unroll 1
    for (int o = lane; o < 16 * T; o += 32) {
        const int t = o >> 4, row = 16 * r + (o & 15);
        float y[kDecodeMaxK];
#pragma unroll
        for (int j = 0; j < kDecodeMaxK; ++j)
            if (j < k) y[j] = __ldcg(a.ws.ypart + ((size_t)t * k + j) * H + row);
        float acc = __ldcg(a.ws.ysh + (size_t)t * H + row);
        const float rv = bf16_bits_to_float(__ldcg(res + (size_t)t * H + row));
#pragma unroll
        for (int j = 0; j < kDecodeMaxK; ++j)
            if (j < k) acc = __fadd_rn(acc, y[j]);
        acc = __fadd_rn(acc, rv);
        const __nv_bfloat16 ob = __float2bfloat16_rn(acc);
        out[(size_t)t * H + row] = *reinterpret_cast<const uint16_t*>(&ob);
    }
    __syncwarp();
    if (lane == 0) red_release_add(layer_cnt(a, l) + kCntHDone, 1);
}

// ---------------------------------------------------------------- step 8
template <bool W4A4>
__device__ __noinline__ bool st_down_tiles(const StackArgs& a, StackCta& c, int l, int base, int rd_b, int n_rd) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = a.T, k = a.k, H = a.H, I = a.I, S = a.S, RH = H >> 4;
    const int n_sd = c.sd_e - c.sd_b;
    int* const cnt = layer_cnt(a, l);
    const int U = c.plan.U;
    const __half* bslot2 = c.bslot + (size_t)2 * T * I;
    const int end = base + n_sd + n_rd;
#pragma unroll 1
    for (int li = first_item(base, warp % kGroups, kGroups); li < end; li += kGroups) {
        const bool routed = li >= base + n_sd;
        int u = -1, r, sl, K;
        if (routed) {
            const int i = rd_b + (li - base - n_sd);
            u = i / RH;
            r = i % RH;
            sl = u == c.slot_u[0] ? 0 : (u == c.slot_u[1] ? 1 : -1);
            K = I;
        } else {
            r = c.sd_b + (li - base);
            sl = 2;
            K = S;
        }
        if (sl < 0 && lane == 0) set_dev_error(kErrBadInput);
        const __half* bs = sl == 2 ? bslot2 : c.bslot + (size_t)(sl < 0 ? 0 : sl) * T * I;
        const __half* bcol = nullptr;
        if (sl >= 0 && g < T && (!routed || c.plan.choice[u][g] >= 0)) bcol = bs + (size_t)g * K;
        float acc[4];
        bool ok;
        const bool lead = bgroup_tile(c, li, K, bcol, acc, ok);
        if (!ok) return false;
        if (!lead) continue;
        const float gw = routed ? c.down_g[u] : c.shd_g;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int t = 2 * q + (v & 1);
            const int row = 16 * r + g + 8 * (v >> 1);
            if (t >= T || sl < 0) continue;
            const float gs = W4A4 ? __fmul_rn(gw, c.gbf[sl * T + t]) : gw;
            const float y = __fmul_rn(acc[v], gs);
            if (routed) {
                const int j = c.plan.choice[u][t];
                if (j >= 0) a.ws.ypart[((size_t)t * k + j) * H + row] = __fmul_rn(c.plan.gate[u][t], y);
            } else {
                a.ws.ysh[(size_t)t * H + row] = y;
            }
        }
        // count this contribution to output tile r; the last one combines it
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atom_acq_rel_add(cnt + kCntTile + r, 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == U) {
            __syncwarp();  // lane 0's acquire orders the other lanes' loads too
            combine_tile(a, c, l, r);
        }
    }
    return true;
}

// ---------------------------------------------------------------- producer

// The producer is one thread among twelve busy warps, so its per-tile work is
// kept short: the ring position lives in registers (phys = vhead mod cap,
// advanced without divisions), the fill is inlined, and the routed tiles'
// addresses advance without divisions.
__device__ __noinline__ void st_producer(const StackArgs& a, StackCta& c) {
    const int H = a.H, I = a.I, S = a.S, RI = I >> 4, RH = H >> 4;
    const int G = c.G, b = c.b;
    BRing& r = c.br;
    const int cap = c.ring_cap;
    uint8_t* const rbase = c.ring_base;
    int pli = 0, tail = 0, vhead = 0, phys = 0;
    bool alive = true;
    // item pli: a 16-row tile of K columns (9 K bytes), placed after the
    // previous one (or at offset 0 if it would cross the end), once the item
    // that last used its slot and every older item whose bytes it overwrites
    // are released (waited for in issue order)
    auto fill = [&](const uint8_t* codes, const uint8_t* scales, int K) {
        if (!alive) return;
        if (cta_abort(c)) {
            alive = false;
            return;
        }
        const int size = 9 * K;
        if (phys + size > cap) {
            vhead += cap - phys;
            phys = 0;
        }
        const int lim = vhead + size - cap;
#pragma unroll 1
        while (tail < pli && (tail <= pli - kSlots || r.vs[tail & (kSlots - 1)] < lim)) {
            if (!mbar_wait_abortable(&r.empty[tail & (kSlots - 1)], static_cast<uint32_t>((tail / kSlots) & 1),
                                     &c.abort_s, kErrWaitEmpty)) {
                alive = false;
                set_cta_abort(c);
                return;
            }
            ++tail;
        }
        const int s = pli & (kSlots - 1);
        r.vs[s] = vhead;
        r.off[s] = static_cast<uint32_t>(phys);
        uint8_t* dst = rbase + phys;
        mbar_arrive_expect_tx(&r.full[s], static_cast<uint32_t>(size));
        bulk_g2s(dst, codes, static_cast<uint32_t>(8 * K), &r.full[s]);
        bulk_g2s(dst + 8 * K, scales, static_cast<uint32_t>(K), &r.full[s]);
        r.uses[s] += 1;
        vhead += size;
        phys += size;
        ++pli;
    };
    // router rows of this CTA's experts and the layer's bias (E * 4 bytes,
    // E % 8 == 0: a multiple of 16 bytes), on one barrier phase per layer
    auto issue_gate = [&](int l) {
        mbar_arrive_expect_tx(&c.gbar, (uint32_t)(c.ng * H * 4 + 3 * a.E * 4));
#pragma unroll 1
        for (int j = 0; j < c.ng; ++j)
            bulk_g2s(c.gsm + (size_t)j * H, a.layer[l].router_w + (size_t)(b + j * G) * H, (uint32_t)(H * 4),
                     &c.gbar);
        bulk_g2s(c.bias_s, a.layer[l].router_b, (uint32_t)(a.E * 4), &c.gbar);
        bulk_g2s(c.upg_s, a.layer[l].up_global, (uint32_t)(a.E * 4), &c.gbar);
        bulk_g2s(c.dng_s, a.layer[l].down_global, (uint32_t)(a.E * 4), &c.gbar);
        c.gate_issued += 1;
    };
    auto issue_shared_up = [&](int l) {
        const StackLayer& P = a.layer[l];
#pragma unroll 1
        for (int sr = c.su_b; sr < c.su_e; ++sr)
            fill(P.shu_codes + (size_t)16 * sr * (H >> 1), P.shu_scales + (size_t)16 * sr * (H >> 4), H);
    };
    issue_gate(0);
    issue_shared_up(0);
#pragma unroll 1
    for (int l = 0; l < a.L && alive; ++l) {
        if (!mbar_wait_abortable(&c.pbar, l & 1, &c.abort_s)) {
            set_cta_abort(c);
            break;
        }
        if (l + 1 < a.L) issue_gate(l + 1);
        const StackLayer& P = a.layer[l];
        const int NU = c.plan.U * RI, ND = c.plan.U * RH;
        {  // routed up tiles: tile rr of unique expert u
            const uint8_t* const uc = P.up_codes;
            const uint8_t* const us = P.up_scales;
            const int i0 = share_begin32(NU, b, G), n = share_begin32(NU, b + 1, G) - i0;
            int u = i0 / RI, rr = i0 - u * RI;
#pragma unroll 1
            for (int j = 0; j < n; ++j) {
                const int64_t row = (int64_t)c.plan.expert[u] * I + 16 * rr;
                fill(uc + row * (H >> 1), us + row * (H >> 4), H);
                if (++rr == RI) {
                    rr = 0;
                    ++u;
                }
            }
        }
#pragma unroll 1
        for (int sr = c.sd_b; sr < c.sd_e; ++sr)
            fill(P.shd_codes + (size_t)16 * sr * (S >> 1), P.shd_scales + (size_t)16 * sr * (S >> 4), S);
        {  // routed down tiles
            const uint8_t* const dc = P.down_codes;
            const uint8_t* const ds = P.down_scales;
            const int i0 = share_begin32(ND, b, G), n = share_begin32(ND, b + 1, G) - i0;
            int u = i0 / RH, rr = i0 - u * RH;
#pragma unroll 1
            for (int j = 0; j < n; ++j) {
                const int64_t row = (int64_t)c.plan.expert[u] * H + 16 * rr;
                fill(dc + row * (I >> 1), ds + row * (I >> 4), I);
                if (++rr == RH) {
                    rr = 0;
                    ++u;
                }
            }
        }
        mbar_arrive(&c.qbar);  // the plan of layer l is no longer read here
        if (l + 1 < a.L) issue_shared_up(l + 1);
    }
    if (!alive) atomicExch(abort_flag(a), 1);
}

// ---------------------------------------------------------------- consumers
template <bool W4A4>
__device__ __noinline__ void st_consumers(const StackArgs& a, StackCta& c) {
    const int ctid = threadIdx.x;
    const int T = a.T, E = a.E, H = a.H, I = a.I, RI = I >> 4, RH = H >> 4;
    const int G = c.G, b = c.b;
    int base = 0;  // first ring item of the current step
    bool bad = false;
#pragma unroll 1
    for (int l = 0; l < a.L; ++l) {
        int* const cnt = layer_cnt(a, l);
        // 1-2. the layer input, once every tile of it is final
        if (l > 0) {
            bool ok = true;
            if (ctid == 0) ok = wait_geq(layer_cnt(a, l - 1) + kCntHDone, RH, abort_flag(a));
            if (consumer_bar_or(!ok || cta_abort(c))) {
                bad = true;
                break;
            }
        }
        st_input<W4A4>(a, c, l == 0 ? a.hidden_in : a.hidden_out + (size_t)(l - 1) * T * H, l);
        // 3. router logits (the wait also covers the staged bias)
        if (!st_router(a, c, l)) {
            bad = true;
            break;
        }
        // 4. top-k and plan as soon as every logit is posted (and the producer
        // has stopped reading the previous plan), so that the routed weights
        // start streaming while this CTA still works on the shared tiles
        {
            bool ok = true;
            if (ctid == 0) ok = wait_geq(cnt + kCntLogits, E, abort_flag(a));
            if (l > 0 && !mbar_wait_abortable(&c.qbar, static_cast<uint32_t>((l - 1) & 1), &c.abort_s)) ok = false;
            if (consumer_bar_or(!ok || cta_abort(c))) {
                bad = true;
                break;
            }
        }
        st_topk_plan(a, c, l);
        st_layer_globals(c);
        if (ctid == 0) mbar_arrive(&c.pbar);  // the producer may stream the routed tiles now
        // 5. shared-expert up tiles (staged during the previous layer)
        const int n_su = c.su_e - c.su_b;
        if (!st_up_tiles<W4A4>(a, c, l, base, n_su, false, 0)) set_cta_abort(c);
        base += n_su;
        // 6. routed up tiles
        const int U = c.plan.U;
        const int NU = U * RI, ND = U * RH;
        const int ru_b = share_begin32(NU, b, G), ru_e = share_begin32(NU, b + 1, G);
        const int rd_b = share_begin32(ND, b, G), rd_e = share_begin32(ND, b + 1, G);
        if (!st_up_tiles<W4A4>(a, c, l, base, ru_e - ru_b, true, ru_b)) set_cta_abort(c);
        base += ru_e - ru_b;
        // 7. down operands
        if (!st_down_operands<W4A4>(a, c, l, rd_b, rd_e)) {
            bad = true;
            break;
        }
        // 8. down tiles, counted per output tile; the last contribution combines it
        if (!st_down_tiles<W4A4>(a, c, l, base, rd_b, rd_e - rd_b)) set_cta_abort(c);
        base += (c.sd_e - c.sd_b) + (rd_e - rd_b);
        if (consumer_bar_or(cta_abort(c))) {
            bad = true;
            break;
        }
    }
    if (bad && ctid == 0) {
        set_cta_abort(c);
        atomicExch(abort_flag(a), 1);
    }
}

template <bool W4A4>
__global__ void __launch_bounds__(kThreads, 1) k_moe_stack(const __grid_constant__ StackArgs args) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ StackCta c;
    // the steps read the arguments from a shared-memory copy: a kernel
    // parameter read through a reference in an out-of-line function is a
    // generic load several hundred cycles long, on every step's critical path
    __shared__ __align__(16) StackArgs a;
    static_assert(sizeof(StackArgs) % 4 == 0, "StackArgs copy");
    for (int i = threadIdx.x; i < (int)(sizeof(StackArgs) / 4); i += blockDim.x)
        reinterpret_cast<uint32_t*>(&a)[i] = reinterpret_cast<const uint32_t*>(&args)[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&c.br.full[s], 1);
            mbar_init(&c.br.empty[s], kGroupWarps);
            c.br.uses[s] = 0;
        }
        mbar_init(&c.gbar, 1);
        mbar_init(&c.pbar, 1);
        mbar_init(&c.qbar, 1);
        fence_mbar_init();
        c.abort_s = 0;
        c.gate_issued = 0;
        c.G = G;
        c.b = b;
        c.ring_cap = a.ring_cap;
        c.ng = b < a.E ? (a.E - b + G - 1) / G : 0;
        c.amax_stride = a.T * a.k + a.T;
        const int RS = a.S >> 4, RH = a.H >> 4;
        c.su_b = share_begin32(RS, b, G);
        c.su_e = share_begin32(RS, b + 1, G);
        c.sd_b = share_begin32(RH, b, G);
        c.sd_e = share_begin32(RH, b + 1, G);
        c.ring_base = smem;
        c.gsm = reinterpret_cast<float*>(smem + a.off_gate);
        c.X = reinterpret_cast<uint16_t*>(smem + a.off_uni);
        c.xq = reinterpret_cast<__half*>(smem + a.off_uni + (size_t)a.T * a.H * 2);
        c.bslot = reinterpret_cast<__half*>(smem + a.off_uni);
        c.tk_c = reinterpret_cast<float*>(smem + a.off_tk);
        c.tk_s = c.tk_c + (size_t)a.T * a.E;
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        if (lane == 0) st_producer(a, c);
    } else {
        st_consumers<W4A4>(a, c);
    }

    __syncthreads();
    // no bulk copy may still be landing in shared memory when the CTA exits
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s)
            if (c.br.uses[s] > 0 && !mbar_wait_bounded(&c.br.full[s], (c.br.uses[s] - 1) & 1))
                set_dev_error(kErrWaitDrain);
    }
    if (threadIdx.x == 0 && c.gate_issued > 0 && !mbar_wait_bounded(&c.gbar, (c.gate_issued - 1) & 1))
        set_dev_error(kErrWaitDrain);
    // the last CTA to leave resets the counters and the row amax for the next
    // call (from the kernel parameters: stores through the workspace pointers
    // would make every read of the shared copy a reload)
    const int ncnt = args.L * stack_cnt_per_layer(args.H);
    int* const cnt_exit = args.ws.cnt + ncnt;
    if (threadIdx.x == 0) {
        __threadfence();
        c.last_cta = atomicAdd(cnt_exit, 1) == G - 1;
    }
    __syncthreads();
    if (c.last_cta) {
        for (int i = threadIdx.x; i < ncnt; i += blockDim.x) args.ws.cnt[i] = 0;
        for (int i = threadIdx.x; i < 2 * (args.T * args.k + args.T); i += blockDim.x) args.ws.amax[i] = 0u;
        __syncthreads();
        if (threadIdx.x == 0) {
            cnt_exit[1] = 0;
            __threadfence();
            *cnt_exit = 0;
        }
    }
}

}  // namespace nvfp4moe
