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
//     1. wait until every CTA has written its share of h_l (counter); load h_l;
//     2. x = RMSNorm(h_l); B operand of the up tiles (NVFP4 in W4A4);
//     3. router logits of this CTA's experts (gate rows staged in shared
//        memory during the previous layer) -> workspace, count them;
//     4. wait for all E logits; sigmoid + bias top-k (rank per expert, every
//        CTA computes the same selection), the step plan (unique experts);
//        from here the producer streams the routed weights;
//     5. its units: a unit is 16 rows of one expert's intermediate dimension;
//        each CTA takes units of one expert (the shared expert's S/16 are
//        split over a fixed set of CTAs, each routed expert's I/16 over its
//        share of the others). Per unit, the up tile (16 rows of W_up) gives
//        16 intermediate values relu^2 -> bf16, kept in shared memory, and
//        their amax is posted per (expert, token) (W4A4);
//     6. count its up tiles on the expert's counter and wait (W4A4) until
//        all of them are done: the row amax, and with it the per-tensor
//        global of the intermediate row, is final. Quantise each unit's 16
//        values (one NVFP4 block) as a down B operand;
//     7. per unit, the matching 16 columns of W_down (all H rows; a
//        column-block copy of W_down keeps them contiguous) times the unit's
//        block: a split-K partial of the expert's output, accumulated raw in
//        registers and scaled once (gate x globals) into the CTA's FP32
//        partial of the layer output in the workspace; count it;
//     8. wait for every CTA's partial; add, for its share of the H rows, the
//        G partials in CTA order and the residual: h_{l+1} = bf16(sum + h_l).
//
// The down weights of a unit depend only on the plan, so they stream while
// the up tiles are still computing, and no intermediate row leaves the CTA
// that computed it: across CTAs only the per-row amax and the H-wide partial
// sums meet.
//
// One producer thread streams every tile the CTA owns through the staging
// ring in consumption order, and fills the next layer's constant tiles
// (router rows, shared-expert up tiles) as soon as stages free up, so they
// land while the current layer is still waiting on its dependencies.
// Every wait is bounded; a CTA that gives up sets the workspace abort flag,
// which ends every other CTA's waits, and the last CTA to leave clears it
// for the next call.
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
    const uint8_t* down_cb;  // [E][I/16][9 H] column blocks of W_down (layout below)
    const float* down_global;
    const uint8_t* shu_codes;  // [S][H/2]
    const uint8_t* shu_scales;
    const float* shu_global;
    const uint8_t* shd_cb;  // [S/16][9 H] column blocks of the shared W_down
    const float* shd_global;
    const float* router_w;  // [E][H]
    const float* router_b;  // [E]
};

// Control words of the workspace: the count of CTAs that have left, the
// abort flag, the epoch (completed calls).
constexpr int kCtlExit = 0, kCtlAbort = 1, kCtlEpoch = 2, kCtlWords = 3;

// Column-block layout of a down matrix W [H][C] (NVFP4, C the reduction
// dimension): block c holds columns [16 c, 16 c + 16) of every row, 9 H bytes:
// codes [H/32][32 lanes][8 B], then scales [H/32][8][4 B]. Within pair p (rows
// 32 p .. 32 p + 31, two 16-row MMA tiles m = 0, 1), lane 4 g + q holds, for
// tile m, bytes 4m .. 4m + 3: row 32p + 16m + g, columns 4q, 4q + 1 and 4q + 2,
// 4q + 3 (one E2M1 pair each, low nibble first), then the same for row
// 32p + 16m + g + 8; scale group g holds, for tile m, bytes 2m, 2m + 1: the
// block scales of rows 32p + 16m + g and 32p + 16m + g + 8. So each lane loads
// the A fragment of an m16n8k16 MMA with one 8-byte load per pair of tiles.
constexpr int kUnitRows = 16;
constexpr int kMaxUnits = 32;      // units per CTA and layer
constexpr int kDownMaxPairs = 8;   // 32-row pairs per consumer warp: H <= 12 x 8 x 32 = 3072

// Values that every CTA waits for carry the layer they belong to: a router
// logit is one 64-bit word {float bits, tag}, an element of a layer output one
// 32-bit word {bf16 bits, low 16 bits of the tag}, each written with a single
// store. A reader polls the words themselves until every tag is the current
// layer's, so one round trip to L2 both waits and reads (a count that
// publishes separate data costs a second one). tag = 32 epoch + l + 1, where
// the epoch word counts completed calls on this workspace: never 0 (the value
// of a zeroed workspace), and a word left by an earlier layer or call never
// carries the current tag.
struct StackWs {
    int* cnt;                // control words [kCtlWords]
    unsigned long long* zt;  // [L][T][E] tagged router logits
    unsigned int* hx;        // [T][H] tagged layer output (the next layer's input)
    unsigned long long* amx;   // [G][T] tagged amax of each CTA's intermediate values per token (W4A4)
    unsigned long long* part;  // [G][T][H] tagged per-CTA partials of the layer output
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
    int off_uact, off_ubq;          // per-unit intermediate values, per-unit down B operands
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u32(unsigned int* p, unsigned int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Poll-and-read of tagged words (StackWs), called after every poll that
// found a word not yet written: true (give up) if the wait expired (flags the
// error word and the abort flag) or the abort flag rose. Both are checked on
// the second poll and then every 16 (so that even a short wait sees a short
// limit set by nvfp4_set_peer_wait_limit).
__device__ __forceinline__ bool poll_give_up(unsigned long long& t0, int it, const int* abort_g) {
    if (it == 0) {
        t0 = globaltimer();
        return false;
    }
    if (it != 1 && (it & 15) != 0) return false;
    if (ld_acquire_gpu(abort_g)) return true;
    if (globaltimer() - t0 > g_peer_wait_ns) {
        set_dev_error(kErrWaitPeer);
        atomicExch(const_cast<int*>(abort_g), 1);
        return true;
    }
    return false;
}
// Eight consecutive bf16 elements of a tagged layer output -> out (packed).
__device__ __noinline__ bool poll_h8(const unsigned int* p, uint32_t tag16, uint4& out, const int* abort_g) {
    unsigned long long t0 = 0;
    for (int it = 0;; ++it) {
        const uint4 a = ld_relaxed_v4(p), b = ld_relaxed_v4(p + 4);
        const uint32_t hi = tag16 << 16;
        if (((a.x & 0xFFFF0000u) == hi) & ((a.y & 0xFFFF0000u) == hi) & ((a.z & 0xFFFF0000u) == hi) &
            ((a.w & 0xFFFF0000u) == hi) & ((b.x & 0xFFFF0000u) == hi) & ((b.y & 0xFFFF0000u) == hi) &
            ((b.z & 0xFFFF0000u) == hi) & ((b.w & 0xFFFF0000u) == hi)) {
            out = make_uint4((a.x & 0xFFFFu) | (a.y << 16), (a.z & 0xFFFFu) | (a.w << 16), (b.x & 0xFFFFu) | (b.y << 16),
                             (b.z & 0xFFFFu) | (b.w << 16));
            return true;
        }
        if (poll_give_up(t0, it, abort_g)) return false;
    }
}
// One tagged router logit.
__device__ __noinline__ bool poll_logit(const unsigned long long* p, uint32_t tag, float& out, const int* abort_g) {
    unsigned long long t0 = 0;
    for (int it = 0;; ++it) {
        const unsigned long long w = ld_relaxed_u64(p);
        if (static_cast<uint32_t>(w >> 32) == tag) {
            out = __uint_as_float(static_cast<uint32_t>(w));
            return true;
        }
        if (poll_give_up(t0, it, abort_g)) return false;
    }
}
__device__ __forceinline__ unsigned long long tagged_logit(float z, uint32_t tag) {
    return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(z);
}
__device__ __forceinline__ unsigned long long tagged_f32(float v, uint32_t tag) { return tagged_logit(v, tag); }

// Spins on the non-blocking test (the producer's hand-offs are on the
// critical path of every layer); gives up on the CTA abort flag or after 1 s.
__device__ __noinline__ bool mbar_wait_abortable(uint64_t* b, uint32_t parity, volatile int* abort_s,
                                                unsigned int err = kErrWaitFull) {
    if (mbar_test_wait(b, parity)) return true;  // no timer read when the phase is done
    const unsigned long long t0 = globaltimer();
    for (int it = 1;; ++it) {
        if (mbar_test_wait(b, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_s) return false;
            if (globaltimer() - t0 > kWaitTimeoutNs) {
                set_dev_error(err);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- phase trace
// Built with -DNVFP4MOE_TRACE, every CTA records the global timer at the
// phase boundaries of every layer (consumer thread 0 and the producer) into
// g_stack_trace[CTA][layer][event], read back by nvfp4moe_stack_trace_read.
// Without the flag the trace points compile to nothing.
enum StackTraceEvent : int {
    kTrStart = 0,    // layer begins (consumer)
    kTrHReady,       // thread 0 has read its elements of h_l (tagged words)
    kTrRouter,       // input, norm and this CTA's router logits posted
    kTrLogits,       // the producer has released the previous layer's plan
    kTrPlan,         // top-k and the plan of unique experts written
    kTrUp,           // this CTA's up tiles done
    kTrAmax,         // (W4A4) the expert's row amax final; down operands ready
    kTrDown,         // this CTA's down units done, partial posted
    kTrParts,        // every CTA's partial of this CTA's rows read
    kTrReduce,       // this CTA's rows of h_{l+1} written
    kTrProdFirst,    // producer: first item of the layer issued
    kTrProdLast,     // producer: last item of the layer issued
    kTrProdPlan,     // producer: the plan of the layer seen
    kTrEvents = 16
};
constexpr int kTraceMaxCtas = 256;
#if defined(NVFP4MOE_TRACE)
__device__ unsigned long long g_stack_trace[kTraceMaxCtas * kStackMaxLayers * kTrEvents];
#define STACK_TRACE(cond, b, l, ev)                                                                        \
    do {                                                                                                   \
        if ((cond) && (b) < kTraceMaxCtas) g_stack_trace[((b) * kStackMaxLayers + (l)) * kTrEvents + (ev)] = \
                                              globaltimer();                                               \
    } while (0)
#else
#define STACK_TRACE(cond, b, l, ev) \
    do {                            \
    } while (0)
#endif

// ---------------------------------------------------------------- staging ring
// A byte ring over the CTA's free shared memory. Items of 9 H bytes (an up
// tile: codes [16][H/2], then scales [16][H/16]; or a down column block) are
// placed one after another in issue order (an item that would cross the end
// starts again at offset 0), so that as many items are in flight as fit.
// Item li completes on full[li % kSlots]. Up items are computed by warp group
// li % kGroups (the consumer warps w with w % kGroups == li % kGroups), whose
// kGroupWarps warps each take a contiguous share of its 128-k chunks; down
// items by all consumer warps, each taking its own rows. Either way the
// consumers release an item on empty[li % kSlots] with kConsumerWarps arrivals
// in all (an up item's three warps arrive kGroups each). kSlots is a multiple
// of kGroups, so the same warps wait on every up use of a slot, in order, and
// every warp waits on a down item only once all of the layer's up items are
// consumed (a parity wait can only tell the current phase of an mbarrier from
// the one before it, so no warp may wait on use u of a slot before use u - 1
// has completed). The producer reclaims space in issue order: before placing
// an item it waits until the item that last used the slot, and every older
// item whose bytes the new one would overwrite, have been released.
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
    uint32_t tag0;  // tag of layer 0 of this call (StackWs)
    // geometry
    int G, b, ring_cap, ng;
    int cs;          // CTAs [0, cs) take the shared expert's units
    int ex, ub, ue;  // this layer's units of this CTA: expert (-1 shared, else slot), [ub, ue) of its units
    uint8_t* ring_base;
    float* gsm;      // [ng][H] router rows
    uint16_t* X;     // [T][H] h_l, then x_l
    __half* xq;      // [T][H] up B operand
    uint16_t* uact;  // [units][T][16] bf16 relu^2 values of this CTA's units
    __half* ubq;     // [units][T][16] their down B operands
    float* tk_c;     // [T][E] biased scores
    float* tk_s;     // [T][E] sigmoids
    // step scratch
    float norm_part[kDecodeMaxT][kNormMaxChunks];
    float norm_inv[kDecodeMaxT];
    float gx[kDecodeMaxT];
    unsigned int red[kDecodeMaxT];
    unsigned int amax_s[kDecodeMaxT];   // this CTA's intermediate values, max per token (W4A4)
    float fct[kDecodeMaxT];             // per token: gate x down global (x B global)
    float gb[kDecodeMaxT];              // per token: the down B global (W4A4)
    int sel_idx[kDecodeMaxT][kDecodeMaxK];
    float sel_sig[kDecodeMaxT][kDecodeMaxK];
    float sel_w[kDecodeMaxT][kDecodeMaxK];
    float zred[kConsumerWarps][kDecodeMaxT];
    float wmax[kConsumerWarps];
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
    if (lane == 0) mbar_arrive_cnt(&r.empty[s], kGroups);
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

__device__ __forceinline__ int* abort_flag(const StackArgs& a) { return a.ws.cnt + kCtlAbort; }
__device__ __forceinline__ int* epoch_word(const StackArgs& a) { return a.ws.cnt + kCtlEpoch; }

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
__device__ __noinline__ bool st_input(const StackArgs& a, StackCta& c, int l) {
    const int ctid = threadIdx.x, warp = ctid >> 5, lane = ctid & 31;
    const int T = a.T, H = a.H;
    uint16_t* X = c.X;
    if (ctid == kConsumerThreads - 1) {  // used by the epilogues later in the layer
        c.shu_g = __ldg(a.layer[l].shu_global);
        c.shd_g = __ldg(a.layer[l].shd_global);
    }
    bool ok = true;
    const uint32_t tag16 = (c.tag0 + l - 1) & 0xFFFFu;  // h_l is layer l - 1's output
#pragma unroll 1
    for (int i = 8 * ctid; i < T * H && ok; i += 8 * kConsumerThreads) {
        uint4 v;
        if (l == 0) v = __ldcg(reinterpret_cast<const uint4*>(a.hidden_in + i));
        else ok = poll_h8(a.ws.hx + i, tag16, v, abort_flag(a));
        *reinterpret_cast<uint4*>(X + i) = v;
    }
    STACK_TRACE(ctid == 0, c.b, l, kTrHReady);
    if (consumer_bar_or(!ok || cta_abort(c))) return false;
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
    // B operand: the row amax gives the row factor (W4A4 the global amax /
    // 2688, W4A16 the prescale 2^e), then each 16-block
    const int nb = H >> 4;
    {
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
    if (ctid < T) {
        const float amax = __uint_as_float(c.red[ctid]);
        c.gx[ctid] = W4A4 ? __fdiv_rn(amax, 2688.0f) : w4a16_row_scale(amax);
    }
#pragma unroll 1
    for (int i = ctid; i < T * nb; i += kConsumerThreads) {
        const int r = i / nb;
        const uint16_t* p = X + (size_t)r * H + 16 * (i % nb);
        const float amax = __uint_as_float(c.red[r]);
        const float g = W4A4 ? __fdiv_rn(amax, 2688.0f) : w4a16_row_inv_scale(amax);
        b_block_store<W4A4>(*reinterpret_cast<const uint4*>(p), *reinterpret_cast<const uint4*>(p + 8), g,
                            reinterpret_cast<uint4*>(c.xq + (size_t)r * H + 16 * (i % nb)));
    }
    consumer_bar();
    return true;
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
    unsigned long long* z = a.ws.zt + (size_t)l * T * E;
    const uint32_t tag = c.tag0 + l;
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
            st_relaxed_u64(z + (size_t)ctid * E + c.b + j * c.G, tagged_logit(s, tag));
        }
        consumer_bar();
    }
    return true;
}

constexpr int kT1MaxNg = 2;  // router rows per CTA on the one-token path

template <bool W4A4>
__device__ __noinline__ bool st_input_router_t1(const StackArgs& a, StackCta& c, int l) {
    const int ctid = threadIdx.x, warp = ctid >> 5, lane = ctid & 31;
    const int H = a.H, E = a.E;
    if (ctid == kConsumerThreads - 1) {  // used by the epilogues later in the layer
        c.shu_g = __ldg(a.layer[l].shu_global);
        c.shd_g = __ldg(a.layer[l].shd_global);
    }
    const int i = 8 * ctid;
    const bool mine = i < H;
    uint4 hv = make_uint4(0, 0, 0, 0);
    bool hok = true;
    if (mine) {
        if (l == 0) hv = __ldcg(reinterpret_cast<const uint4*>(a.hidden_in + i));
        else hok = poll_h8(a.ws.hx + i, (c.tag0 + l - 1) & 0xFFFFu, hv, abort_flag(a));  // layer l - 1's output
    }
    STACK_TRACE(ctid == 0, c.b, l, kTrHReady);
    uint32_t w[4] = {hv.x, hv.y, hv.z, hv.w};
    if (a.rms_eps > 0.0f) {
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float x0 = __uint_as_float(w[j] << 16), x1 = __uint_as_float(w[j] & 0xFFFF0000u);
            ss = __fmaf_rn(x0, x0, ss);
            ss = __fmaf_rn(x1, x1, ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        if (lane == 0) c.norm_part[0][warp] = ss;
        consumer_bar();
        // chunk sums in chunk order (all loaded first: nch <= 12 here)
        const int nch = (H + 255) >> 8;
        float part[kConsumerWarps];
#pragma unroll
        for (int ch = 0; ch < kConsumerWarps; ++ch) part[ch] = ch < nch ? c.norm_part[0][ch] : 0.0f;
        float sum = 0.0f;
#pragma unroll
        for (int ch = 0; ch < kConsumerWarps; ++ch)
            if (ch < nch) sum = __fadd_rn(sum, part[ch]);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, static_cast<float>(H)), a.rms_eps)));
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = bf16x2_rn(__fmul_rn(__uint_as_float(w[j] << 16), inv),
                             __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), inv));
    }
    // router partials of this thread's eight elements, the row amax
    const bool ok = mbar_wait_bounded(&c.gbar, static_cast<uint32_t>(l & 1));
    float zp[kT1MaxNg] = {0.0f, 0.0f};
    float mx = 0.0f;
    if (mine) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
        if (ok) {
#pragma unroll
            for (int r = 0; r < kT1MaxNg; ++r) {
                if (r < c.ng) {
                    const float4* g4 = reinterpret_cast<const float4*>(c.gsm + (size_t)r * H + i);
                    const float4 ga = g4[0], gb = g4[1];
                    const float gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        zp[r] = fmaf(gw[2 * j], __uint_as_float(w[j] << 16), zp[r]);
                        zp[r] = fmaf(gw[2 * j + 1], __uint_as_float(w[j] & 0xFFFF0000u), zp[r]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
        for (int r = 0; r < kT1MaxNg; ++r) zp[r] = __fadd_rn(zp[r], __shfl_xor_sync(0xffffffffu, zp[r], o));
    }
    if (lane == 0) {
        c.wmax[warp] = mx;
#pragma unroll
        for (int r = 0; r < kT1MaxNg; ++r) c.zred[warp][r] = zp[r];
    }
    if (consumer_bar_or(!ok || !hok || cta_abort(c))) {
        if (ctid == 0 && !ok) set_dev_error(kErrWaitFull);
        return false;
    }
    // the logits of this CTA's experts, warps added in order (first: every
    // CTA waits for them), by the last thread: its warp holds no input
    // elements when H <= 8 x 352, and warp 0 waits for the logits next
    if (ctid == kConsumerThreads - 1 && c.ng > 0) {
        unsigned long long* z = a.ws.zt + (size_t)l * E;
#pragma unroll 1
        for (int r = 0; r < c.ng; ++r) {
            float zw[kConsumerWarps];  // all loaded first, then added in warp order
#pragma unroll
            for (int ww = 0; ww < kConsumerWarps; ++ww) zw[ww] = c.zred[ww][r];
            float s = 0.0f;
#pragma unroll
            for (int ww = 0; ww < kConsumerWarps; ++ww) s = __fadd_rn(s, zw[ww]);
            st_relaxed_u64(z + c.b + r * c.G, tagged_logit(s, c.tag0 + l));
        }
    }
    // the B operand: each even lane quantises the 16-block it shares with the
    // next lane, under the row global amax / 2688 (W4A4), or converts it to
    // f16 under the row prescale (W4A16)
    float g = 0.0f;
    {
        float rm = 0.0f;
#pragma unroll
        for (int ww = 0; ww < kConsumerWarps; ++ww) rm = fmaxf(rm, c.wmax[ww]);
        g = W4A4 ? __fdiv_rn(rm, 2688.0f) : w4a16_row_inv_scale(rm);
        if (ctid == 0) c.gx[0] = W4A4 ? g : w4a16_row_scale(rm);
    }
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) p[j] = __shfl_down_sync(0xffffffffu, w[j], 1);
    if (mine && (lane & 1) == 0)
        b_block_store<W4A4>(make_uint4(w[0], w[1], w[2], w[3]), make_uint4(p[0], p[1], p[2], p[3]), g,
                            reinterpret_cast<uint4*>(c.xq + i));
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

__device__ __noinline__ bool st_topk_plan(const StackArgs& a, StackCta& c, int l) {
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
    const unsigned long long* const z = a.ws.zt + (size_t)l * T * E;
    bool ok = true;
#pragma unroll 1
    for (int i = ctid; i < T * E && ok; i += kConsumerThreads) {
        float zi = 0.0f;
        ok = poll_logit(z + i, c.tag0 + l, zi, abort_flag(a));
        const float s = __frcp_rn(__fadd_rn(1.0f, expf(-zi)));
        float v = __fadd_rn(s, c.bias_s[i % E]);
        if (v != v) v = -INFINITY;
        c.tk_s[i] = s;
        keys[i] = order_key(__fadd_rn(v, 0.0f));  // -0 and +0 compare equal
    }
    if (consumer_bar_or(!ok || cta_abort(c))) return false;
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
    if (ctid < kDecodeMaxT) c.amax_s[ctid] = 0u;
    consumer_bar();
    return true;
}

// Step 4 for one token: the sigmoids and keys as in st_topk_plan (one expert
// per thread), then warp 0 alone picks the top k, writes the plan (with one
// token the k picks are the unique experts; slot u holds the u-th smallest
// id, as in the general plan) and the unique experts' per-tensor globals; one
// CTA barrier publishes it (three fewer than the general plan and
// st_layer_globals).
__device__ __noinline__ bool st_topk_plan_t1(const StackArgs& a, StackCta& c, int l) {
    const int ctid = threadIdx.x, lane = ctid & 31;
    const int E = a.E, k = a.k;
    uint32_t* const keys = reinterpret_cast<uint32_t*>(c.tk_c);
    bool ok = true;
    if (ctid < E) {
        float zi = 0.0f;
        ok = poll_logit(a.ws.zt + (size_t)l * E + ctid, c.tag0 + l, zi, abort_flag(a));
        const float s = __frcp_rn(__fadd_rn(1.0f, expf(-zi)));
        float v = __fadd_rn(s, c.bias_s[ctid]);
        if (v != v) v = -INFINITY;
        c.tk_s[ctid] = s;
        keys[ctid] = order_key(__fadd_rn(v, 0.0f));  // -0 and +0 compare equal
    }
    if (consumer_bar_or(!ok || cta_abort(c))) return false;
    if (ctid < 32) {
        uint32_t key[kTopkPerLane];
        float sg[kTopkPerLane];
#pragma unroll
        for (int q = 0; q < kTopkPerLane; ++q) {
            const int e = lane + 32 * q;
            key[q] = e < E ? keys[e] : 0u;
            sg[q] = e < E ? c.tk_s[e] : 0.0f;
        }
        float ssum = 0.0f, my_s = 0.0f;
        int my_e = 0x7FFFFFFF;
#pragma unroll 1
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
            float pick = 0.0f;
#pragma unroll
            for (int q = 0; q < kTopkPerLane; ++q)
                if (q == qs) {
                    pick = sg[q];
                    if (lane == (es & 31)) key[q] = 0u;  // taken
                }
            const float sj = __shfl_sync(0xffffffffu, pick, es & 31);
            ssum = __fadd_rn(ssum, sj);
            if (lane == j) {
                my_e = es;
                my_s = sj;
            }
        }
        int slot = 0;
#pragma unroll 1
        for (int jj = 0; jj < k; ++jj)
            if (__shfl_sync(0xffffffffu, my_e, jj) < my_e) ++slot;
        if (lane < k) {
            const float wj = __fdiv_rn(my_s, ssum);
            if (c.b == 0) {
                a.topk_idx[(size_t)l * k + lane] = my_e;
                a.topk_w[(size_t)l * k + lane] = wj;
            }
            c.plan.expert[slot] = my_e;
#pragma unroll
            for (int t = 0; t < kDecodeMaxT; ++t) {
                c.plan.choice[slot][t] = static_cast<int8_t>(t == 0 ? lane : -1);
                c.plan.gate[slot][t] = t == 0 ? wj : 0.0f;
            }
            c.up_g[slot] = c.upg_s[my_e];
            c.down_g[slot] = c.dng_s[my_e];
        }
        if (lane < kDecodeMaxT) c.amax_s[lane] = 0u;
        __syncwarp();
        if (lane == 0) {
            c.plan.U = k;
            mbar_arrive(&c.pbar);  // the producer may stream the routed weights now (release: the plan is visible)
        }
    }
    consumer_bar();
    return true;
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

// ---------------------------------------------------------------- units
// Every CTA works on units of one expert per layer: the shared expert's RS
// units go evenly to CTAs [0, cs), the U routed experts' RI units each to the
// other Gr = G - cs CTAs, expert slot u to CTAs [cs + Gr u / U,
// cs + Gr (u + 1) / U), evenly. The shared CTAs' share does not depend on the
// routing, so their weights stream before the plan exists: cs is the fewest
// CTAs (from the even split G RS / (RS + Umax RI) down, Umax = min(T k, E))
// with which a shared CTA holds at most 1.5 units more than a routed CTA,
// RS / cs <= Umax RI / (G - cs) + 1.5 (at one token 32 of 152 CTAs, measured
// better than the even 38 and than 28; at four tokens the even 11). Every
// CTA and its producer compute the same ranges.
struct UnitRange {
    int ex, ub, ue;  // expert (-1 shared, else routed slot), units [ub, ue) of it
};

__host__ __device__ inline int stack_shared_ctas(int G, int RS, int RI, int Umax) {
    int cs = static_cast<int>((long long)G * RS / (RS + (long long)Umax * RI));
    cs = cs < 1 ? 1 : (cs > G - Umax ? G - Umax : cs);
    // 2 RS (G - c) <= c (2 Umax RI + 3 (G - c)): RS / c <= Umax RI / (G - c) + 1.5
    while (cs > 1 && 2LL * RS * (G - cs + 1) <= (long long)(cs - 1) * (2LL * Umax * RI + 3LL * (G - cs + 1))) --cs;
    return cs;
}

__device__ __forceinline__ UnitRange stack_units(int b, int G, int cs, int RS, int RI, int U) {
    UnitRange r;
    if (b < cs) {
        r.ex = -1;
        r.ub = RS * b / cs;
        r.ue = RS * (b + 1) / cs;
        return r;
    }
    const int Gr = G - cs, bb = b - cs;
    int u = bb * U / Gr;
    while (u > 0 && Gr * u / U > bb) --u;
    while (u + 1 < U && Gr * (u + 1) / U <= bb) ++u;
    const int c0 = Gr * u / U, nc = Gr * (u + 1) / U - c0;
    r.ex = u;
    r.ub = RI * (bb - c0) / nc;
    r.ue = RI * (bb - c0 + 1) / nc;
    return r;
}

// ---------------------------------------------------------------- step 5
// Up tiles [base, base + n): the CTA's units (of expert ex: -1 shared, else
// routed slot). relu^2 -> bf16 values of each unit (shared memory), their
// amax per (expert, token) (W4A4; counted once per CTA in step 6). Returns
// false on a timeout.
template <bool W4A4>
__device__ __noinline__ bool st_up_tiles(const StackArgs& a, StackCta& c, int l, int base, int n, int ex) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = a.T, H = a.H;
    const bool routed = ex >= 0;
    const int u = routed ? ex : 0;
    const __half* bcol = g < T ? c.xq + (size_t)g * H : nullptr;
    const int end = base + n;
#pragma unroll 1
    for (int li = first_item(base, warp % kGroups, kGroups); li < end; li += kGroups) {
        float acc[4];
        bool ok;
        const bool lead = bgroup_tile(c, li, H, bcol, acc, ok);
        if (!ok) return false;
        if (!lead) continue;
        const float gw = routed ? c.up_g[u] : c.shu_g;
        float m[2] = {0.0f, 0.0f};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int t = 2 * q + (v & 1);
            if (t >= T) continue;
            const int j = routed ? c.plan.choice[u][t] : 0;
            if (j < 0) continue;
            const float gs = __fmul_rn(gw, c.gx[t]);  // gx: W4A4 row global, W4A16 row prescale
            const float rl = fmaxf(__fmul_rn(acc[v], gs), 0.0f);
            const __nv_bfloat16 bv = __float2bfloat16_rn(__fmul_rn(rl, rl));
            c.uact[((size_t)(li - base) * T + t) * kUnitRows + g + 8 * (v >> 1)] =
                *reinterpret_cast<const uint16_t*>(&bv);
            m[v & 1] = fmaxf(m[v & 1], __bfloat162float(bv));
        }
        {  // the CTA's amax per token (the W4A4 row global; the W4A16 prescale)
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
                    if (!routed || c.plan.choice[u][t] >= 0) atomicMax(&c.amax_s[t], __float_as_uint(m[p]));
                }
            }
        }
    }
    return true;
}

// ---------------------------------------------------------------- step 6
// The down B operands of this CTA's units. It counts its up tiles on its
// expert's counter (one release, after the CTA barrier that orders every
// warp's amax updates before it); in W4A4 it then waits until every up tile
// of the expert is done, so that the intermediate row amax is final. Each
// (unit, token) block of 16 values is quantised under the row global
// amax / 2688 (W4A4) or converted to f16 (W4A16), and the factor per token
// gate x down global (x B global in W4A4) recorded; a token that does not
// route to the expert gets a zero block and factor. Returns false if a wait
// failed.
template <bool W4A4>
__device__ __noinline__ bool st_down_prep(const StackArgs& a, StackCta& c, int l) {
    const int ctid = threadIdx.x, warp = ctid >> 5, lane = ctid & 31;
    const int T = a.T;
    const int ex = c.ex, nu = c.ue - c.ub;
    const uint32_t tag = c.tag0 + l;
    consumer_bar();  // every up tile of this CTA is done
    // W4A4: post this CTA's amax per token as a tagged word, then poll the
    // words of every CTA of the expert: their max is the row amax, final
    if (W4A4 && ctid < T) st_relaxed_u64(a.ws.amx + (size_t)c.b * T + ctid, tagged_f32(__uint_as_float(c.amax_s[ctid]), tag));
    bool ok = true;
    if (warp < T) {
        const int t = warp;
        float gB = 0.0f;
        if (W4A4) {
            const int c0 = ex < 0 ? 0 : c.cs + (c.G - c.cs) * ex / c.plan.U;
            const int c1 = ex < 0 ? c.cs : c.cs + (c.G - c.cs) * (ex + 1) / c.plan.U;
            float m = 0.0f;
#pragma unroll 1
            for (int j = c0 + lane; j < c1 && ok; j += 32) {
                float v = 0.0f;
                ok = poll_logit(a.ws.amx + (size_t)j * T + t, tag, v, abort_flag(a));
                m = fmaxf(m, v);
            }
            ok = __all_sync(0xffffffffu, ok);
            gB = __fdiv_rn(warp_max(m), 2688.0f);
        }
        // W4A16: this CTA's own units convert under the prescale of their
        // amax (its partial carries the matching factor)
        const float pre = W4A4 ? gB : w4a16_row_scale(__uint_as_float(c.amax_s[t]));
        if (lane == 0) {
            int jj = 0;
            float gate = 1.0f, dg = c.shd_g;
            if (ex >= 0) {
                jj = c.plan.choice[ex][t];
                gate = c.plan.gate[ex][t];
                dg = c.down_g[ex];
            }
            float f = 0.0f;
            if (ok && jj >= 0 && nu > 0) f = __fmul_rn(gate, __fmul_rn(dg, pre));
            c.gb[t] = W4A4 ? gB : w4a16_row_inv_scale(__uint_as_float(c.amax_s[t]));
            c.fct[t] = f;
        }
    }
    if (consumer_bar_or(!ok || cta_abort(c))) return false;
#pragma unroll 1
    for (int i = ctid; i < nu * T; i += kConsumerThreads) {
        const int j = i / T, t = i - j * T;
        uint4 u0 = make_uint4(0, 0, 0, 0), u1 = make_uint4(0, 0, 0, 0);
        if (ex < 0 || c.plan.choice[ex][t] >= 0) {  // else the token's values were never written
            const uint4* src = reinterpret_cast<const uint4*>(c.uact + ((size_t)j * T + t) * kUnitRows);
            u0 = src[0];
            u1 = src[1];
        }
        b_block_store<W4A4>(u0, u1, c.gb[t], reinterpret_cast<uint4*>(c.ubq + ((size_t)j * T + t) * kUnitRows));
    }
    consumer_bar();
    return true;
}

// ---------------------------------------------------------------- step 7
// The down column blocks of this CTA's units (ring items base .. base + nu - 1),
// by every consumer warp: warp w takes the 32-row pairs [P w / 12,
// P (w + 1) / 12) of the H rows (P = H / 32) of every block. The raw products
// add up in registers (FP32; one expert, so one factor per token); the warp
// then writes factor x sum for its rows to the CTA's partial in the
// workspace, and the CTA counts it once every warp has. Returns false on a
// timeout.
__device__ __noinline__ bool st_down_units(const StackArgs& a, StackCta& c, int l, int base) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = a.T, H = a.H, P = H >> 5;
    const int p0 = P * warp / kConsumerWarps, np = P * (warp + 1) / kConsumerWarps - p0;
    const int nu = c.ue - c.ub;
    BRing& r = c.br;
    float acc[kDownMaxPairs][2][4];
#pragma unroll
    for (int p = 0; p < kDownMaxPairs; ++p)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[p][mt][v] = 0.0f;
    // one unit's products into acc: B (token g's block, elements 4q .. 4q + 3,
    // the MMA's k-slots 2q, 2q + 1, 2q + 8, 2q + 9 in the order the block's
    // layout gives the weights) times this warp's rows of block blk
    auto unit_mma = [&](const uint8_t* blk, uint2 bv) {
        const uint8_t* cw = blk + (size_t)p0 * 256 + lane * 8;
        const uint8_t* sw = blk + (size_t)8 * H + (size_t)p0 * 32 + g * 4;
#pragma unroll
        for (int p = 0; p < kDownMaxPairs; ++p) {
            if (p >= np) break;
            const uint2 w = *reinterpret_cast<const uint2*>(cw + p * 256);
            const uint32_t sc = *reinterpret_cast<const uint32_t*>(sw + p * 32);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint32_t s2 = e4m3x2_to_f16x2(mt ? sc >> 16 : sc);  // rows g (low), g + 8
                const uint32_t sa = bcast_lo(s2), sb = bcast_hi(s2);
                uint32_t f[4];
                e2m1x8_to_f16x8(mt ? w.y : w.x, f);
                mma_16816(acc[p][mt], hmul2(f[0], sa), hmul2(f[2], sb), hmul2(f[1], sa), hmul2(f[3], sb), bv.x,
                          bv.y);
            }
        }
    };
    auto b_of = [&](int j) {
        return g < T ? *reinterpret_cast<const uint2*>(c.ubq + ((size_t)j * T + g) * kUnitRows + 4 * q)
                     : make_uint2(0u, 0u);
    };
    // two units per round: their waits, loads and MMAs overlap
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < nu; j += 2) {
        const bool two = j + 1 < nu;
        const int li0 = base + j, s0 = li0 % kSlots, s1 = (li0 + 1) % kSlots;
        bool waited = mbar_wait_bounded(&r.full[s0], static_cast<uint32_t>((li0 / kSlots) & 1));
        if (two && waited) waited = mbar_wait_bounded(&r.full[s1], static_cast<uint32_t>(((li0 + 1) / kSlots) & 1));
        const bool got = __all_sync(0xffffffffu, waited);
        if (got) {
            const uint2 b0 = b_of(j);
            unit_mma(c.ring_base + r.off[s0], b0);
            if (two) unit_mma(c.ring_base + r.off[s1], b_of(j + 1));
        } else if (lane == 0) {
            set_dev_error(kErrWaitFull);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&r.empty[s0]);
            if (two) mbar_arrive(&r.empty[s1]);
        }
        if (!got) {
            ok = false;
            break;
        }
    }
    // factor x sum -> this CTA's partial: lane (g, q) holds rows g, g + 8 of
    // each 16-row tile for tokens 2q, 2q + 1
    const bool t0 = 2 * q < T, t1 = 2 * q + 1 < T;
    const float f0 = t0 ? c.fct[2 * q] : 0.0f, f1 = t1 ? c.fct[2 * q + 1] : 0.0f;
    unsigned long long* const d0 = a.ws.part + ((size_t)c.b * T + 2 * q) * H + 32 * p0 + g;
    unsigned long long* const d1 = d0 + H;
    const uint32_t tag = c.tag0 + l;
#pragma unroll
    for (int p = 0; p < kDownMaxPairs; ++p) {
        if (p >= np) break;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int o = 32 * p + 16 * mt + 8 * (v >> 1);
                if (v & 1) {
                    if (t1) st_relaxed_u64(d1 + o, tagged_f32(__fmul_rn(f1, acc[p][mt][v]), tag));
                } else if (t0) {
                    st_relaxed_u64(d0 + o, tagged_f32(__fmul_rn(f0, acc[p][mt][v]), tag));
                }
            }
    }
    if (consumer_bar_or(!ok || cta_abort(c))) return false;
    return true;
}

// ---------------------------------------------------------------- step 8
// This CTA's rows [h0, h1) of h_{l+1}, once every CTA's partial is written:
// the G partials of a (token, row) are split into chunks of kPartChunk
// consecutive CTAs; thread i takes chunk i / (T nr) of item i % (T nr), adds
// its partials in CTA order (all its loads in flight at once), and the chunk
// sums are added in chunk order; then the residual h_l; then bf16. CTA 0 also
// clears the row amax buffer of layer l + 1 (its last readers, the down steps
// of layer l - 1, are done; its first writers wait for this layer's rows).
// Returns false if the wait failed.
constexpr int kPartChunk = 8;

__device__ __noinline__ bool st_reduce(const StackArgs& a, StackCta& c, int l) {
    const int ctid = threadIdx.x;
    const int T = a.T, H = a.H, G = c.G;
    const uint16_t* res = l == 0 ? a.hidden_in : a.hidden_out + (size_t)(l - 1) * T * H;
    uint16_t* out = a.hidden_out + (size_t)l * T * H;
    const int h0 = share_begin32(H, c.b, G), nr = share_begin32(H, c.b + 1, G) - h0;
    const int items = T * nr, nch = (G + kPartChunk - 1) / kPartChunk;
    float resv = 0.0f;  // the residual of item ctid (final since the layer began), loaded early
    if (ctid < items) {
        const int t = ctid / nr, row = h0 + ctid - t * nr;
        resv = bf16_bits_to_float(__ldcg(res + (size_t)t * H + row));
    }
    // the chunk sums, [chunk][item], over the (dead) layer input and up B
    // operand: T nr nch <= T (H/G + 1)(G/8 + 1) floats, within their T H;
    // the partials are tagged words, polled until every one is this layer's
    bool ok = true;
    const uint32_t tag = c.tag0 + l;
    float* const csum = reinterpret_cast<float*>(c.X);
#pragma unroll 1
    for (int i = ctid; i < items * nch && ok; i += kConsumerThreads) {
        const int ch = i / items, it = i - ch * items;
        const int t = it / nr, row = h0 + it - t * nr;
        const unsigned long long* src = a.ws.part + (size_t)t * H + row + (size_t)kPartChunk * ch * T * H;
        const int n = min(kPartChunk, G - kPartChunk * ch);
        float v[kPartChunk];
        unsigned long long t0 = 0;
        for (int it2 = 0;; ++it2) {
            unsigned long long w[kPartChunk];
#pragma unroll
            for (int j = 0; j < kPartChunk; ++j) w[j] = j < n ? ld_relaxed_u64(src + (size_t)j * T * H) : 0ull;
            bool all = true;
#pragma unroll
            for (int j = 0; j < kPartChunk; ++j) {
                all = all && (j >= n || static_cast<uint32_t>(w[j] >> 32) == tag);
                v[j] = j < n ? __uint_as_float(static_cast<uint32_t>(w[j])) : 0.0f;
            }
            if (all) break;
            if (poll_give_up(t0, it2, abort_flag(a))) {
                ok = false;
                break;
            }
        }
        float s = v[0];
#pragma unroll
        for (int j = 1; j < kPartChunk; ++j) s = __fadd_rn(s, v[j]);
        csum[ch * items + it] = s;
    }
    STACK_TRACE(ctid == 0, c.b, l, kTrParts);
    if (consumer_bar_or(!ok || cta_abort(c))) return false;
    if (ctid < items) {
        const int t = ctid / nr, row = h0 + ctid - t * nr;
        float s = csum[ctid];
#pragma unroll 1
        for (int ch = 1; ch < nch; ++ch) s = __fadd_rn(s, csum[ch * items + ctid]);
        const float h = __fadd_rn(s, resv);
        const __nv_bfloat16 ob = __float2bfloat16_rn(h);
        const uint32_t bits = *reinterpret_cast<const uint16_t*>(&ob);
        out[(size_t)t * H + row] = static_cast<uint16_t>(bits);
        if (l + 1 < a.L) st_relaxed_u32(a.ws.hx + (size_t)t * H + row, bits | (((c.tag0 + l) & 0xFFFFu) << 16));
    }
    consumer_bar();
    return true;
}

// ---------------------------------------------------------------- producer
// Per layer l the items go out in the order the consumers take them: the up
// tiles of the CTA's units, then their down column blocks; a shared-expert
// CTA issues them before the plan of layer l exists (right after the plan of
// layer l - 1, so they stream while that layer finishes), a routed CTA once
// the plan is posted. All items are 9 H bytes. The producer is one thread
// among twelve busy warps, so its per-item work is kept short: the ring
// position lives in registers (phys = vhead mod cap, advanced without
// divisions) and all items go through one fill site.
__device__ __noinline__ void st_producer(const StackArgs& a, StackCta& c) {
    const int H = a.H, I = a.I, RI = I >> 4;
    const int G = c.G, b = c.b;
    BRing& r = c.br;
    const int cap = c.ring_cap, size = 9 * H;
    uint8_t* const rbase = c.ring_base;
    int pli = 0, tail = 0, vhead = 0, phys = 0;
    bool alive = true;
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
    issue_gate(0);
    const int RS = a.S >> 4;
    const bool sh = b < c.cs;  // a shared-expert CTA: its units do not depend on the plan
#pragma unroll 1
    for (int l = 0; l < a.L && alive; ++l) {
        const StackLayer& P = a.layer[l];
#pragma unroll 1
        for (int ph = 0; ph < 2 && alive; ++ph) {
            if (ph == 1 && !mbar_wait_abortable(&c.pbar, l & 1, &c.abort_s)) {  // the plan of layer l
                set_cta_abort(c);
                alive = false;
                break;
            }
            STACK_TRACE(ph == 1, b, l, kTrProdPlan);
            if ((ph == 0) != sh) continue;
            // the units' up tiles (16 rows of W_up: codes, then scales, from
            // two arrays), then their down column blocks (codes, then scales,
            // contiguous)
            const UnitRange ur = stack_units(b, G, c.cs, RS, RI, sh ? 1 : c.plan.U);
            const int n = ur.ue - ur.ub;
            const int64_t e = sh ? 0 : c.plan.expert[ur.ex];
#pragma unroll 1
            for (int it = 0; it < 2 * n; ++it) {
                const bool up = it < n;
                const int rr = ur.ub + (up ? it : it - n);
                const uint8_t *src_c, *src_s;
                if (up) {
                    const int64_t row = e * I + 16 * rr;
                    src_c = (sh ? P.shu_codes : P.up_codes) + row * (H >> 1);
                    src_s = (sh ? P.shu_scales : P.up_scales) + row * (H >> 4);
                } else {
                    src_c = (sh ? P.shd_cb : P.down_cb) + (e * RI + rr) * size;
                    src_s = src_c + 8 * H;
                }
                // item pli goes after the previous one, or at offset 0 if it
                // would cross the end, once the item that last used its slot
                // and every older item whose bytes it overwrites are released
                // (waited for in issue order)
                if (cta_abort(c)) {
                    alive = false;
                    break;
                }
                if (phys + size > cap) {
                    vhead += cap - phys;
                    phys = 0;
                }
                const int lim = vhead + size - cap;
#pragma unroll 1
                while (tail < pli && (tail <= pli - kSlots || r.vs[tail & (kSlots - 1)] < lim)) {
                    if (!mbar_wait_abortable(&r.empty[tail & (kSlots - 1)],
                                             static_cast<uint32_t>((tail / kSlots) & 1), &c.abort_s, kErrWaitEmpty)) {
                        alive = false;
                        set_cta_abort(c);
                        break;
                    }
                    ++tail;
                }
                if (!alive) break;
                STACK_TRACE(it == 0, b, l, kTrProdFirst);
                STACK_TRACE(it == 2 * n - 1, b, l, kTrProdLast);
                const int s = pli & (kSlots - 1);
                r.vs[s] = vhead;
                r.off[s] = static_cast<uint32_t>(phys);
                uint8_t* dst = rbase + phys;
                mbar_arrive_expect_tx(&r.full[s], static_cast<uint32_t>(size));
                bulk_g2s(dst, src_c, static_cast<uint32_t>(8 * H), &r.full[s]);
                bulk_g2s(dst + 8 * H, src_s, static_cast<uint32_t>(H), &r.full[s]);
                r.uses[s] += 1;
                vhead += size;
                phys += size;
                ++pli;
            }
        }
        // the next layer's router rows, once this layer's weights are on their
        // way (they are needed a layer later)
        if (alive && l + 1 < a.L) issue_gate(l + 1);
        if (alive) mbar_arrive(&c.qbar);  // the plan of layer l is no longer read here
    }
    if (!alive) atomicExch(abort_flag(a), 1);
}

// ---------------------------------------------------------------- consumers
template <bool W4A4>
__device__ __noinline__ void st_consumers(const StackArgs& a, StackCta& c) {
    const int ctid = threadIdx.x;
    const int T = a.T, H = a.H, I = a.I, RI = I >> 4;
    const int G = c.G, b = c.b;
    int base = 0;  // first ring item of the current step
    bool bad = false;
    const bool one_token = T == 1 && H <= 8 * kConsumerThreads && c.ng <= kT1MaxNg;
#pragma unroll 1
    for (int l = 0; l < a.L; ++l) {
        STACK_TRACE(ctid == 0, b, l, kTrStart);
        // 1-2. the layer input (tagged words: the read waits until every CTA's
        // rows of it are final)
        if (one_token) {  // 1-3 for one token from registers
            if (!st_input_router_t1<W4A4>(a, c, l)) {
                bad = true;
                break;
            }
        } else {
            if (!st_input<W4A4>(a, c, l)) {
                bad = true;
                break;
            }
            // 3. router logits (the wait also covers the staged bias)
            if (!st_router(a, c, l)) {
                bad = true;
                break;
            }
        }
        STACK_TRACE(ctid == 0, b, l, kTrRouter);
        // 4. top-k and plan (the logits are tagged words: the read waits until
        // all are posted) once the producer has stopped reading the previous
        // plan, so that the routed weights start streaming while this CTA
        // still works on the shared tiles
        {
            bool ok = true;
            if (l > 0 && !mbar_wait_abortable(&c.qbar, static_cast<uint32_t>((l - 1) & 1), &c.abort_s)) ok = false;
            if (consumer_bar_or(!ok || cta_abort(c))) {
                bad = true;
                break;
            }
        }
        STACK_TRACE(ctid == 0, b, l, kTrLogits);
        if (one_token) {
            if (!st_topk_plan_t1(a, c, l)) {
                bad = true;
                break;
            }
        } else {
            if (!st_topk_plan(a, c, l)) {
                bad = true;
                break;
            }
            st_layer_globals(c);
        }
        if (ctid == 0 && !one_token) mbar_arrive(&c.pbar);  // the producer may stream the routed weights now
        STACK_TRACE(ctid == 0, b, l, kTrPlan);
        // 5. up tiles of this CTA's units (one expert)
        const UnitRange ur = stack_units(b, G, c.cs, a.S >> 4, RI, c.plan.U);
        const int nu = ur.ue - ur.ub;
        if (ctid == 0) {  // read after the barrier that opens step 6
            c.ex = ur.ex;
            c.ub = ur.ub;
            c.ue = ur.ue;
        }
        if (!st_up_tiles<W4A4>(a, c, l, base, nu, ur.ex)) set_cta_abort(c);
        STACK_TRACE(ctid == 0, b, l, kTrUp);
        base += nu;
        // 6. the units' down B operands
        if (!st_down_prep<W4A4>(a, c, l)) {
            bad = true;
            break;
        }
        STACK_TRACE(ctid == 0, b, l, kTrAmax);
        // 7. the units' down column blocks -> this CTA's partial
        if (!st_down_units(a, c, l, base)) {
            bad = true;
            break;
        }
        STACK_TRACE(ctid == 0, b, l, kTrDown);
        base += nu;
        // 8. this CTA's rows of h_{l+1}
        if (!st_reduce(a, c, l)) {
            bad = true;
            break;
        }
        STACK_TRACE(ctid == 0, b, l, kTrReduce);
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
            mbar_init(&c.br.empty[s], kConsumerWarps);
            c.br.uses[s] = 0;
        }
        mbar_init(&c.gbar, 1);
        mbar_init(&c.pbar, 1);
        mbar_init(&c.qbar, 1);
        fence_mbar_init();
        c.abort_s = 0;
        c.gate_issued = 0;
        c.tag0 = 32u * static_cast<uint32_t>(__ldcg(epoch_word(a))) + 1u;
        c.G = G;
        c.b = b;
        c.ring_cap = a.ring_cap;
        c.ng = b < a.E ? (a.E - b + G - 1) / G : 0;
        const int RS = a.S >> 4;
        c.cs = stack_shared_ctas(G, RS, a.I >> 4, min(a.T * a.k, a.E));
        c.ex = c.ub = c.ue = 0;
        c.ring_base = smem;
        c.gsm = reinterpret_cast<float*>(smem + a.off_gate);
        c.X = reinterpret_cast<uint16_t*>(smem + a.off_uni);
        c.xq = reinterpret_cast<__half*>(smem + a.off_uni + (size_t)a.T * a.H * 2);
        c.uact = reinterpret_cast<uint16_t*>(smem + a.off_uact);
        c.ubq = reinterpret_cast<__half*>(smem + a.off_ubq);
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
    // the last CTA to leave clears the abort flag and the exit count and
    // advances the epoch for the next call (from the kernel parameters:
    // stores through the workspace pointers would make every read of the
    // shared copy a reload)
    int* const ctl = args.ws.cnt;
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(ctl + kCtlExit, 1) == G - 1) {
            ctl[kCtlAbort] = 0;
            ctl[kCtlEpoch] += 1;  // the next call's tags differ from every word this one wrote
            __threadfence();
            ctl[kCtlExit] = 0;
        }
    }
}

}  // namespace nvfp4moe
