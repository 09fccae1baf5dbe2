// moe_grouped.cuh - moe_expert_forward for more than 4 tokens (prefill and
// high-concurrency decode: "Let's optimize Nemotron 3.5 Lightning - a
// worklog", Step 3, where the routed experts run as a grouped FP4 GEMM over
// the tokens each expert received).
//
//   k_permute      (token, choice) pairs grouped by expert, stable in pair
//                  order: offsets [E+1], per-expert 64-position tile offsets,
//                  perm (position -> pair) and inv (pair -> position)
//   k_prep_rows    B operand rows: bf16 rows (optionally RMS-normalised) ->
//                  exact f16 values, NVFP4-quantised per row in W4A4
//   k_grouped      one GEMM over ragged groups: CTA tile = 64 weight rows x
//                  64 positions, K in 128-element chunks staged with cp.async;
//                  each warp decodes its 16 rows once per chunk and applies
//                  them to 4 column blocks of 8 positions (the up epilogue is
//                  relu^2 -> bf16 + row amax, the down epilogue the gate-
//                  weighted FP32 partial row)
//   k_combine      out = bf16(shared + sum_j y_j + residual), fixed order
//
// The shared expert is one more group (all tokens, identity order).
#pragma once

#include "gemv_tile.cuh"

namespace nvfp4moe {

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kGTile = 64;  // positions per n-tile and weight rows per m-tile
constexpr int kGThreads = 256;

// ---------------------------------------------------------------- permute
// offsets[e] = first position of expert e; positions of one expert keep the
// pairs' order (t * k + j ascending). tiles[e] = first 64-position n-tile of
// expert e and chunks[e] the first 128-position chunk (tiles[E], chunks[E] =
// their totals; either is skipped when null). Expert ids outside [0, E) are
// counted as expert 0 and flagged in the error word.
//
// One CTA; warp w owns the contiguous pairs [w seg, (w + 1) seg). Three
// steps with a barrier after each: every warp counts its pairs per expert;
// per expert the warps' counts become their first positions (an exclusive
// prefix over warps, then the experts' offsets by a warp scan); every warp
// places its pairs in order, 32 at a time (match_any gives each lane its rank
// among the lanes of its expert, the expert's leader advances the warp's
// running position). So the order of equal experts is the pair order.
__global__ void __launch_bounds__(kPermThreads) k_permute(const int32_t* __restrict__ idx, int P, int E,
                                                          int32_t* __restrict__ offsets, int32_t* __restrict__ tiles,
                                                          int32_t* __restrict__ chunks, int32_t* __restrict__ perm,
                                                          int32_t* __restrict__ inv) {
    __shared__ int wpos[kPermWarps][256];  // per warp and expert: its count, then its next position
    __shared__ int first[256];             // per expert: its first position
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < kPermWarps * 256; i += kPermThreads) (&wpos[0][0])[i] = 0;
    __syncthreads();
    auto expert_of = [&](int p) {
        int e = __ldg(idx + p);
        if (e < 0 || e >= E) {
            set_dev_error(kErrBadInput);
            e = 0;
        }
        return e;
    };
    const int seg = (P + kPermWarps - 1) / kPermWarps;
    const int s0 = min(P, warp * seg), s1 = min(P, s0 + seg);
    for (int p = s0 + lane; p < s1; p += 32) atomicAdd(&wpos[warp][expert_of(p)], 1);
    __syncthreads();
    // per expert: the warps' counts -> their positions relative to the expert's first
    for (int e = tid; e < E; e += kPermThreads) {
        int run = 0;
        for (int w = 0; w < kPermWarps; ++w) {
            const int c = wpos[w][e];
            wpos[w][e] = run;
            run += c;
        }
        first[e] = run;  // the expert's count for now
    }
    __syncthreads();
    if (warp == 0) {  // offsets, tiles, chunks: exclusive scans over the experts, 8 per lane
        int cnt[8], ls = 0, lt = 0, lc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 8 * lane + i;
            cnt[i] = e < E ? first[e] : 0;
            ls += cnt[i];
            lt += (cnt[i] + kGTile - 1) / kGTile;
            lc += (cnt[i] + 127) / 128;
        }
        int xs = ls, xt = lt, xc = lc;  // inclusive warp scans
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, xs, o), b = __shfl_up_sync(0xffffffffu, xt, o),
                      d = __shfl_up_sync(0xffffffffu, xc, o);
            if (lane >= o) {
                xs += a;
                xt += b;
                xc += d;
            }
        }
        int off = xs - ls, toff = xt - lt, coff = xc - lc;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 8 * lane + i;
            if (e < E) {
                offsets[e] = off;
                if (tiles) tiles[e] = toff;
                if (chunks) chunks[e] = coff;
                first[e] = off;
            }
            off += cnt[i];
            toff += (cnt[i] + kGTile - 1) / kGTile;
            coff += (cnt[i] + 127) / 128;
        }
        if (lane == 31) {
            offsets[E] = off;
            if (tiles) tiles[E] = toff;
            if (chunks) chunks[E] = coff;
        }
    }
    __syncthreads();
    for (int p0 = s0; p0 < s1; p0 += 32) {
        const int p = p0 + lane;
        const bool valid = p < s1;
        const int e = valid ? expert_of(p) : -1;
        const unsigned act = __ballot_sync(0xffffffffu, valid);
        unsigned peers = 0;
        int lrank = 0;
        if (valid) {
            peers = __match_any_sync(act, e);
            lrank = __popc(peers & ((1u << lane) - 1u));
            const int pos = first[e] + wpos[warp][e] + lrank;
            perm[pos] = p;
            inv[p] = pos;
        }
        __syncwarp();
        if (valid && lrank == 0) wpos[warp][e] += __popc(peers);
        __syncwarp();
    }
}

// ---------------------------------------------------------------- operand rows
// One CTA per row: src bf16 row r [K] -> dst f16 row r [K] with exact values; W4A4 quantises with the row's global
// (g = amax / 2688, amax given in amax_bits[r] or computed here) and writes
// it to gout[r]. rms_eps > 0 normalises the row first (unit-weight RMS norm).
template <bool W4A4>
__global__ void __launch_bounds__(kGThreads) k_prep_rows(const uint16_t* __restrict__ src, int K, int nrows,
                                                         float rms_eps, const unsigned int* __restrict__ amax_bits,
                                                         __half* __restrict__ dst, float* __restrict__ gout) {
    extern __shared__ __align__(16) uint16_t row[];  // [K] bf16
    __shared__ float red[kGThreads / 32];
    __shared__ unsigned int amax_s;
    const int r = blockIdx.x;
    if (r >= nrows) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint16_t* s = src + (size_t)r * K;
    for (int i = 8 * tid; i < K; i += 8 * kGThreads)
        *reinterpret_cast<uint4*>(row + i) = __ldcg(reinterpret_cast<const uint4*>(s + i));
    if (tid == 0) amax_s = 0u;
    __syncthreads();
    if (rms_eps > 0.0f) {
        // sum of squares: thread-ordered FMA chains, warp xor tree, warps in order
        float ss = 0.0f;
        for (int i = tid; i < K; i += kGThreads) {
            const float x = __uint_as_float(static_cast<uint32_t>(row[i]) << 16);
            ss = __fmaf_rn(x, x, ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kGThreads / 32; ++w) sum = __fadd_rn(sum, red[w]);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, static_cast<float>(K)), rms_eps)));
        __syncthreads();
        for (int i = tid; i < K; i += kGThreads) {
            const __nv_bfloat16 b =
                __float2bfloat16_rn(__fmul_rn(__uint_as_float(static_cast<uint32_t>(row[i]) << 16), inv));
            row[i] = *reinterpret_cast<const uint16_t*>(&b);
        }
        __syncthreads();
    }
    // the row factor: W4A4 the row global amax / 2688 (g quantises the row);
    // W4A16 the prescale 2^e of a row whose amax reaches 2^15 (g = 2^-e)
    float g = 0.0f, amax = 0.0f;
    if (amax_bits) {
        amax = __uint_as_float(__ldcg(amax_bits + r));
    } else {
        float mx = 0.0f;
        for (int i = tid; i < K; i += kGThreads)
            mx = fmaxf(mx, fabsf(__uint_as_float(static_cast<uint32_t>(row[i]) << 16)));
        mx = warp_max(mx);
        if (lane == 0) atomicMax(&amax_s, __float_as_uint(mx));
        __syncthreads();
        amax = __uint_as_float(amax_s);
    }
    g = W4A4 ? __fdiv_rn(amax, 2688.0f) : w4a16_row_inv_scale(amax);
    if (tid == 0 && gout) gout[r] = W4A4 ? g : w4a16_row_scale(amax);
    __half* d = dst + (size_t)r * K;
    for (int b = tid; b < (K >> 4); b += kGThreads) {
        const uint4 u0 = *reinterpret_cast<const uint4*>(row + 16 * b);
        const uint4 u1 = *reinterpret_cast<const uint4*>(row + 16 * b + 8);
        b_block_store<W4A4>(u0, u1, g, reinterpret_cast<uint4*>(d + 16 * b));
    }
}

// ---------------------------------------------------------------- grouped GEMM
enum GroupedKind { kGroupedUp = 0, kGroupedDown = 1 };

struct GroupedArgs {
    // routed weights [E][M][K] (NVFP4) and the shared expert's [MS][K]
    const uint8_t* codes;
    const uint8_t* scales;
    const float* global;
    const uint8_t* sh_codes;
    const uint8_t* sh_scales;
    const float* sh_global;
    int E, M, K;  // routed: M output rows, K reduction
    int MS, KS;   // shared expert: output rows, reduction
    int T, k;
    const int32_t* offsets;  // [E+1]
    const int32_t* tiles;    // [E+1]
    const int32_t* perm;     // [P] position -> pair (t * k + j)
    // B operands: routed rows (up: token rows xq [T][K] indexed by pair / k;
    // down: position rows aq [P][K]) and shared rows [T][K]
    const __half* b_routed;
    const float* g_routed;  // row globals of b_routed (W4A4)
    const __half* b_shared;
    const float* g_shared;
    // up outputs: bf16 rows [P][M] (position order) and [T][MS]; row amax
    uint16_t* act;
    uint16_t* act_sh;
    unsigned int* amax;     // [P]
    unsigned int* amax_sh;  // [T]
    // down outputs: FP32 rows [P][M] gate-weighted, [T][MS]
    float* ypart;
    float* ysh;
    const float* topk_w;  // [T][k]
};

// Stage of the grouped GEMM: one 128-k chunk of 64 weight rows (codes, then
// 8 scale bytes per row) and 64 B rows (f16, 128 halves each).
constexpr int kGCodeBytes = kGTile * 64;
constexpr int kGScaleBytes = kGTile * 8;
constexpr int kGBRowHalves = 128 + 8;  // padded row: fewer bank conflicts
constexpr int kGBBytes = kGTile * kGBRowHalves * 2;
constexpr int kGStageBytes = kGCodeBytes + kGScaleBytes + kGBBytes;
constexpr int kGStages = 5;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool W4A4, int KIND>
__global__ void __launch_bounds__(kGThreads) k_grouped(const GroupedArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int brow[kGTile];    // B row of each position of the tile (-1: none)
    __shared__ float bglob[kGTile];  // its row global (W4A4)
    __shared__ int posv[kGTile];     // output row (position or token) of each column
    __shared__ float gatev[kGTile];  // gate of each column (down, routed)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int rg = warp & 3, ch = warp >> 2;  // row group (16 rows), column half (32 positions)
    const int MT = a.M / kGTile, MTS = a.MS / kGTile;
    const int routed_items = __ldg(a.tiles + a.E) * MT;
    const int shared_items = ((a.T + kGTile - 1) / kGTile) * MTS;
    const int total = routed_items + shared_items;

    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        // ---- what this tile is
        // Items are m-major inside each group (an expert's tiles, then the
        // shared expert's): the n-tiles that share a weight tile run on
        // neighbouring CTAs at about the same time and meet it in L2.
        bool routed = item < routed_items;
        int e = 0, m0, pos0, npos;
        if (routed) {
            int lo = 0, hi = a.E;  // largest e with tiles[e] * MT <= item
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(a.tiles + mid) * MT <= item) lo = mid;
                else hi = mid;
            }
            e = lo;
            const int t0 = __ldg(a.tiles + e), nte = __ldg(a.tiles + e + 1) - t0;
            const int local = item - t0 * MT;
            m0 = (local / nte) * kGTile;
            pos0 = __ldg(a.offsets + e) + (local % nte) * kGTile;
            npos = min(kGTile, __ldg(a.offsets + e + 1) - pos0);
        } else {
            const int i = item - routed_items;
            const int nts = (a.T + kGTile - 1) / kGTile;
            m0 = (i / nts) * kGTile;
            pos0 = (i % nts) * kGTile;
            npos = min(kGTile, a.T - pos0);
        }
        __syncthreads();  // previous tile's users of brow / posv are done
        if (tid < kGTile) {
            int br = -1, pv = -1;
            float gl = 0.0f, gt = 1.0f;
            if (tid < npos) {
                const int pos = pos0 + tid;
                if (routed) {
                    const int pair = __ldg(a.perm + pos);
                    br = KIND == kGroupedUp ? pair / a.k : pos;
                    pv = pos;
                    if (KIND == kGroupedDown) gt = __ldg(a.topk_w + pair);
                } else {
                    br = pos;
                    pv = pos;
                }
                gl = __ldg((routed ? a.g_routed : a.g_shared) + br);  // W4A4 global, W4A16 prescale
            }
            brow[tid] = br;
            posv[tid] = pv;
            bglob[tid] = gl;
            gatev[tid] = gt;
        }
        __syncthreads();
        const int K = routed ? a.K : a.KS;
        const int nchunks = (K + 127) >> 7;
        const uint8_t* wc = routed ? a.codes + ((size_t)e * a.M + m0) * (K >> 1) : a.sh_codes + (size_t)m0 * (K >> 1);
        const uint8_t* ws = routed ? a.scales + ((size_t)e * a.M + m0) * (K >> 4) : a.sh_scales + (size_t)m0 * (K >> 4);
        const __half* bsrc = routed ? a.b_routed : a.b_shared;

        // ---- staging of chunk c into stage s
        auto stage = [&](int c, int s) {
            uint8_t* st = smem + (size_t)s * kGStageBytes;
            const int kb = 64 * c;                       // code byte offset of the chunk in a row
            const int kvalid = min(128, K - 128 * c);    // 128 or 64 valid k in this chunk
            // codes: 64 rows x 4 x 16 B
            for (int i = tid; i < kGTile * 4; i += kGThreads) {
                const int r = i >> 2, part = i & 3;
                const bool ok = 16 * part < kvalid / 2;
                cp_async16(st + r * 64 + 16 * part, wc + (size_t)r * (K >> 1) + kb + (ok ? 16 * part : 0), ok ? 16 : 0);
            }
            // scales: 64 rows x 2 x 4 B
            for (int i = tid; i < kGTile * 2; i += kGThreads) {
                const int r = i >> 1, part = i & 1;
                const bool ok = 4 * part < kvalid / 16;
                cp_async4(st + kGCodeBytes + r * 8 + 4 * part, ws + (size_t)r * (K >> 4) + 8 * c + (ok ? 4 * part : 0),
                          ok ? 4 : 0);
            }
            // B rows: 64 positions x 16 x 16 B
            __half* bs = reinterpret_cast<__half*>(st + kGCodeBytes + kGScaleBytes);
            for (int i = tid; i < kGTile * 16; i += kGThreads) {
                const int p = i >> 4, part = i & 15;
                const int br = brow[p];
                const bool ok = br >= 0 && 8 * part < kvalid;
                const __half* src = bsrc + (size_t)(br >= 0 ? br : 0) * K + 128 * c + (ok ? 8 * part : 0);
                cp_async16(bs + p * kGBRowHalves + 8 * part, src, ok ? 16 : 0);
            }
        };

        float acc[4][4];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[cb][v] = 0.0f;

        // ---- K loop, kGStages-deep cp.async pipeline
#pragma unroll
        for (int s = 0; s < kGStages - 1; ++s) {
            if (s < nchunks) stage(s, s);
            cp_async_commit();
        }
        for (int c = 0; c < nchunks; ++c) {
            if (c + kGStages - 1 < nchunks) stage(c + kGStages - 1, (c + kGStages - 1) % kGStages);
            cp_async_commit();
            cp_async_wait<kGStages - 1>();
            __syncthreads();
            const uint8_t* st = smem + (size_t)(c % kGStages) * kGStageBytes;
            const uint8_t* cr = st + (rg * 16) * 64;
            const uint8_t* sr = st + kGCodeBytes + (rg * 16) * 8;
            const __half* bs = reinterpret_cast<const __half*>(st + kGCodeBytes + kGScaleBytes);
            const uint4 wa = *reinterpret_cast<const uint4*>(cr + g * 64 + 16 * q);
            const uint4 wb = *reinterpret_cast<const uint4*>(cr + (g + 8) * 64 + 16 * q);
            const uint32_t sA = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sr + g * 8 + 2 * q));
            const uint32_t sB = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sr + (g + 8) * 8 + 2 * q));
            const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t fa[4], fb[4];
                e2m1x8_to_f16x8(wA[h], fa);
                e2m1x8_to_f16x8(wB[h], fb);
                const uint32_t scA = h < 2 ? bcast_lo(sA) : bcast_hi(sA);
                const uint32_t scB = h < 2 ? bcast_lo(sB) : bcast_hi(sB);
                const uint32_t a0 = hmul2(fa[0], scA), a1 = hmul2(fb[0], scB), a2 = hmul2(fa[1], scA),
                               a3 = hmul2(fb[1], scB);
                const uint32_t a4 = hmul2(fa[2], scA), a5 = hmul2(fb[2], scB), a6 = hmul2(fa[3], scA),
                               a7 = hmul2(fb[3], scB);
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    const int col = ch * 32 + cb * 8 + g;
                    const uint4 bv = *reinterpret_cast<const uint4*>(bs + col * kGBRowHalves + 32 * q + 8 * h);
                    mma_16816(acc[cb], a0, a1, a2, a3, bv.x, bv.y);
                    mma_16816(acc[cb], a4, a5, a6, a7, bv.z, bv.w);
                }
            }
            __syncthreads();  // stage c % kGStages may be refilled next
        }
        cp_async_wait<0>();

        // ---- epilogue
        const float gw = routed ? __ldg(a.global + e) : __ldg(a.sh_global);
        float m[4][2];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int col = ch * 32 + cb * 8 + 2 * q + (v & 1);
                const int row = m0 + rg * 16 + g + 8 * (v >> 1);
                if (v < 2) m[cb][v] = 0.0f;
                if (col >= npos) continue;
                const float gs = __fmul_rn(gw, bglob[col]);
                const float y = __fmul_rn(acc[cb][v], gs);
                const int pv = posv[col];
                if (KIND == kGroupedUp) {
                    const float rl = fmaxf(y, 0.0f);
                    const __nv_bfloat16 bv = __float2bfloat16_rn(__fmul_rn(rl, rl));
                    uint16_t* dst = routed ? a.act + (size_t)pv * a.M : a.act_sh + (size_t)pv * a.MS;
                    dst[row] = *reinterpret_cast<const uint16_t*>(&bv);
                    m[cb][v & 1] = fmaxf(m[cb][v & 1], __bfloat162float(bv));
                } else {
                    if (routed) a.ypart[(size_t)pv * a.M + row] = __fmul_rn(gatev[col], y);
                    else a.ysh[(size_t)pv * a.MS + row] = y;
                }
            }
        }
        if (KIND == kGroupedUp && W4A4) {
            // row amax of each column over this warp's 16 rows (lanes g)
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    float v = m[cb][p];
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    const int col = ch * 32 + cb * 8 + 2 * q + p;
                    if (g == 0 && col < npos)
                        atomicMax((routed ? a.amax : a.amax_sh) + posv[col], __float_as_uint(v));
                }
            }
        }
    }
}

// ---------------------------------------------------------------- combine
// out[t][i] = bf16(((ysh + y_{inv(t,0)}) + ...) + y_{inv(t,k-1)} + res), FP32.
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ ysh, const float* __restrict__ ypart,
                                                 const int32_t* __restrict__ inv, const uint16_t* __restrict__ res,
                                                 uint16_t* __restrict__ out, int T, int H, int k) {
    const int n4 = T * (H >> 2);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += gridDim.x * blockDim.x) {
        const int t = i / (H >> 2), c = 4 * (i % (H >> 2));
        float4 acc = __ldcg(reinterpret_cast<const float4*>(ysh + (size_t)t * H + c));
        for (int j = 0; j < k; ++j) {
            const int pos = __ldg(inv + t * k + j);
            const float4 y = __ldcg(reinterpret_cast<const float4*>(ypart + (size_t)pos * H + c));
            acc.x = __fadd_rn(acc.x, y.x);
            acc.y = __fadd_rn(acc.y, y.y);
            acc.z = __fadd_rn(acc.z, y.z);
            acc.w = __fadd_rn(acc.w, y.w);
        }
        if (res) {
            const uint2 rv = __ldcg(reinterpret_cast<const uint2*>(res + (size_t)t * H + c));
            acc.x = __fadd_rn(acc.x, __uint_as_float(rv.x << 16));
            acc.y = __fadd_rn(acc.y, __uint_as_float(rv.x & 0xFFFF0000u));
            acc.z = __fadd_rn(acc.z, __uint_as_float(rv.y << 16));
            acc.w = __fadd_rn(acc.w, __uint_as_float(rv.y & 0xFFFF0000u));
        }
        const __nv_bfloat16 o0 = __float2bfloat16_rn(acc.x), o1 = __float2bfloat16_rn(acc.y),
                            o2 = __float2bfloat16_rn(acc.z), o3 = __float2bfloat16_rn(acc.w);
        uint2 o;
        o.x = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&o0)) |
              (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&o1)) << 16);
        o.y = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&o2)) |
              (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&o3)) << 16);
        *reinterpret_cast<uint2*>(out + (size_t)t * H + c) = o;
    }
}

}  // namespace nvfp4moe
