// gemv_tile.cuh - the inner engine of every NVFP4 GEMV/skinny GEMM here:
// one warp computes a 16-row x 8-column tile D = W_tile . B, where W_tile is
// 16 rows x K of an NVFP4 matrix staged in shared memory (canonical layout:
// codes [16][K/2], then scales [16][K/16]) and B holds up to 8 activation
// columns as f16 rows of length K.
//
// Arithmetic: each weight is decoded to f16 as E2M1 * E4M3 (cvt.rn.f16x2.e2m1x2
// and cvt.rn.f16x2.e4m3x2, then one f16 multiply). The product has at most six
// significant bits and lies in [2^-10, 2688], so the decode is exact; the
// per-tensor global is applied to the FP32 result by the caller. The tensor
// core (mma.sync m16n8k16, f16 in, FP32 accumulate) then forms exact products
// of the decoded weight and the activation and accumulates them in FP32.
//
// Reduction-index permutation: the MMA sums over its 16 k-slots, so any
// bijection between slots and physical k is valid as long as A and B use the
// same one. Thread (g = lane/4, q = lane%4) supplies slots {2q, 2q+1, 2q+8,
// 2q+9}; they are mapped to four consecutive physical k, so each thread reads
// 16 contiguous code bytes (32 k) per row per 128-k chunk and the matching 8
// contiguous f16 of B per MMA pair, with no shuffles.
#pragma once

#include "common.cuh"

namespace nvfp4moe {

// Accumulates into acc: thread (g, q) holds acc[0..1] = rows g, cols 2q, 2q+1;
// acc[2..3] = rows g+8, cols 2q, 2q+1. `bcol` points to the f16 row of column
// g (K elements, 16-byte aligned) or is null for an all-zero column.
// K % 64 == 0.
//
// Latency: the next chunk's code, scale and B words are loaded while the
// current chunk is decoded, and the MMAs of a chunk go to four independent
// accumulator sets (summed at the end), so one warp keeps several MMAs and
// shared-memory loads in flight instead of one dependent chain.
struct TileChunk {
    uint4 wa, wb, b0, b1, b2, b3;
    uint32_t sva, svb;
};

__device__ __forceinline__ void tile_load_chunk(TileChunk& t, const uint8_t* ca, const uint8_t* cb,
                                                const uint8_t* sa, const uint8_t* sb, const __half* bp,
                                                int c, bool valid) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    t.wa = t.wb = t.b0 = t.b1 = t.b2 = t.b3 = z;
    t.sva = t.svb = 0;
    if (valid) {
        t.wa = *reinterpret_cast<const uint4*>(ca + 64 * c);
        t.wb = *reinterpret_cast<const uint4*>(cb + 64 * c);
        t.sva = *reinterpret_cast<const uint16_t*>(sa + 8 * c);
        t.svb = *reinterpret_cast<const uint16_t*>(sb + 8 * c);
        if (bp) {
            const uint4* b = reinterpret_cast<const uint4*>(bp + 128 * c);
            t.b0 = b[0];
            t.b1 = b[1];
            t.b2 = b[2];
            t.b3 = b[3];
        }
    }
}

__device__ __forceinline__ void tile_mma_16x8(const uint8_t* __restrict__ tcodes,
                                              const uint8_t* __restrict__ tscales, int K,
                                              const __half* __restrict__ bcol, float (&acc)[4]) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int KB = K >> 1, KS = K >> 4;
    const uint8_t* ca = tcodes + g * KB + 16 * q;
    const uint8_t* cb = tcodes + (g + 8) * KB + 16 * q;
    const uint8_t* sa = tscales + g * KS + 2 * q;
    const uint8_t* sb = tscales + (g + 8) * KS + 2 * q;
    const __half* bp = bcol ? bcol + 32 * q : nullptr;
    const int nchunks = (K + 127) >> 7;
    const bool half_tail = (K & 127) != 0;

    float a4[4][4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int v = 0; v < 4; ++v) a4[h][v] = 0.0f;

    TileChunk cur, nxt;
    tile_load_chunk(cur, ca, cb, sa, sb, bp, 0, !(half_tail && nchunks == 1 && q >= 2));
    for (int c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks)
            tile_load_chunk(nxt, ca, cb, sa, sb, bp, c + 1, !(half_tail && c + 2 == nchunks && q >= 2));
        const uint32_t sA = e4m3x2_to_f16x2(cur.sva), sB = e4m3x2_to_f16x2(cur.svb);
        const uint32_t sA0 = bcast_lo(sA), sA1 = bcast_hi(sA);
        const uint32_t sB0 = bcast_lo(sB), sB1 = bcast_hi(sB);
        const uint32_t wA[4] = {cur.wa.x, cur.wa.y, cur.wa.z, cur.wa.w};
        const uint32_t wB[4] = {cur.wb.x, cur.wb.y, cur.wb.z, cur.wb.w};
        const uint4 bq[4] = {cur.b0, cur.b1, cur.b2, cur.b3};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            uint32_t fa[4], fb[4];
            e2m1x8_to_f16x8(wA[h], fa);
            e2m1x8_to_f16x8(wB[h], fb);
            const uint32_t scA = h < 2 ? sA0 : sA1;
            const uint32_t scB = h < 2 ? sB0 : sB1;
            mma_16816(a4[h], hmul2(fa[0], scA), hmul2(fb[0], scB), hmul2(fa[1], scA), hmul2(fb[1], scB),
                      bq[h].x, bq[h].y);
            mma_16816(a4[h], hmul2(fa[2], scA), hmul2(fb[2], scB), hmul2(fa[3], scA), hmul2(fb[3], scB),
                      bq[h].z, bq[h].w);
        }
        cur = nxt;
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[v] += (a4[0][v] + a4[1][v]) + (a4[2][v] + a4[3][v]);
}

// ------------------------------------------------------------------ staging
// A ring of `nstages` shared-memory stages, each holding one 16-row tile
// (codes then scales), filled by one producer thread with bulk TMA copies.
// Stage s is owned by consumer warp s: local item li goes to stage and warp
// li % nstages, so every stage's uses are waited on, in order, by one warp.
// (An mbarrier parity wait names the current or the immediately preceding
// phase; a waiter for use u must not start while the barrier is still in
// phase u - 2, which single ownership guarantees.) full[s] completes when the
// tile has landed, empty[s] when its warp has finished reading it.
constexpr int kConsumerWarps = 8;
constexpr int kMaxStages = kConsumerWarps;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp

struct Ring {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int uses[kMaxStages];  // producer-side count of fills per stage
    int abort;
};

__device__ __forceinline__ void ring_init(Ring& r, int nstages) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], 1);
            r.uses[s] = 0;
        }
        r.abort = 0;
        fence_mbar_init();
    }
}

// Producer side: fill stage for local item li with a tile of 16 rows.
// Returns false (and flags the ring) if the stage never became free.
__device__ __forceinline__ bool ring_fill(Ring& r, uint8_t* ring_base, int stage_bytes, int nstages,
                                          int li, const uint8_t* codes, const uint8_t* scales, int K) {
    const int s = li % nstages;
    if (li >= nstages && !mbar_wait_bounded(&r.empty[s], ((li / nstages) - 1) & 1)) {
        set_dev_error(kErrWaitEmpty);
        r.abort = 1;
        return false;
    }
    const uint32_t cbytes = 16u * (uint32_t)(K >> 1), sbytes = 16u * (uint32_t)(K >> 4);
    uint8_t* dst = ring_base + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&r.full[s], cbytes + sbytes);
    bulk_g2s(dst, codes, cbytes, &r.full[s]);
    bulk_g2s(dst + cbytes, scales, sbytes, &r.full[s]);
    r.uses[s] += 1;
    return true;
}

// Consumer side (whole warp): wait for local item li. False on timeout.
__device__ __forceinline__ bool ring_acquire(Ring& r, int nstages, int li) {
    const int s = li % nstages;
    const bool ok = mbar_wait_bounded(&r.full[s], (li / nstages) & 1);
    const bool all_ok = __all_sync(0xffffffffu, ok);
    if (!all_ok && (threadIdx.x & 31) == 0) set_dev_error(kErrWaitFull);
    return all_ok;
}

__device__ __forceinline__ void ring_release(Ring& r, int nstages, int li) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[li % nstages]);
}

// After every warp is done (call after __syncthreads): make sure no bulk copy
// is still landing in shared memory before the CTA exits.
__device__ __forceinline__ void ring_drain(Ring& r, int nstages) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            if (r.uses[s] > 0 && !mbar_wait_bounded(&r.full[s], (r.uses[s] - 1) & 1))
                set_dev_error(kErrWaitDrain);
        }
    }
}

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Quantise (W4A4) or convert (W4A16) nrows bf16 rows of length K into f16
// B-operand rows; W4A4 also writes each row's global to gout. Rows with
// src == null are zero-filled. Runs on the 256 consumer threads.
template <bool W4A4>
__device__ __forceinline__ void prepare_b_rows(const uint16_t* const* src, int nrows, int K,
                                               __half* dst, float* gout, unsigned int* red) {
    const int ctid = threadIdx.x;  // 0..255
    const int nb = K >> 4;
    if (W4A4) {
        if (ctid < nrows) red[ctid] = 0u;
        consumer_bar();
        for (int i = ctid; i < nrows * nb; i += kConsumerWarps * 32) {
            const int r = i / nb, b = i % nb;
            if (!src[r]) continue;
            const uint4* p = reinterpret_cast<const uint4*>(src[r] + 16 * b);
            const uint4 u0 = p[0], u1 = p[1];
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
                m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
            }
            atomicMax(&red[r], __float_as_uint(m));
        }
        consumer_bar();
        if (ctid < nrows) gout[ctid] = __fdiv_rn(__uint_as_float(red[ctid]), 2688.0f);
    }
    for (int i = ctid; i < nrows * nb; i += kConsumerWarps * 32) {
        const int r = i / nb, b = i % nb;
        uint4* d = reinterpret_cast<uint4*>(dst + (size_t)r * K + 16 * b);
        if (!src[r]) {
            d[0] = make_uint4(0, 0, 0, 0);
            d[1] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const uint4* p = reinterpret_cast<const uint4*>(src[r] + 16 * b);
        const uint4 u0 = p[0], u1 = p[1];
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float v[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
        uint32_t o[8];
        if (W4A4) {
            const float g = __fdiv_rn(__uint_as_float(red[r]), 2688.0f);
            dequant_block16_f16(quantize_block16(v, g), o);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __half2 h2 = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
                o[j] = *reinterpret_cast<const uint32_t*>(&h2);
            }
        }
        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    consumer_bar();
}

}  // namespace nvfp4moe
