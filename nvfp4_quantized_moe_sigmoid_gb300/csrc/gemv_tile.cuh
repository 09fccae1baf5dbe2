// gemv_tile.cuh - the inner engine of every NVFP4 GEMV/skinny GEMM here:
// a 16-row x 8-column tile D = W_tile . B, where W_tile is 16 rows x K of an
// NVFP4 matrix staged in shared memory (canonical layout: codes [16][K/2],
// then scales [16][K/16]) and B holds up to 8 activation columns as f16 rows
// of length K. Two warps share a tile, each taking half of its 128-k chunks.
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

struct ChunkRegs {
    uint4 wa, wb;       // 16 code bytes of rows g and g + 8
    uint32_t sva, svb;  // two scale bytes of rows g and g + 8
};

__device__ __forceinline__ void chunk_load(ChunkRegs& r, const uint8_t* ca, const uint8_t* cb,
                                           const uint8_t* sa, const uint8_t* sb, int c, bool valid) {
    if (valid) {
        r.wa = *reinterpret_cast<const uint4*>(ca + 64 * c);
        r.wb = *reinterpret_cast<const uint4*>(cb + 64 * c);
        r.sva = *reinterpret_cast<const uint16_t*>(sa + 8 * c);
        r.svb = *reinterpret_cast<const uint16_t*>(sb + 8 * c);
    } else {
        r.wa = r.wb = make_uint4(0, 0, 0, 0);
        r.sva = r.svb = 0;
    }
}

// Four MMA accumulator sets (one per 32-k quarter of a chunk) keep four
// independent dependency chains in flight.
__device__ __forceinline__ void chunk_mma(const ChunkRegs& r, const __half* bp, int c, bool valid,
                                          float (&a4)[4][4]) {
    const uint32_t sA = e4m3x2_to_f16x2(r.sva), sB = e4m3x2_to_f16x2(r.svb);
    const uint32_t sA0 = bcast_lo(sA), sA1 = bcast_hi(sA);
    const uint32_t sB0 = bcast_lo(sB), sB1 = bcast_hi(sB);
    const uint32_t wA[4] = {r.wa.x, r.wa.y, r.wa.z, r.wa.w};
    const uint32_t wB[4] = {r.wb.x, r.wb.y, r.wb.z, r.wb.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        uint4 bv = make_uint4(0, 0, 0, 0);
        if (valid && bp) bv = *reinterpret_cast<const uint4*>(bp + 128 * c + 8 * h);
        uint32_t fa[4], fb[4];
        e2m1x8_to_f16x8(wA[h], fa);
        e2m1x8_to_f16x8(wB[h], fb);
        const uint32_t scA = h < 2 ? sA0 : sA1;
        const uint32_t scB = h < 2 ? sB0 : sB1;
        mma_16816(a4[h], hmul2(fa[0], scA), hmul2(fb[0], scB), hmul2(fa[1], scA), hmul2(fb[1], scB), bv.x,
                  bv.y);
        mma_16816(a4[h], hmul2(fa[2], scA), hmul2(fb[2], scB), hmul2(fa[3], scA), hmul2(fb[3], scB), bv.z,
                  bv.w);
    }
}

// Accumulates chunks [c0, c1) of the tile into acc: thread (g, q) holds
// acc[0..1] = rows g, cols 2q, 2q+1; acc[2..3] = rows g+8, cols 2q, 2q+1.
// `bcol` points to the f16 row of column g (K elements, 16-byte aligned) or
// is null for an all-zero column. K % 64 == 0. The next chunk's code and scale
// words are loaded while the current one is decoded (ping-pong registers).
__device__ __forceinline__ void tile_mma_16x8(const uint8_t* __restrict__ tcodes,
                                              const uint8_t* __restrict__ tscales, int K,
                                              const __half* __restrict__ bcol, int c0, int c1,
                                              float (&acc)[4]) {
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
    auto valid = [&](int c) { return !(half_tail && c == nchunks - 1 && q >= 2); };

    float a4[4][4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int v = 0; v < 4; ++v) a4[h][v] = 0.0f;

    ChunkRegs r0, r1;
    if (c0 < c1) chunk_load(r0, ca, cb, sa, sb, c0, valid(c0));
    int c = c0;
    for (; c + 1 < c1; c += 2) {
        chunk_load(r1, ca, cb, sa, sb, c + 1, valid(c + 1));
        chunk_mma(r0, bp, c, valid(c), a4);
        if (c + 2 < c1) chunk_load(r0, ca, cb, sa, sb, c + 2, valid(c + 2));
        chunk_mma(r1, bp, c + 1, valid(c + 1), a4);
    }
    if (c < c1) chunk_mma(r0, bp, c, valid(c), a4);
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[v] += (a4[0][v] + a4[1][v]) + (a4[2][v] + a4[3][v]);
}

// ------------------------------------------------------------------ staging
// A ring of `nstages` shared-memory stages, each holding one 16-row tile
// (codes then scales), filled by one producer thread with bulk TMA copies.
// The consumer warps are dealt into `groups` groups (warp w in group
// w % groups; nstages a multiple of groups): local item li goes to stage
// li % nstages and to group li % groups, whose warps each take a contiguous
// share of the tile's k-chunks and all release the stage. A group thus owns
// nstages / groups stages (one in every kernel here: with the warps of two
// CTAs per SM sharing the issue slots, more groups measured faster than
// deeper buffering per group).
// Every use of a stage is waited on, in order, by the same warps (an mbarrier
// parity wait names the current or the immediately preceding phase; a waiter
// for use u must not start while the barrier is still in phase u - 2, which
// fixed ownership guarantees).
constexpr int kConsumerWarps = 12;
constexpr int kMaxStages = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kConsumerThreads = kConsumerWarps * 32;

// Warps of group g when the consumer warps are dealt into `groups` groups (w % groups).
__device__ __forceinline__ int group_size(int g, int groups) { return (kConsumerWarps - g + groups - 1) / groups; }

struct Ring {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int uses[kMaxStages];  // producer-side count of fills per stage
    int abort;
    // partial tiles handed from the non-leading warps of a group to its
    // leader, double-buffered by the parity of the group's item count; warp
    // w >= groups uses slot w - groups
    float4 xred[kConsumerWarps - 1][2][32];
};

__device__ __forceinline__ void ring_init(Ring& r, int nstages, int groups) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], group_size(s % groups, groups));
            r.uses[s] = 0;
        }
        r.abort = 0;
        fence_mbar_init();
    }
}

// Producer side. The position of the next local item li is carried from one
// item to the next (stage li % nstages, phase (li / nstages) & 1), so that no
// item divides by the run-time stage count.
struct FillCursor {
    int li, s;
    uint32_t ph;
};

__device__ __forceinline__ FillCursor fill_cursor(int li, int nstages) {
    return FillCursor{li, li % nstages, static_cast<uint32_t>((li / nstages) & 1)};
}

// Fill the stage of item f.li with a 16-row tile and move f to the next item.
// Returns false (and flags the ring) if the stage never became free.
__device__ __forceinline__ bool ring_fill(Ring& r, uint8_t* ring_base, int stage_bytes, int nstages, FillCursor& f,
                                          const uint8_t* codes, const uint8_t* scales, int K) {
    const int s = f.s;
    if (f.li >= nstages && !mbar_wait_bounded(&r.empty[s], f.ph ^ 1u)) {
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
    ++f.li;
    if (++f.s == nstages) {
        f.s = 0;
        f.ph ^= 1u;
    }
    return true;
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

// All consumer warps (named barrier 1).
__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// All consumer warps; returns the OR of `pred` over them (the same value in
// every thread, so that all take the same branch).
__device__ __forceinline__ bool consumer_bar_or(bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(pred ? 1u : 0u), "n"(kConsumerThreads)
        : "memory");
    return out != 0;
}

// The warps of stage group s (named barrier 2 + s, 32 * gs threads); returns
// the AND of `pred` over them, so that all take the same decision.
__device__ __forceinline__ bool group_bar_and(int s, int gs, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(pred ? 1u : 0u), "r"(2 + s), "r"(32 * gs)
        : "memory");
    return out != 0;
}

// First local item index >= base that belongs to stage s.
__device__ __forceinline__ int first_item(int base, int s, int nstages) {
    return base + ((s - base % nstages) + nstages) % nstages;
}

// One staged tile, split between the warps of its group: rank p of gs
// computes k-chunks [nc p / gs, nc (p + 1) / gs); the other warps hand their
// partials to the leader (rank 0), which adds them in rank order. The leader
// gets lead = 1 and the finished tile in acc; ok = 0 for every warp of the
// group if any of them timed out waiting. Kept out of line: every kernel calls
// it from several loops, and one shared copy keeps the instruction footprint
// small.
//
// A consumer warp carries its group's place in the ring from one item to the
// next: the stage s = li % nstages of the group's current item li, its phase
// (li / nstages) & 1 and the group's item parity (li / groups) & 1, and its
// k-chunk share of the (at most two) tile widths the kernel uses, so that no
// tile divides by a run-time count.
struct GroupCursor {
    int li, s, grp, rank, gs, groups, nstages;
    uint32_t ph, u;
    int k0, c00, c10, k1, c01, c11;  // widths and this warp's chunk shares of them
};

__device__ __forceinline__ GroupCursor group_cursor(int nstages, int groups, int K0, int K1) {
    GroupCursor c;
    const int warp = threadIdx.x >> 5;
    c.grp = warp % groups;
    c.rank = warp / groups;
    c.gs = group_size(c.grp, groups);
    c.groups = groups;
    c.nstages = nstages;
    c.li = c.grp;
    c.s = c.grp;
    c.ph = 0;
    c.u = 0;
    const int n0 = (K0 + 127) >> 7, n1 = (K1 + 127) >> 7;
    c.k0 = K0;
    c.c00 = n0 * c.rank / c.gs;
    c.c10 = n0 * (c.rank + 1) / c.gs;
    c.k1 = K1;
    c.c01 = n1 * c.rank / c.gs;
    c.c11 = n1 * (c.rank + 1) / c.gs;
    return c;
}

__device__ __forceinline__ void cursor_next(GroupCursor& c) {
    c.li += c.groups;
    if ((c.s += c.groups) >= c.nstages) {
        c.s -= c.nstages;
        c.ph ^= 1u;
    }
    c.u ^= 1u;
}

struct TileOut {
    float4 acc;
    int lead, ok;
};

__device__ __noinline__ TileOut group_tile_at(Ring* r, int s, uint32_t ph, uint32_t u, int grp, int rank, int gs,
                                              int groups, const uint8_t* st, int K, const __half* bcol, int c0,
                                              int c1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool waited = mbar_wait_bounded(&r->full[s], ph);
    const bool got = __all_sync(0xffffffffu, waited);
    if (!got && lane == 0) set_dev_error(kErrWaitFull);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (got) tile_mma_16x8(st, st + 16 * (K >> 1), K, bcol, c0, c1, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&r->empty[s]);
    TileOut o;
    o.acc = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (gs == 1) {
        o.ok = got;
        o.lead = got;
        return o;
    }
    if (rank) r->xred[warp - groups][u][lane] = o.acc;
    o.ok = group_bar_and(grp, gs, got);
    o.lead = 0;
    if (rank || !o.ok) return o;
    for (int p = 1; p < gs; ++p) {
        const float4 x = r->xred[grp + p * groups - groups][u][lane];
        o.acc.x += x.x;
        o.acc.y += x.y;
        o.acc.z += x.z;
        o.acc.w += x.w;
    }
    o.lead = 1;
    return o;
}

// The group's current item (cursor c, tile width K: one of the two the cursor
// was made for) into acc; the caller then moves the cursor on.
__device__ __forceinline__ bool group_tile(Ring& r, const GroupCursor& c, uint8_t* ring_base, int stage_bytes, int K,
                                           const __half* bcol, float (&acc)[4], bool& ok) {
    const bool w0 = K == c.k0;
    const TileOut o = group_tile_at(&r, c.s, c.ph, c.u, c.grp, c.rank, c.gs, c.groups,
                                    ring_base + (size_t)c.s * stage_bytes, K, bcol, w0 ? c.c00 : c.c01,
                                    w0 ? c.c10 : c.c11);
    acc[0] = o.acc.x;
    acc[1] = o.acc.y;
    acc[2] = o.acc.z;
    acc[3] = o.acc.w;
    ok = o.ok != 0;
    return o.lead != 0;
}

// Quantise (W4A4) or convert (W4A16) nrows bf16 rows of length K into f16
// B-operand rows; W4A4 also writes each row's global to gout. Rows with
// src == null are zero-filled. Runs on the consumer threads. GSRC: the rows
// are global memory written by an earlier kernel (read through L2). Each
// thread loads all of its blocks (up to kBRegBlocks) before using any, and
// keeps them in registers between the row-amax and the quantisation passes.
template <bool GSRC>
__device__ __forceinline__ uint4 ld_row16(const uint16_t* p) {
    if (GSRC) return __ldcg(reinterpret_cast<const uint4*>(p));
    return *reinterpret_cast<const uint4*>(p);
}

constexpr int kBRegBlocks = 4;

// One 16-element block of a B row: W4A4 quantises it with the row global g
// (then stores its exact f16 dequantisation without g); W4A16 stores
// f16(x * g), g the row's power-of-two prescale 2^-e (w4a16_row_inv_scale).
template <bool W4A4>
__device__ __noinline__ void b_block_store(uint4 u0, uint4 u1, float g, uint4* d) {
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    uint32_t o[8];
    if (W4A4) {
        dequant_block16_f16(quantize_block16(v, g), o);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __half2 h2 = __floats2half2_rn(__fmul_rn(v[2 * j], g), __fmul_rn(v[2 * j + 1], g));
            o[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
    }
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// B rows for the GEMV engine: per row the amax (red[r], scratch), then the
// row factor gout[r] the epilogue multiplies in: W4A4 the row global
// amax / 2688, W4A16 the prescale 2^e (1 for rows below 2^15).
template <bool W4A4, bool GSRC>
__device__ __noinline__ void prepare_b_rows(const uint16_t* const* src, int nrows, int K,
                                               __half* dst, float* gout, unsigned int* red) {
    const int ctid = threadIdx.x;  // consumer thread index
    const int nb = K >> 4;
    const int total = nrows * nb;
    if (ctid < nrows) red[ctid] = 0u;
    consumer_bar();
    uint4 u[kBRegBlocks][2];
#pragma unroll
    for (int m = 0; m < kBRegBlocks; ++m) {
        const int i = ctid + m * kConsumerThreads;
        u[m][0] = u[m][1] = make_uint4(0, 0, 0, 0);
        if (i < total) {
            const int r = i / nb, b = i % nb;
            if (src[r]) {
                u[m][0] = ld_row16<GSRC>(src[r] + 16 * b);
                u[m][1] = ld_row16<GSRC>(src[r] + 16 * b + 8);
            }
        }
    }
    {
#pragma unroll
        for (int m = 0; m < kBRegBlocks; ++m) {
            const int i = ctid + m * kConsumerThreads;
            if (i >= total) break;
            const uint32_t w[8] = {u[m][0].x, u[m][0].y, u[m][0].z, u[m][0].w,
                                   u[m][1].x, u[m][1].y, u[m][1].z, u[m][1].w};
            float mx = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] << 16)));
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
            }
            atomicMax(&red[i / nb], __float_as_uint(mx));
        }
        // rows longer than the register window: amax over the rest, reloading
        for (int i = ctid + kBRegBlocks * kConsumerThreads; i < total; i += kConsumerThreads) {
            const int r = i / nb, b = i % nb;
            if (!src[r]) continue;
            const uint4 a0 = ld_row16<GSRC>(src[r] + 16 * b), a1 = ld_row16<GSRC>(src[r] + 16 * b + 8);
            const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float mx = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] << 16)));
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
            }
            atomicMax(&red[r], __float_as_uint(mx));
        }
        consumer_bar();
        if (gout && ctid < nrows)
            gout[ctid] = W4A4 ? __fdiv_rn(__uint_as_float(red[ctid]), 2688.0f)
                              : w4a16_row_scale(__uint_as_float(red[ctid]));
    }
#pragma unroll
    for (int m = 0; m < kBRegBlocks; ++m) {
        const int i = ctid + m * kConsumerThreads;
        if (i >= total) break;
        const int r = i / nb, b = i % nb;
        const float g = W4A4 ? __fdiv_rn(__uint_as_float(red[r]), 2688.0f)
                             : w4a16_row_inv_scale(__uint_as_float(red[r]));
        b_block_store<W4A4>(u[m][0], u[m][1], g, reinterpret_cast<uint4*>(dst + (size_t)r * K + 16 * b));
    }
    for (int i = ctid + kBRegBlocks * kConsumerThreads; i < total; i += kConsumerThreads) {
        const int r = i / nb, b = i % nb;
        uint4 a0 = make_uint4(0, 0, 0, 0), a1 = make_uint4(0, 0, 0, 0);
        if (src[r]) {
            a0 = ld_row16<GSRC>(src[r] + 16 * b);
            a1 = ld_row16<GSRC>(src[r] + 16 * b + 8);
        }
        const float g = W4A4 ? __fdiv_rn(__uint_as_float(red[r]), 2688.0f)
                             : w4a16_row_inv_scale(__uint_as_float(red[r]));
        b_block_store<W4A4>(a0, a1, g, reinterpret_cast<uint4*>(dst + (size_t)r * K + 16 * b));
    }
    consumer_bar();
}


}  // namespace nvfp4moe
