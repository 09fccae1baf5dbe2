// moe_grouped_tc.cuh - the grouped expert GEMMs of moe_expert_forward in W4A4
// for more than 4 tokens (prefill and high-concurrency decode: "Let's
// optimize Nemotron 3.5 Lightning - a worklog", Step 3) on the 5th-generation
// tensor cores: tcgen05.mma kind::mxf4nvf4 multiplies the NVFP4 weights by the
// NVFP4-quantised activations directly (E2M1 x E2M1 products, one E4M3 scale
// per 16 elements on each side, FP32 accumulation in tensor memory), so no
// operand is ever decoded on the CUDA cores.
//
//   D[m][n] = sum_k W[m][k] X[n][k]   (m: 128 weight rows of one expert,
//                                      n: up to 128 positions of that expert)
//   up:   act[n][m] = bf16(relu(D gw gx[n])^2), row amax of act[n] (atomic)
//   down: y[n][m]   = gate[n] (D gw gx[n])
//
// Operand layout in shared memory: K-major with the 128-byte swizzle. Each
// row holds 256 k (128 bytes), rows in 1024-byte atoms of 8, and 16-byte chunk
// c of row r stored at chunk c ^ (r % 8); descriptor: stride between 8-row
// groups 1024 bytes, and the 64-k step s starts 32 s bytes into the row. A 2-D
// TMA box {128 bytes, rows} of the row-major [rows][K/2] code matrix with the
// 128-byte swizzle lands exactly in that layout (whole 128-byte rows per
// request; a 16-byte-wide box of the unswizzled layout limits the copy engine
// to 16-byte requests).
//
// Scale factors live in tensor memory. For M = 128 the MMA reads the scales of
// row m from TMEM lane m, column sfa + m / 32 (byte b = 16-element block b of
// the 64-k step), and those of output column n from lane 32 q + n % 32 of each
// lane quarter q, column sfb + n / 32. Both are written with tcgen05.st by four
// warps, one per lane quarter, from row-major scale bytes in shared memory
// (the weights' per item, the activations' per stage).
//
// Warp roles (one CTA per SM, persistent over the work items):
//   warp 0      producer: TMA for the codes, a bulk copy per item for the
//               weight scales, cp.async for the activation scales
//   warp 1      tensor memory allocation; lane 0 issues the MMAs
//   warps 2-5   scale warps (lane quarter = warp % 4)
//   warps 6-9   epilogue warps (lane quarter = warp % 4), accumulator in TMEM
//               double-buffered so that an item's epilogue overlaps the next
//               item's MMAs
// Every wait is bounded (1 s); a role that gives up flags the error word and
// the CTA abort flag, and the others stop at their next wait.
#pragma once

#include <cuda.h>

#include "moe_decode.cuh"
#include "moe_grouped.cuh"

namespace nvfp4moe {

constexpr int kTcThreads = 320;
constexpr int kTcSlots = 8;  // pipeline stages in flight (mbarrier slots)
constexpr int kTcRows = 128;                     // weight rows per item (MMA M)
constexpr int kTcPos = 128;                      // positions per item (MMA N <= 128)
constexpr int kTcKStage = 256;                   // k per pipeline stage (4 MMAs of 64)
constexpr int kTcCodeA = kTcRows * kTcKStage / 2;  // 16 KB
constexpr int kTcCodeB = kTcPos * kTcKStage / 2;   // 16 KB (32 positions per 4 KB)
// A pipeline stage: [A codes 16 KB][B codes ng x 4 KB][B scales ng x 512 B]
// for an item with ng groups of 32 positions, rounded up to the 1024-byte
// swizzle atom; stages of any size are packed in issue order into a byte ring
// over the rest of shared memory (one that would cross the end starts again
// at its beginning), so that items with few positions keep more stages in
// flight.
constexpr int kTcOffB = kTcCodeA;
__host__ __device__ constexpr int tc_stage_bytes(int ng) { return (kTcCodeA + ng * (4096 + 512) + 1023) & ~1023; }
// The weight scales of an item (128 rows x K/16 bytes, contiguous in the
// caller's matrix) arrive in one bulk copy into one of two per-item blocks:
// the rows are only 4-byte aligned, so a per-stage copy would take 512
// separate 4-byte requests. 16 bytes of slack after the block (the last row's
// final step may read past it; those words are never used).
constexpr int kTcScBlk = 30720;
constexpr int kTcOffScBlk = 0;
constexpr int kTcOffRing = 2 * kTcScBlk;  // a multiple of 1024
constexpr int kTcSmemSlack = 1024;        // the kernel aligns its dynamic shared memory to 1024 bytes
// tensor memory columns: two 128-column accumulators, then per slot 16
// columns of A scales (4 steps x 4 lane quarters) and 16 of B scales
// (4 steps x 4 column groups of 32)
constexpr uint32_t kTcCols = 512;
constexpr uint32_t kTcColSFA = 256;
constexpr uint32_t kTcColSFB = kTcColSFA + 16 * kTcSlots;
static_assert(kTcColSFB + 16 * kTcSlots <= kTcCols, "tensor memory columns");

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
// the mbarrier counts one arrival when every earlier cp.async of this thread has landed
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_alloc(uint32_t* dst, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate ? 1u : 0u)
        : "memory");
}
// arrives once on the mbarrier when every earlier MMA of this thread is complete
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_st_x1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tc_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
                 "r"(v2), "r"(v3)
                 : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
        "[%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 consecutive columns of a lane quarter in one load (one wait)
__device__ __forceinline__ void tc_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of tcgen05.mma for the K-major 128-byte
// swizzled layout: start address (16-byte units), leading byte offset 16
// (unused by this layout), stride byte offset 1024 (8-row groups),
// descriptor version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1), both
// K-major, E4M3 scales, M = 128, N = n.
__device__ __forceinline__ uint32_t umma_idesc_mxf4(int n) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
}

// Bounded mbarrier wait that also gives up when the CTA abort flag is raised.
// It spins on the non-blocking test: each pipeline hand-off here is on the
// critical path, and a suspended waiter resumes only some hundreds of
// nanoseconds after the phase completes; the few waiting warps cost no issue
// slots the tensor cores need.
__device__ __noinline__ bool tc_wait(uint64_t* b, uint32_t parity, volatile int* abort_s) {
    if (mbar_test_wait(b, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (int it = 1;; ++it) {
        if (mbar_test_wait(b, parity)) return true;
        if ((it & 255) == 0) {
            if (*abort_s) return false;
            if (globaltimer() - t0 > kWaitTimeoutNs) {
                set_dev_error(kErrWaitFull);
                *abort_s = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- stage trace
// Built with -DNVFP4MOE_TRACE, CTAs 0 .. kTcTrCtas - 1 of the tensor-core
// kernels record the SM clock (clock64) at the hand-offs of each pipeline stage and
// work item into g_tc_trace[kernel][CTA][event][index] (kernel 0: grouped up,
// 1: grouped down, 2: lm_head GEMM), read back by nvfp4moe_tc_trace_read.
// Without the flag the trace points compile to nothing.
enum TcTraceEvent : int {
    kTcTrProdWait = 0,  // producer: before waiting for the stage's space (index: stage)
    kTcTrProdIssued,    // producer: stage copies issued
    kTcTrFullSeen,      // scale / decoder warp 2: the stage's bytes landed
    kTcTrPrepDone,      // scale / decoder warp 2: the stage's operands ready for the MMA
    kTcTrMmaIssue,      // MMA thread: the stage's waits passed, MMAs issued
    kTcTrItemStart,     // MMA thread: accumulator free, item begins (index: item)
    kTcTrEpiStart,      // epilogue warp (quarter 0): the item's accumulator complete
    kTcTrEpiEnd,        // epilogue warp (quarter 0): the item's outputs written
    kTcTrProdSpace,     // producer: the stage's space is free
    kTcTrProdTma,       // producer: the stage's tensor copies issued
    kTcTrProdCpa,       // producer: the stage's scale copies issued
    kTcTrEvents
};
constexpr int kTcTrCtas = 4, kTcTrIdx = 1024;
#if defined(NVFP4MOE_TRACE)
__device__ unsigned long long g_tc_trace[3][kTcTrCtas][kTcTrEvents][kTcTrIdx];
#define TC_TRACE(cond, kern, ev, idx)                                                               \
    do {                                                                                           \
        if ((cond) && blockIdx.x < kTcTrCtas && (idx) < kTcTrIdx)                                   \
            g_tc_trace[kern][blockIdx.x][ev][idx] = clock64();                                      \
    } while (0)
#else
#define TC_TRACE(cond, kern, ev, idx) \
    do {                              \
    } while (0)
#endif

// ---------------------------------------------------------------- arguments
// A segment is one weight tensor over its positions: the routed experts
// (positions grouped by expert) or the shared expert (all tokens in order).
struct TcSeg {
    int nexp, M, K;          // experts, weight rows per expert, reduction length (K % 64 == 0)
    const int32_t* offsets;  // [nexp + 1] position range of each expert; null: one range [0, npos)
    const int32_t* chunks;   // [nexp + 1] prefix sums of ceil(n_e / 128) (with offsets)
    int npos;
    const uint8_t* a_scales;  // [nexp * M][K / 16] E4M3
    const float* a_global;    // [nexp]
    const uint8_t* b_scales;  // [b_rows][b_spitch] E4M3 (b_spitch % 16 == 0)
    int b_spitch, b_rows;
    const float* b_global;  // [b_rows] row globals of the quantised B rows
    uint16_t* act;          // up: [positions][M] bf16
    unsigned int* amax;     // up: [positions] row amax bits
    float* y;               // down: [positions][M] FP32
    const float* gate;      // down: topk_w of each pair (null: 1)
    const int32_t* perm;    // position -> pair
};

struct TcArgs {
    CUtensorMap a_map[2];     // weight codes: 2-D {K / 2, nexp * M}, box {128, 128}, 128-byte swizzle
    CUtensorMap b_map[2][4];  // B codes: 2-D {K / 2, b_rows}, box {128, 32 (g + 1)}, 128-byte swizzle
    TcSeg seg[2];
    int nseg;
    int ring_cap;  // bytes of the stage ring (a multiple of 1024, >= 2 stages of 4 groups)
};

struct TcItem {
    int seg, e, row0, n, mt;
};

// Independent accumulators of an item: its 64-k steps go round-robin to nc
// accumulators of 32 ng columns in the item's 128 (steps that accumulate
// into one accumulator form a dependent chain, and at small N each MMA is
// short enough for that chain's latency to set the pace); the epilogue adds
// them in order.
__device__ __forceinline__ int tc_chains(int ng, int nks) { return min(min(4 / ng, 4), nks); }

// The position ranges and chunk prefixes of both segments, copied to shared
// memory at the start: every role looks an item up at every item start (a
// binary search of dependent reads), which from global memory would stall
// each role for several round trips per item.
constexpr int kTcMaxExperts = 256;
struct TcTab {
    int off[2][kTcMaxExperts + 1];
    int chk[2][kTcMaxExperts + 1];
};

__device__ __forceinline__ int tc_seg_items(const TcSeg& s, const int* chk) {
    const int MT = (s.M + kTcRows - 1) / kTcRows;
    const int nch = s.offsets ? chk[s.nexp] : (s.npos + kTcPos - 1) / kTcPos;
    return nch * MT;
}

// Item i: m-major inside a chunk of positions, so that consecutive items (on
// neighbouring CTAs at about the same time) share their B rows in L2.
// Work item i of the launch goes to CTA i % G. The second segment's items
// (the shared expert: all tokens, so the widest, up to 128 positions) take
// the slots [r0, r0 + n1) of the order, r0 = total % G, so that they land on
// CTAs that get one item fewer than the others; the first segment's items
// fill the rest in their order. (When they do not fit there, the segments
// stay in order.)
struct TcOrder {
    int items0, n1, r0;
};
__device__ __forceinline__ TcOrder tc_order(int items0, int total, int G) {
    TcOrder o;
    o.items0 = items0;
    o.n1 = total - items0;
    o.r0 = total % G;
    if (o.n1 > G - o.r0 || o.r0 + o.n1 > total) o.r0 = items0;  // the segments in order
    return o;
}
__device__ __forceinline__ TcItem tc_item(const TcSeg* segs, const TcTab& tab, int i, const TcOrder& ord) {
    TcItem it;
    if (i >= ord.r0 && i < ord.r0 + ord.n1) {
        it.seg = 1;
        i -= ord.r0;
    } else {
        it.seg = 0;
        if (i >= ord.r0 + ord.n1) i -= ord.n1;
    }
    const TcSeg& s = segs[it.seg];
    const int MT = (s.M + kTcRows - 1) / kTcRows;
    const int ch = i / MT;
    it.mt = i - ch * MT;
    if (s.offsets) {
        const int* chunks = tab.chk[it.seg];
        const int* offsets = tab.off[it.seg];
        int lo = 0, hi = s.nexp;  // chunks[lo] <= ch < chunks[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (chunks[mid] <= ch) lo = mid;
            else hi = mid;
        }
        it.e = lo;
        it.row0 = offsets[lo] + (ch - chunks[lo]) * kTcPos;
        it.n = min(kTcPos, offsets[lo + 1] - it.row0);
    } else {
        it.e = 0;
        it.row0 = ch * kTcPos;
        it.n = min(kTcPos, s.npos - it.row0);
    }
    return it;
}

// ---------------------------------------------------------------- the GEMM
template <int KIND>
__global__ void __launch_bounds__(kTcThreads, 1) k_grouped_tc(const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    // the swizzled stages need 1024-byte aligned addresses
    uint8_t* const smem = tc_smem + ((1024u - (smem_u32(tc_smem) & 1023u)) & 1023u);
    __shared__ __align__(8) uint64_t full[kTcSlots], empty[kTcSlots], sfready[kTcSlots];
    __shared__ uint32_t stage_off[kTcSlots];  // shared-memory offset of the slot's current stage
    // producer bookkeeping (in shared memory: a run-time indexed local array
    // lives in local memory, whose lines the streaming traffic evicts from L1)
    __shared__ int p_uses[kTcSlots], p_vs[kTcSlots], p_scuses[2];
    // the segment descriptors, read in every step of every role: from shared
    // memory (a run-time indexed kernel parameter is a slow generic load)
    __shared__ TcSeg segs[2];
    // per epilogue warp: the item's column factors gw gx[p] and gates
    __shared__ float ep_scale[4][kTcPos], ep_gate[4][kTcPos];
    static_assert(sizeof(TcSeg) % 8 == 0, "TcSeg copy");
    for (int i = threadIdx.x; i < (int)(2 * sizeof(TcSeg) / 8); i += blockDim.x)
        reinterpret_cast<uint64_t*>(segs)[i] = reinterpret_cast<const uint64_t*>(a.seg)[i];
    __shared__ TcTab tab;
    for (int sg = 0; sg < a.nseg; ++sg) {
        const TcSeg& s = a.seg[sg];
        if (!s.offsets) continue;
        for (int i = threadIdx.x; i <= s.nexp; i += blockDim.x) {
            tab.off[sg][i] = __ldg(s.offsets + i);
            tab.chk[sg][i] = __ldg(s.chunks + i);
        }
    }
    __shared__ __align__(8) uint64_t dfull[2], dempty[2], drain;
    __shared__ __align__(8) uint64_t scfull[2], scempty[2];  // per-item weight scale blocks
    __shared__ uint32_t tmem_s;
    __shared__ int abort_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcSlots; ++s) {
            mbar_init(&full[s], 33);  // the producer's expect_tx + one cp.async arrival per lane
            mbar_init(&empty[s], 1);
            mbar_init(&sfready[s], 4);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(&dfull[d], 1);
            mbar_init(&dempty[d], 4);
            mbar_init(&scfull[d], 1);
            mbar_init(&scempty[d], 4);
        }
        mbar_init(&drain, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc_alloc(&tmem_s, kTcCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;
    volatile int* ab = &abort_s;
    const int items0 = tc_seg_items(segs[0], tab.chk[0]);
    const int total = items0 + (a.nseg > 1 ? tc_seg_items(segs[1], tab.chk[1]) : 0);
    const TcOrder ord = tc_order(items0, total, gridDim.x);

    if (warp == 0) {
        // ---- producer
        // tensor maps into the copy engine's descriptor cache up front
        if (lane < 5 * a.nseg) {
            const CUtensorMap* tm = lane % 5 == 0 ? &a.a_map[lane / 5] : &a.b_map[lane / 5][lane % 5 - 1];
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
        }
        int g = 0, n_it = 0, tail = 0, vhead = 0;
        const int cap = a.ring_cap;
        int* const uses = p_uses;
        int* const vs = p_vs;
        int* const scuses = p_scuses;
        if (lane < kTcSlots) uses[lane] = vs[lane] = 0;
        if (lane < 2) scuses[lane] = 0;
        __syncwarp();
        bool ok = true;
        for (int i = blockIdx.x; i < total && ok; i += gridDim.x, ++n_it) {
            const TcItem it = tc_item(segs, tab, i, ord);
            const TcSeg& s = segs[it.seg];
            const int nstage = ((s.K >> 6) + 3) >> 2, ng = (it.n + 31) >> 5;
            const int arow0 = it.e * s.M + it.mt * kTcRows;
            const int arows = s.nexp * s.M, sp = s.K >> 4;
            const uint8_t* const b_scales = s.b_scales;
            const int b_rows = s.b_rows, b_spitch = s.b_spitch;
            const CUtensorMap* const amap = &a.a_map[it.seg];
            const CUtensorMap* const bmap = &a.b_map[it.seg][ng - 1];
            // the item's weight scales: min(128, rows left) x K/16 bytes
            {
                const int b = n_it & 1;
                bool w = true;
                if (lane == 0 && n_it >= 2) w = tc_wait(&scempty[b], ((n_it >> 1) - 1) & 1, ab);
                if (!__shfl_sync(0xffffffffu, w, 0)) break;
                if (lane == 0) {
                    const uint32_t bytes = (uint32_t)(min(kTcRows, arows - arow0) * sp);
                    mbar_arrive_expect_tx(&scfull[b], bytes);
                    bulk_g2s(smem + kTcOffScBlk + b * kTcScBlk, s.a_scales + (size_t)arow0 * sp, bytes, &scfull[b]);
                }
                if (lane == 0) scuses[b] += 1;
            }
            for (int ks = 0; ks < nstage; ++ks, ++g) {
                const int st = g % kTcSlots;
                const int size = tc_stage_bytes(ng);
                int v = vhead;
                if (v % cap + size > cap) v += cap - v % cap;
                // release in issue order: the slot's previous stage and every
                // older stage whose bytes this one overwrites
                const int lim = v + size - cap;
                bool w = true;
                TC_TRACE(lane == 0, KIND, kTcTrProdWait, g);
                if (lane == 0) {
                    while (tail < g && (tail <= g - kTcSlots || vs[tail % kTcSlots] < lim)) {
                        w = tc_wait(&empty[tail % kTcSlots], (tail / kTcSlots) & 1, ab);
                        if (!w) break;
                        ++tail;
                    }
                }
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    ok = false;
                    break;
                }
                tail = __shfl_sync(0xffffffffu, tail, 0);
                TC_TRACE(lane == 0, KIND, kTcTrProdSpace, g);
                if (lane == 0) vs[st] = v;  // read by lane 0 only
                vhead = v + size;
                const uint32_t off = (uint32_t)(kTcOffRing + v % cap);
                uint8_t* base = smem + off;
                if (lane == 0) {
                    stage_off[st] = off;
                    mbar_arrive_expect_tx(&full[st], (uint32_t)(kTcCodeA + ng * 4096));
                    tma_load_2d(base, amap, ks * 128, arow0, &full[st]);
                    tma_load_2d(base + kTcOffB, bmap, ks * 128, it.row0, &full[st]);
                }
                TC_TRACE(lane == 0, KIND, kTcTrProdTma, g);
                // B scales: 32 ng rows x 16 bytes
                for (int r = lane; r < 32 * ng; r += 32) {
                    const int row = it.row0 + r;
                    const bool in = row < b_rows;
                    cp_async16(base + kTcOffB + 4096 * ng + 16 * r,
                               in ? b_scales + (size_t)row * b_spitch + ks * 16 : b_scales, in ? 16 : 0);
                }
                TC_TRACE(lane == 0, KIND, kTcTrProdCpa, g);
                cp_async_mbar_arrive(&full[st]);
                TC_TRACE(lane == 0, KIND, kTcTrProdIssued, g);
                if (lane == 0) uses[st] += 1;
            }
        }
        // nothing may still be landing in shared memory when the CTA exits
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < kTcSlots; ++s)
                if (uses[s] > 0 && !mbar_wait_bounded(&full[s], (uses[s] - 1) & 1)) set_dev_error(kErrWaitDrain);
            for (int b = 0; b < 2; ++b)  // the last scale block issued into each buffer
                if (scuses[b] > 0 && !mbar_wait_bounded(&scfull[b], (scuses[b] - 1) & 1)) set_dev_error(kErrWaitDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue
        if (lane == 0) {
            int g = 0, n_it = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < total && ok; i += gridDim.x, ++n_it) {
                const TcItem it = tc_item(segs, tab, i, ord);
                const TcSeg& s = segs[it.seg];
                const int nks = s.K >> 6, nstage = (nks + 3) >> 2, ng = (it.n + 31) >> 5;
                const int db = n_it & 1;
                if (n_it >= 2 && !tc_wait(&dempty[db], ((n_it >> 1) - 1) & 1, ab)) break;
                tc_fence_after();
                TC_TRACE(true, KIND, kTcTrItemStart, n_it);
                const uint32_t idesc = umma_idesc_mxf4(32 * ng);
                const uint32_t dcol = tmem + 128u * db;
                const int nc = tc_chains(ng, nks);
                for (int ks = 0; ks < nstage; ++ks, ++g) {
                    const int st = g % kTcSlots;
                    const uint32_t par = (g / kTcSlots) & 1;
                    if (!tc_wait(&full[st], par, ab) || !tc_wait(&sfready[st], par, ab)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    TC_TRACE(true, KIND, kTcTrMmaIssue, g);
                    const uint32_t sbase = smem_u32(smem + stage_off[st]);
                    const int nk = min(4, nks - 4 * ks);
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint64_t ad = umma_desc_sw128(sbase + 32u * kk);
                        const uint64_t bd = umma_desc_sw128(sbase + kTcOffB + 32u * kk);
                        const int q = 4 * ks + kk;  // 64-k step of the item
                        tc_mma_mxf4(dcol + 32u * ng * (q % nc), ad, bd, idesc, tmem + kTcColSFA + 16u * st + 4u * kk,
                                    tmem + kTcColSFB + 16u * st + 4u * kk, q >= nc);
                    }
                    tc_commit(&empty[st]);  // stage (and its scale columns) free once these MMAs are done
                }
                if (!ok) break;
                tc_commit(&dfull[db]);
            }
            // every MMA of this CTA is complete before the tensor memory is released
            tc_commit(&drain);
            if (!mbar_wait_bounded(&drain, 0)) set_dev_error(kErrWaitDrain);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---- scale factors -> tensor memory (lane quarter q)
        const int q = warp & 3;
        const uint32_t lb = (uint32_t)(32 * q) << 16;
        int g = 0, n_it = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < total && ok; i += gridDim.x, ++n_it) {
            const TcItem it = tc_item(segs, tab, i, ord);
            const TcSeg& s = segs[it.seg];
            const int nstage = ((s.K >> 6) + 3) >> 2, ng = (it.n + 31) >> 5;
            const int sp = s.K >> 4;
            const int b = n_it & 1;
            {
                bool w = true;
                if (lane == 0) w = tc_wait(&scfull[b], (n_it >> 1) & 1, ab);
                if (!__shfl_sync(0xffffffffu, w, 0)) break;
            }
            const uint8_t* scrow = smem + kTcOffScBlk + b * kTcScBlk + (size_t)(32 * q + lane) * sp;
            for (int ks = 0; ks < nstage; ++ks, ++g) {
                const int st = g % kTcSlots;
                bool w = true;
                if (lane == 0) w = tc_wait(&full[st], (g / kTcSlots) & 1, ab);
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    ok = false;
                    break;
                }
                TC_TRACE(warp == 2 && lane == 0, KIND, kTcTrFullSeen, g);
                const uint8_t* base = smem + stage_off[st];
                // A: row 32 q + lane, step kk -> column sfa(kk) + q
                const uint32_t* sw = reinterpret_cast<const uint32_t*>(scrow + 16 * ks);
                const uint32_t ca = tmem + lb + kTcColSFA + 16u * st + q;
                tc_st_x1(ca, sw[0]);
                tc_st_x1(ca + 4, sw[1]);
                tc_st_x1(ca + 8, sw[2]);
                tc_st_x1(ca + 12, sw[3]);
                // B: position 32 j + lane, step kk -> column sfb(kk) + j (every quarter)
                uint4 sb[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    sb[j] = j < ng ? *reinterpret_cast<const uint4*>(base + kTcOffB + 4096 * ng + 16 * (32 * j + lane))
                                   : make_uint4(0, 0, 0, 0);
                const uint32_t cb = tmem + lb + kTcColSFB + 16u * st;
                tc_st_x4(cb, sb[0].x, sb[1].x, sb[2].x, sb[3].x);
                tc_st_x4(cb + 4, sb[0].y, sb[1].y, sb[2].y, sb[3].y);
                tc_st_x4(cb + 8, sb[0].z, sb[1].z, sb[2].z, sb[3].z);
                tc_st_x4(cb + 12, sb[0].w, sb[1].w, sb[2].w, sb[3].w);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfready[st]);
                TC_TRACE(warp == 2 && lane == 0, KIND, kTcTrPrepDone, g);
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&scempty[b]);  // done with this item's scale block
        }
    } else {
        // ---- epilogue (lane quarter q: weight rows 32 q .. 32 q + 31 of the item)
        const int q = warp & 3;
        const uint32_t lb = (uint32_t)(32 * q) << 16;
        int n_it = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x, ++n_it) {
            const TcItem it = tc_item(segs, tab, i, ord);
            const TcSeg& s = segs[it.seg];
            const int db = n_it & 1;
            bool w = true;
            if (lane == 0) w = tc_wait(&dfull[db], (n_it >> 1) & 1, ab);
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            tc_fence_after();
            TC_TRACE(q == 0 && lane == 0, KIND, kTcTrEpiStart, n_it);
            const float gw = __ldg(s.a_global + it.e);
            const int m = it.mt * kTcRows + 32 * q + lane;
            // the item's column factors, every load in flight at once (one
            // round trip per item instead of dependent loads per column)
            {
                float f[kTcPos / 32], gt[kTcPos / 32];
#pragma unroll
                for (int u = 0; u < kTcPos / 32; ++u) {
                    const int c = lane + 32 * u;
                    f[u] = c < it.n ? __ldg(s.b_global + it.row0 + c) : 0.0f;
                    gt[u] = 1.0f;
                    if (KIND == kGroupedDown && s.gate && c < it.n) gt[u] = __ldg(s.gate + __ldg(s.perm + it.row0 + c));
                }
#pragma unroll
                for (int u = 0; u < kTcPos / 32; ++u) {
                    ep_scale[q][lane + 32 * u] = __fmul_rn(gw, f[u]);
                    ep_gate[q][lane + 32 * u] = gt[u];
                }
                __syncwarp();
            }
            const bool mv = m < s.M;
            const int ng = (it.n + 31) >> 5, nc = tc_chains(ng, s.K >> 6);
            // this item's output pointers in registers (stores would otherwise
            // make every read of the shared descriptor a reload)
            const int M = s.M;
            uint16_t* const act = s.act;
            unsigned int* const amax = s.amax;
            float* const yout = s.y;
            const bool gated = s.gate != nullptr;
            // wide items (more than 64 positions): 32 columns per TMEM load (one
            // wait), and the warp's maximum of column c0 + j kept in lane j,
            // which posts it (one atomic per lane per 32 columns); narrow
            // items: 16 columns per load, lane 0 posting each column's maximum
            if (it.n > 64) {
                for (int c0 = 0; c0 < it.n; c0 += 32) {
                    uint32_t r[32];
                    tc_ld_x32(tmem + lb + 128u * db + c0, r);
                    for (int c = 1; c < nc; ++c) {  // the other accumulators, added in order
                        uint32_t r2[32];
                        tc_ld_x32(tmem + lb + 128u * db + 32u * ng * c + c0, r2);
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), __uint_as_float(r2[j])));
                    }
                    unsigned int mine = 0u;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int p = it.row0 + c0 + j;
                        if (c0 + j >= it.n) break;
                        const float v = __fmul_rn(__uint_as_float(r[j]), ep_scale[q][c0 + j]);
                        if (KIND == kGroupedUp) {
                            const float rl = fmaxf(v, 0.0f);
                            const __nv_bfloat16 bv = __float2bfloat16_rn(__fmul_rn(rl, rl));
                            if (mv) act[(size_t)p * M + m] = *reinterpret_cast<const uint16_t*>(&bv);
                            const unsigned int mx =
                                __reduce_max_sync(0xffffffffu, mv ? __float_as_uint(__bfloat162float(bv)) : 0u);
                            if (lane == j) mine = mx;
                        } else {
                            if (mv) yout[(size_t)p * M + m] = gated ? __fmul_rn(ep_gate[q][c0 + j], v) : v;
                        }
                    }
                    if (KIND == kGroupedUp && mine != 0u) atomicMax(amax + it.row0 + c0 + lane, mine);
                }
            } else {
                for (int c0 = 0; c0 < it.n; c0 += 16) {
                    uint32_t r[16];
                    tc_ld_x16(tmem + lb + 128u * db + c0, r);
                    for (int c = 1; c < nc; ++c) {  // the other accumulators, added in order
                        uint32_t r2[16];
                        tc_ld_x16(tmem + lb + 128u * db + 32u * ng * c + c0, r2);
#pragma unroll
                        for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), __uint_as_float(r2[j])));
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int p = it.row0 + c0 + j;
                        if (c0 + j >= it.n) break;
                        const float v = __fmul_rn(__uint_as_float(r[j]), ep_scale[q][c0 + j]);
                        if (KIND == kGroupedUp) {
                            const float rl = fmaxf(v, 0.0f);
                            const __nv_bfloat16 bv = __float2bfloat16_rn(__fmul_rn(rl, rl));
                            if (mv) act[(size_t)p * M + m] = *reinterpret_cast<const uint16_t*>(&bv);
                            const unsigned int mx =
                                __reduce_max_sync(0xffffffffu, mv ? __float_as_uint(__bfloat162float(bv)) : 0u);
                            if (lane == 0 && mx != 0u) atomicMax(amax + p, mx);
                        } else {
                            if (mv) yout[(size_t)p * M + m] = gated ? __fmul_rn(ep_gate[q][c0 + j], v) : v;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();  // also: this warp's column factors may be rewritten
            if (lane == 0) mbar_arrive(&dempty[db]);
            TC_TRACE(q == 0 && lane == 0, KIND, kTcTrEpiEnd, n_it);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTcCols);
    }
}

// ---------------------------------------------------------------- B operand rows
// Row r of src (bf16 [K]) -> NVFP4 codes [K/2] (low nibble = even element) and
// E4M3 scales [spitch] with the row's global g = amax / 2688 (amax given in
// amax_bits[r], else of the row); rms_eps > 0 normalises the row first (the
// same unit-weight RMS norm as the other paths). The row goes to row r of
// codes / scales / gout and, when inv is given, also to rows inv[r k + j]
// (j < k) of the position-order copy pcodes / pscales / pgout.
__global__ void __launch_bounds__(kGThreads) k_quant_rows_tc(const uint16_t* __restrict__ src, int K, int nrows,
                                                             float rms_eps, const unsigned int* __restrict__ amax_bits,
                                                             uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                             int spitch, float* __restrict__ gout,
                                                             const int32_t* __restrict__ inv, int k,
                                                             uint8_t* __restrict__ pcodes,
                                                             uint8_t* __restrict__ pscales, float* __restrict__ pgout) {
    extern __shared__ __align__(16) uint16_t row[];  // [K] bf16
    __shared__ float red[kGThreads / 32];
    __shared__ unsigned int amax_s;
    __shared__ int dst_rows[kDecodeMaxK + 1];
    const int r = blockIdx.x;
    if (r >= nrows) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint16_t* s = src + (size_t)r * K;
    for (int i = 8 * tid; i < K; i += 8 * kGThreads)
        *reinterpret_cast<uint4*>(row + i) = __ldcg(reinterpret_cast<const uint4*>(s + i));
    if (tid == 0) amax_s = 0u;
    const int ncopy = inv ? k : 0;
    if (tid <= ncopy) dst_rows[tid] = tid == 0 ? r : __ldg(inv + (size_t)r * k + tid - 1);
    __syncthreads();
    if (rms_eps > 0.0f) {
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
        const float inv_rms = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, static_cast<float>(K)), rms_eps)));
        __syncthreads();
        for (int i = tid; i < K; i += kGThreads) {
            const __nv_bfloat16 b =
                __float2bfloat16_rn(__fmul_rn(__uint_as_float(static_cast<uint32_t>(row[i]) << 16), inv_rms));
            row[i] = *reinterpret_cast<const uint16_t*>(&b);
        }
        __syncthreads();
    }
    float g;
    if (amax_bits) {
        g = __fdiv_rn(__uint_as_float(__ldcg(amax_bits + r)), 2688.0f);
    } else {
        float mx = 0.0f;
        for (int i = tid; i < K; i += kGThreads)
            mx = fmaxf(mx, fabsf(__uint_as_float(static_cast<uint32_t>(row[i]) << 16)));
        mx = warp_max(mx);
        if (lane == 0) atomicMax(&amax_s, __float_as_uint(mx));
        __syncthreads();
        g = __fdiv_rn(__uint_as_float(amax_s), 2688.0f);
    }
    if (tid <= ncopy) (tid == 0 ? gout : pgout)[dst_rows[tid]] = g;
    for (int b = tid; b < (K >> 4); b += kGThreads) {
        const uint4 u0 = *reinterpret_cast<const uint4*>(row + 16 * b);
        const uint4 u1 = *reinterpret_cast<const uint4*>(row + 16 * b + 8);
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float v[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
        const QBlock qb = quantize_block16(v, g);
        for (int c = 0; c <= ncopy; ++c) {
            const size_t dr = static_cast<size_t>(dst_rows[c]);
            uint8_t* cd = (c == 0 ? codes : pcodes) + dr * (K >> 1) + 8 * b;
            *reinterpret_cast<uint2*>(cd) = make_uint2(qb.lo, qb.hi);
            (c == 0 ? scales : pscales)[dr * spitch + b] = static_cast<uint8_t>(qb.scale);
        }
    }
}

}  // namespace nvfp4moe
