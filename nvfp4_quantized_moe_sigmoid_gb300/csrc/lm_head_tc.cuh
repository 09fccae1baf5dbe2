// lm_head_tc.cuh - lm_head_forward for 9..256 tokens per launch on the
// 5th-generation tensor cores ("Let's optimize Nemotron 3.5 Lightning - a
// worklog", Step 4: the 131072 x 2688 NVFP4 weight-only lm_head; at many
// concurrent tokens it is a dense GEMM bound by the 16-bit tensor pipe).
//
//   logits[t][v] = gw gx[t] sum_k W[v][k] x[t][k]
//
// W is NVFP4 (weight-only): every 128-row x 64-k tile of it is decoded once
// to f16 (E2M1 x E4M3 is exact in f16) into shared memory, then multiplied by
// all N tokens at once with tcgen05.mma kind::f16 (M = 128, N <= 256, K = 16
// per instruction, FP32 accumulation in tensor memory). x is the tokens' f16
// rows prepared by k_prep_rows (RMS-normalised and scaled by the row
// prescale 2^-e, gx[t] = 2^e).
//
// Operands in shared memory are K-major with the 128-byte swizzle (rows of
// 64 f16, 8-row atoms of 1024 bytes, 16-byte chunk c of row r at c ^ (r % 8)):
// the activations arrive in that layout by a 2-D TMA box {128 bytes, N rows}
// with the 128-byte swizzle; the decoded weights are written into it by the
// decode warps. The raw codes of a stage arrive by a TMA box {32 bytes, 128
// rows}, its block scales by 4-byte cp.async per row.
//
// Warp roles (one CTA per SM, persistent over the 128-row tiles):
//   warp 0      producer (TMA, cp.async of the scales)
//   warp 1      tensor memory allocation; lane 0 issues the MMAs
//   warps 2-9   decoders: threads 2r and 2r + 1 decode the two 32-k halves
//               of row r of each stage's tile (two warps per scheduler, so
//               that one warp's conversion latency hides behind the other's)
//   warps 10-13 epilogue (lane quarter = warp % 4), accumulator double-
//               buffered in tensor memory so that a tile's epilogue overlaps
//               the next tile's MMAs
// Every wait is bounded (1 s); a role that gives up flags the error word and
// the CTA abort flag, and the others stop at their next wait.
#pragma once

#include "moe_grouped_tc.cuh"

namespace nvfp4moe {

constexpr int kLmTcThreads = 448;
constexpr int kLmTcDecWarps = 8;
constexpr int kLmTcRows = 128;  // weight rows per tile (MMA M)
constexpr int kLmTcK = 64;      // k per stage: one 128-byte row of f16
constexpr int kLmTcStages = 4;
constexpr int kLmTcMaxN = 256;
constexpr int kLmTcA = kLmTcRows * 128;   // decoded weights of a stage: 16 KB
constexpr int kLmTcRaw = kLmTcRows * 32;  // their codes: 4 KB
constexpr int kLmTcScl = kLmTcRows * 4;   // their scales: 512 B
// stage: [A f16][B f16, N rows x 128 B][raw codes][raw scales], 1024-aligned
__host__ __device__ constexpr int lm_tc_stage_bytes(int n) {
    return (kLmTcA + n * 128 + kLmTcRaw + kLmTcScl + 1023) & ~1023;
}

struct LmTcArgs {
    CUtensorMap a_map;      // raw codes [V][H/2] bytes, box {32, 128}, no swizzle
    CUtensorMap b_map;      // f16 rows [T][2 H] bytes, box {128, N}, 128-byte swizzle
    const uint8_t* scales;  // [V][H/16]
    const float* global;    // [1]
    const float* gx;        // [T] row factors of this launch's tokens
    float* logits;          // this launch's first token row, [T][ld]
    int64_t ld;
    int V, H, T, N;         // N: the MMA N, T rounded up to 16
};

// Instruction descriptor of kind::f16: FP32 accumulator, A and B f16 and
// K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t umma_idesc_f16(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kLmTcRows >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_f16(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kLmTcThreads, 1) k_lm_head_tc(const __grid_constant__ LmTcArgs a) {
    extern __shared__ __align__(1024) uint8_t lt_smem[];
    uint8_t* const smem = lt_smem + ((1024u - (smem_u32(lt_smem) & 1023u)) & 1023u);
    __shared__ __align__(8) uint64_t full[kLmTcStages], decoded[kLmTcStages], empty[kLmTcStages];
    __shared__ __align__(8) uint64_t dfull[2], dempty[2], drain;
    __shared__ uint32_t tmem_s;
    __shared__ int abort_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = a.N, H = a.H, nks = H / kLmTcK;
    const int stage = lm_tc_stage_bytes(N);
    const int tiles = a.V / kLmTcRows;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kLmTcStages; ++s) {
            mbar_init(&full[s], 33);  // the producer's expect_tx + one cp.async arrival per lane
            mbar_init(&decoded[s], kLmTcDecWarps);
            mbar_init(&empty[s], 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(&dfull[d], 1);
            mbar_init(&dempty[d], 4);
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

    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.a_map)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.b_map)) : "memory");
        }
        int g = 0;
        bool ok = true;
        const int sp = H >> 4;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            const int row0 = tile * kLmTcRows;
            for (int ks = 0; ks < nks; ++ks, ++g) {
                const int s = g % kLmTcStages;
                bool w = true;
                TC_TRACE(lane == 0, 2, kTcTrProdWait, g);
                if (lane == 0 && g >= kLmTcStages) w = tc_wait(&empty[s], ((g / kLmTcStages) - 1) & 1, ab);
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    ok = false;
                    break;
                }
                uint8_t* const base = smem + (size_t)s * stage;
                TC_TRACE(lane == 0, 2, kTcTrProdSpace, g);
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(kLmTcRaw + N * 128));
                    tma_load_2d(base + kLmTcA + N * 128, &a.a_map, ks * 32, row0, &full[s]);
                    tma_load_2d(base + kLmTcA, &a.b_map, ks * 128, 0, &full[s]);
                }
                TC_TRACE(lane == 0, 2, kTcTrProdTma, g);
                // the stage's block scales: row r's four bytes (k / 16 = 4 ks .. 4 ks + 3)
                uint8_t* const sc = base + kLmTcA + N * 128 + kLmTcRaw;
                for (int r = lane; r < kLmTcRows; r += 32)
                    cp_async4(sc + 4 * r, a.scales + (size_t)(row0 + r) * sp + 4 * ks);
                TC_TRACE(lane == 0, 2, kTcTrProdCpa, g);
                cp_async_mbar_arrive(&full[s]);
                TC_TRACE(lane == 0, 2, kTcTrProdIssued, g);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0) {  // nothing may still be landing when the CTA exits
            const int last = g - 1;
            for (int q = 0; q < kLmTcStages && last - q >= 0; ++q) {
                const int gg = last - q;
                if (!mbar_wait_bounded(&full[gg % kLmTcStages], (gg / kLmTcStages) & 1)) set_dev_error(kErrWaitDrain);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue
        if (lane == 0) {
            int g = 0, n_it = 0;
            bool ok = true;
            const uint32_t idesc = umma_idesc_f16(N);
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++n_it) {
                const int db = n_it & 1;
                if (n_it >= 2 && !tc_wait(&dempty[db], ((n_it >> 1) - 1) & 1, ab)) break;
                tc_fence_after();
                TC_TRACE(true, 2, kTcTrItemStart, n_it);
                const uint32_t dcol = tmem + 256u * db;
                for (int ks = 0; ks < nks; ++ks, ++g) {
                    const int s = g % kLmTcStages;
                    const uint32_t par = (g / kLmTcStages) & 1;
                    if (!tc_wait(&full[s], par, ab) || !tc_wait(&decoded[s], par, ab)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    TC_TRACE(true, 2, kTcTrMmaIssue, g);
                    const uint32_t sbase = smem_u32(smem + (size_t)s * stage);
#pragma unroll
                    for (int kk = 0; kk < kLmTcK / 16; ++kk) {
                        const uint64_t ad = umma_desc_sw128(sbase + 32u * kk);
                        const uint64_t bd = umma_desc_sw128(sbase + kLmTcA + 32u * kk);
                        tc_mma_f16(dcol, ad, bd, idesc, ks > 0 || kk > 0);
                    }
                    tc_commit(&empty[s]);
                }
                if (!ok) break;
                tc_commit(&dfull[db]);
            }
            // every MMA of this CTA is complete before the tensor memory is released
            tc_commit(&drain);
            if (!mbar_wait_bounded(&drain, 0)) set_dev_error(kErrWaitDrain);
        }
        __syncwarp();
    } else if (warp < 2 + kLmTcDecWarps) {
        // ---- decoders: thread d = half d % 2 of row d / 2 of every stage's tile
        const int d = threadIdx.x - 64, r = d >> 1, hf = d & 1;
        int g = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            for (int ks = 0; ks < nks; ++ks, ++g) {
                const int s = g % kLmTcStages;
                bool w = true;
                if (lane == 0) w = tc_wait(&full[s], (g / kLmTcStages) & 1, ab);
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    ok = false;
                    break;
                }
                TC_TRACE(warp == 2 && lane == 0, 2, kTcTrFullSeen, g);
                uint8_t* const base = smem + (size_t)s * stage;
                const uint4 c0 = *reinterpret_cast<const uint4*>(base + kLmTcA + N * 128 + 16 * d);
                const uint32_t sw = *reinterpret_cast<const uint16_t*>(base + kLmTcA + N * 128 + kLmTcRaw + 4 * r + 2 * hf);
                const uint32_t cw[4] = {c0.x, c0.y, c0.z, c0.w};
                uint8_t* const arow = base + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {  // chunk c = 4 hf + i: k = 8c .. 8c + 7, scale block c / 2
                    const int c = 4 * hf + i;
                    const uint32_t s2 = e4m3x2_to_f16x2((sw >> (8 * (i >> 1))) & 0xFFu);
                    const uint32_t sv = bcast_lo(s2);
                    uint32_t f[4];
                    e2m1x8_to_f16x8(cw[i], f);
                    *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) =
                        make_uint4(hmul2(f[0], sv), hmul2(f[1], sv), hmul2(f[2], sv), hmul2(f[3], sv));
                }
                // the tensor core reads these bytes through the async proxy
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&decoded[s]);
                TC_TRACE(warp == 2 && lane == 0, 2, kTcTrPrepDone, g);
            }
        }
    } else {
        // ---- epilogue (lane quarter q: rows 32 q .. 32 q + 31 of the tile)
        const int q = warp & 3;
        const uint32_t lb = (uint32_t)(32 * q) << 16;
        const float gw = __ldg(a.global);
        int n_it = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++n_it) {
            const int db = n_it & 1;
            bool w = true;
            if (lane == 0) w = tc_wait(&dfull[db], (n_it >> 1) & 1, ab);
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            tc_fence_after();
            TC_TRACE(q == 0 && lane == 0, 2, kTcTrEpiStart, n_it);
            const int64_t row = (int64_t)tile * kLmTcRows + 32 * q + lane;
            for (int c0 = 0; c0 < N; c0 += 16) {
                uint32_t v[16];
                tc_ld_x16(tmem + lb + 256u * db + c0, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = c0 + j;
                    if (t < a.T)
                        a.logits[(int64_t)t * a.ld + row] =
                            __fmul_rn(__uint_as_float(v[j]), __fmul_rn(gw, __ldg(a.gx + t)));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[db]);
            TC_TRACE(q == 0 && lane == 0, 2, kTcTrEpiEnd, n_it);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTcCols);
    }
}

}  // namespace nvfp4moe
