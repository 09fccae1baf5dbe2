// common.cuh - device helpers shared by the kernels of libnvfp4moe.so:
// NVFP4 codecs (E2M1 values, E4M3 block scales), mbarrier + bulk-copy (TMA)
// staging with bounded waits, and the f16 tensor-core MMA used by the GEMVs.
//
// Everything here is sm_103a inline PTX or plain CUDA; no vendor library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4moe {

// Device error word (one per library instance): bounded waits that expire OR
// a bit in here and stop their kernel early. Read and cleared by
// nvfp4_last_device_error().
__device__ unsigned int g_dev_error;

enum : unsigned int {
    kErrWaitFull = 1u,   // a consumer waited too long for a staged tile
    kErrWaitEmpty = 2u,  // the producer waited too long for a free stage
    kErrWaitDrain = 4u,  // copies still in flight at exit did not land
    kErrBadInput = 8u,   // an expert index outside [0, E) or a broken plan
    kErrWaitPeer = 16u,  // a wait on another CTA's progress expired
};

// 1 s: device waits in this library normally take microseconds.
constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;

// Limit of the waits of one CTA on another's progress (the stack kernel's
// polls of tagged words), in ns: kWaitTimeoutNs unless changed with
// nvfp4_set_peer_wait_limit. Waits on this CTA's own staging copies keep the
// fixed 1 s, so that a CTA never leaves with copies still landing.
__device__ unsigned long long g_peer_wait_ns = kWaitTimeoutNs;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_dev_error(unsigned int bit) { atomicOr(&g_dev_error, bit); }

// Programmatic dependent launch: the next kernel in the stream may start as
// soon as every CTA of this one has called pdl_trigger(); pdl_wait() blocks
// until the previous kernel has completed and its writes are visible. Code
// before pdl_wait() may only touch arguments, read-only weights and shared
// memory. Both are no-ops when the launch carries no programmatic edge.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// try_wait with a suspend-time hint: a waiting thread sleeps until the phase
// completes (or the hint, in ns, runs out) instead of spinning, so waiting
// warps leave the issue slots to the warps that compute.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
}
// Non-blocking test of a phase: never suspends the thread.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until phase `parity` has completed by spinning on the non-blocking
// test (a thread suspended in try_wait resumes some hundreds of nanoseconds
// after the phase completes, which on a critical path costs more than the
// issue slots of the spin); false after 1 s.
__device__ __noinline__ bool mbar_wait_spin(uint64_t* b, uint32_t parity) {
    if (mbar_test_wait(b, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (int it = 1;; ++it) {
        if (mbar_test_wait(b, parity)) return true;
        if ((it & 255) == 0 && globaltimer() - t0 > kWaitTimeoutNs) return false;
    }
}

// Wait until phase `parity` of the barrier has completed; false after 1 s.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* b, uint32_t parity) {
    if (mbar_try_wait(b, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(b, parity)) return true;
        if (globaltimer() - t0 > kWaitTimeoutNs) return false;
    }
}

// Bulk (non-tensor) TMA copy global -> this CTA's shared memory; completion is
// signalled on `bar` as transaction bytes. dst, src 16-byte aligned; bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- codecs
// Four bytes of packed E2M1 pairs -> four f16x2 (byte b -> o[b]; in each byte
// the low nibble becomes the low half). Exact.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2. Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t out;
    uint16_t v = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(v));
    return out;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// {lo, lo} and {hi, hi} from an f16x2
__device__ __forceinline__ uint32_t bcast_lo(uint32_t x) { return __byte_perm(x, x, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t x) { return __byte_perm(x, x, 0x3232); }

// E4M3 byte -> float (exact). Scales are never negative or NaN here.
__device__ __forceinline__ float e4m3_to_float(uint32_t s) {
    const uint32_t e = (s >> 3) & 15u, m = s & 7u;
    return e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Non-negative float -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t float_to_e4m3_pos(float v) {
#if defined(NVFP4MOE_SOFT_CODECS)
    if (!(v < 448.0f)) return 0x7Eu;
    if (v < 0.015625f) return static_cast<uint32_t>(rintf(v * 512.0f));
    const int e = static_cast<int>((__float_as_uint(v) >> 23) & 0xFFu) - 127;  // [-6, 8]
    const float m = v * __uint_as_float(static_cast<uint32_t>(127 + 3 - e) << 23);  // [8, 16)
    const uint32_t q = static_cast<uint32_t>(rintf(m));
    return (static_cast<uint32_t>(e + 7) << 3) + (q - 8u);
#else
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
#endif
}

// Two floats -> one byte of E2M1 codes (x0 low nibble, x1 high nibble),
// round to nearest even, saturating at 6, sign kept also for a zero result.
__device__ __forceinline__ uint32_t float2_to_e2m1x2(float x0, float x1) {
    const uint32_t sgn = ((__float_as_uint(x0) >> 28) & 0x8u) | ((__float_as_uint(x1) >> 24) & 0x80u);
#if defined(NVFP4MOE_SOFT_CODECS)
    auto mag = [](float x) -> uint32_t {
        const float a = fabsf(x);
        return (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
               (a > 5.0f);
    };
    return (mag(x0) | (mag(x1) << 4)) | sgn;
#else
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "mov.b16 %0, {t, 0};\n\t}"
        : "=h"(r)
        : "f"(fabsf(x1)), "f"(fabsf(x0)));
    return (static_cast<uint32_t>(r) & 0xFFu) | sgn;
#endif
}

// Quantise one 16-element block with global g (NVFP4 rule of nvfp4moe.h):
//   s = E4M3((bamax / 6) / g); d = E4M3(s) * g; code_i = E2M1(x_i / d).
// Returns the 8 code bytes in (lo, hi) and the scale byte.
struct QBlock {
    uint32_t lo, hi, scale;
};
// x / d, IEEE round to nearest; a zero x is returned as it is (the quotient
// is that same signed zero), which keeps it off the division's slow path.
__device__ __forceinline__ float div_rn_or_zero(float x, float d) { return x == 0.0f ? x : __fdiv_rn(x, d); }

// x / d rounded to nearest even from y = RN(1/d), by Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y the correctly
// rounded reciprocal and q within one ulp of x / d, the residual x - q d is
// exact under a fused multiply-add and RN(q + (x - q d) y) is the correctly
// rounded quotient. The product estimate x y can be 1.5 ulp off, so one
// correction first makes it faithful, the second rounds it. Exact for finite x
// and 2^-100 <= d <= 2^100 whenever |x / d| >= 2^-3 (the residuals are then
// representable); a smaller quotient may be an ulp off, keeps its sign and
// stays below every E2M1 rounding boundary, the only use made of it here. A
// zero x is returned as it is (the sum of signed zeros in the corrections
// would turn -0 into +0).
__device__ __forceinline__ float div_by_recip(float x, float d, float y) {
    const float q0 = __fmul_rn(x, y);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, d, x), y, q0);
    const float q2 = __fmaf_rn(__fmaf_rn(-q1, d, x), y, q1);
    return x == 0.0f ? x : q2;
}

__device__ __forceinline__ QBlock quantize_block16(const float (&x)[16], float g) {
    float bamax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(x[i]));
    uint32_t s = 0;
    if (g > 0.0f && bamax > 0.0f) s = float_to_e4m3_pos(__fdiv_rn(__fdiv_rn(bamax, 6.0f), g));
    const float d = __fmul_rn(e4m3_to_float(s), g);
    QBlock q{0u, 0u, s};
    if (d >= 0x1p-100f && d <= 0x1p100f) {
        const float y = __frcp_rn(d);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = float2_to_e2m1x2(div_by_recip(x[2 * i], d, y), div_by_recip(x[2 * i + 1], d, y));
            if (i < 4) q.lo |= byte << (8 * i);
            else q.hi |= byte << (8 * (i - 4));
        }
    } else if (d != 0.0f) {  // extreme per-tensor globals: the plain division
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = float2_to_e2m1x2(div_rn_or_zero(x[2 * i], d), div_rn_or_zero(x[2 * i + 1], d));
            if (i < 4) q.lo |= byte << (8 * i);
            else q.hi |= byte << (8 * (i - 4));
        }
    }
    return q;
}

// Dequantised block values without the global (E2M1 * E4M3, exact in f16) as
// eight f16x2 in element order.
__device__ __forceinline__ void dequant_block16_f16(const QBlock& q, uint32_t (&o)[8]) {
    const uint32_t sv = e4m3x2_to_f16x2(q.scale);  // low half = scale
    const uint32_t s2 = bcast_lo(sv);
    uint32_t a[4], b[4];
    e2m1x8_to_f16x8(q.lo, a);
    e2m1x8_to_f16x8(q.hi, b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[i] = hmul2(a[i], s2);
        o[4 + i] = hmul2(b[i], s2);
    }
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// W4A16: a bf16 activation row (B operand) enters the f16 MMA as f16, whose
// largest finite value is 65504. A row whose amax reaches 2^15 is therefore
// scaled by 2^-e first, e = floor(log2 amax) - 14 (a power of two: exact down
// to f16's subnormal range), and every GEMV result of the row by 2^e, so that
// no element overflows; rows below 2^15 (every normalised row) keep e = 0 and
// convert unscaled. w4a16_row_scale returns 2^e, w4a16_row_inv_scale 2^-e
// (amax finite and >= 0).
__device__ __forceinline__ int w4a16_row_exp(float amax) {
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 14;
    return e > 0 ? e : 0;
}
__device__ __forceinline__ float w4a16_row_scale(float amax) {
    return __uint_as_float(static_cast<uint32_t>(127 + w4a16_row_exp(amax)) << 23);
}
__device__ __forceinline__ float w4a16_row_inv_scale(float amax) {
    return __uint_as_float(static_cast<uint32_t>(127 - w4a16_row_exp(amax)) << 23);
}

// Unit-weight RMS norm of one bf16 row by one warp (the per-block input norm
// of the pre-norm model the pages serve; its norms stay in bf16):
//   inv = 1 / sqrt(sum_i x_i^2 / K + eps),  y_i = bf16(x_i * inv).
// Lane l accumulates elements 8l + 256m .. 8l + 256m + 7 (m = 0, 1, ...) in
// order with fused multiply-adds, then an xor-shuffle tree (commutative at
// every level, so all lanes agree): the result does not depend on which
// kernel runs it. The row is read from global memory once, eight 16-byte
// loads per lane in flight, parked raw in dst (shared memory), and normalised
// there in place. K % 8 == 0; src (global) and dst (shared) 16-byte aligned.
__device__ __forceinline__ void warp_rmsnorm_row(const uint16_t* src, uint16_t* dst, int K, float eps) {
    const int lane = threadIdx.x & 31;
    float ss = 0.0f;
    for (int i0 = 8 * lane; i0 < K; i0 += 256 * 8) {
        uint4 v[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = i0 + 256 * m;
            v[m] = i < K ? __ldcg(reinterpret_cast<const uint4*>(src + i)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = i0 + 256 * m;
            if (i >= K) break;
            *reinterpret_cast<uint4*>(dst + i) = v[m];
            const uint32_t w[4] = {v[m].x, v[m].y, v[m].z, v[m].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xFFFF0000u);
                ss = __fmaf_rn(a, a, ss);
                ss = __fmaf_rn(b, b, ss);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), eps)));
    for (int i = 8 * lane; i < K; i += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(dst + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat16 lo = __float2bfloat16_rn(__fmul_rn(__uint_as_float(w[j] << 16), inv));
            const __nv_bfloat16 hi = __float2bfloat16_rn(__fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), inv));
            o[j] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&lo)) |
                   (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
        }
        *reinterpret_cast<uint4*>(dst + i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncwarp();
}

// Copy one bf16 row (global, written by an earlier kernel) into dst, one warp,
// eight 16-byte loads per lane in flight.
__device__ __forceinline__ void warp_copy_row(const uint16_t* src, uint16_t* dst, int K) {
    const int lane = threadIdx.x & 31;
    for (int i0 = 8 * lane; i0 < K; i0 += 256 * 8) {
        uint4 v[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = i0 + 256 * m;
            v[m] = i < K ? __ldcg(reinterpret_cast<const uint4*>(src + i)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = i0 + 256 * m;
            if (i < K) *reinterpret_cast<uint4*>(dst + i) = v[m];
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MMA
// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace nvfp4moe
