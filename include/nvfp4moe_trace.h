/*
 * nvfp4moe_trace.h - diagnostics of libnvfp4moe_trace.so, the build of the
 * library with -DNVFP4MOE_TRACE (no operation of the pages). The default
 * libnvfp4moe.so does not export this call.
 *
 * In the trace build, every CTA of moe_stack_forward records the global timer
 * (ns) at the phase boundaries of every layer: consumer thread 0 at the layer
 * start, the layer input read, the router logits posted, the top-k and plan,
 * the up tiles, the down operands, the down units, all partials posted and
 * its rows of the layer output written; the producer at the first and last
 * staging copy of the layer (StackTraceEvent in moe_stack.cuh).
 */
#ifndef NVFP4MOE_TRACE_H
#define NVFP4MOE_TRACE_H

#include "nvfp4moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Copies the trace of the last moe_stack_forward call to host memory `dst`:
 * unsigned 64-bit global-timer readings [256 CTAs][32 layers][16 events];
 * entries a call did not reach keep older values. Synchronises the device.
 * `bytes` is the size of dst; at most the whole trace (1 MiB) is copied.
 * Returns NVFP4_ERR_INVALID_ARG for a null dst, NVFP4_ERR_CUDA if the copy
 * fails. */
nvfp4_status nvfp4moe_stack_trace_read(void* dst, size_t bytes);

/* Copies the stage trace of the last launch of one tensor-core kernel to host
 * memory `dst`: kernel 0 the grouped up GEMM, 1 the grouped down GEMM (both
 * of moe_expert_forward above 4 tokens, W4A4), 2 the lm_head GEMM of
 * lm_head_forward above 8 tokens. Unsigned 64-bit SM clock readings (clock64)
 * [4 CTAs][11 events][1024 stages or items] (TcTraceEvent in
 * moe_grouped_tc.cuh: the producer's steps, operands landed and prepared,
 * MMAs issued per stage; item start, epilogue start and end per item).
 * Synchronises the device; at most 352 KiB are copied, and the kernel's
 * trace is then cleared (zeros: entries the next launch does not reach). Returns
 * NVFP4_ERR_INVALID_ARG for a null dst or an unknown kernel, NVFP4_ERR_CUDA
 * if the copy fails. */
nvfp4_status nvfp4moe_tc_trace_read(int32_t kernel, void* dst, size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_TRACE_H */
