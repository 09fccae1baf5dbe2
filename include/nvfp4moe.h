/*
 * nvfp4moe.h - C ABI of libnvfp4moe.so: the decode hot path of an
 * NVFP4-quantised, sigmoid-routed Mixture-of-Experts layer and the NVFP4
 * weight-only lm_head, as hand-written CUDA kernels for sm_103a (GB300).
 *
 * Sources (web pages on serving an NVFP4 Nemotron-3.5 MoE model):
 *   [worklog]   "Let's optimize Nemotron 3.5 Lightning - a worklog": Step 1
 *               (NVFP4: 4-bit values, group size 16; W4A16 keeps 16-bit
 *               activations), Step 3 (routed experts W4A4 with dynamic NVFP4
 *               activations), Step 4 (NVFP4 weight-only lm_head,
 *               131072 x 2688), Interlude (batch-1 decode is a weight stream).
 *   [card-w4a4] "nemotron35-w4a4-v13" model card, precision table.
 *   [card-int4] "NVIDIA-Nemotron-3.5-Lightning-30B-A3B-W4A16" model card,
 *               "Checkpoint layout" (per-expert up_proj / down_proj, no
 *               gate_proj) and "Left at bfloat16" (router .gate and its fp32
 *               e_score_correction_bias).
 *   [super-q]   "Quantization (PTQ + QAD)", Precision Recipes (router compute
 *               FP32; MoE and shared-expert GEMMs NVFP4) and Deployment
 *               (Blackwell runs W4A4).
 *
 * NVFP4 tensor (the canonical layout every call takes; moe_stack_forward also
 * reads a column-block copy of its down weights, nvfp4_colblock_layout), for
 * a matrix of n rows
 * and k columns (k % 16 == 0, element (r, c) = row r, reduction index c):
 *   codes  uint8 [n][k/2]   E2M1 codes, element 2j in the low nibble of byte j
 *   scales uint8 [n][k/16]  E4M3 (OCP "FN") scale of each 16-element block
 *   global float [1]        per-tensor scale (per row for activations)
 *   value(r, c) = E2M1(code) * E4M3(scale[r][c/16]) * global
 * Quantisation rule (the pages name the format and block size; the scale
 * formulas are this library's reading, stated once here):
 *   global  = amax(tensor) / (6 * 448)
 *   scale_b = E4M3_rn_satfinite( (amax(block b) / 6) / global )
 *   code_i  = E2M1_rn_satfinite( x_i / (E4M3(scale_b) * global) )
 * each step one IEEE binary32 operation, ties to even; a block whose
 * E4M3(scale_b) * global is 0 gets codes 0; the sign of a value that rounds
 * to 0 is kept (code 0x8).
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device pointers; the caller owns every
 *     buffer. The library never allocates or frees memory.
 *   - Every call is asynchronous on `stream`; arguments are checked on the host
 *     before anything is launched, and a rejected call launches nothing.
 *   - bf16 tensors are __nv_bfloat16 passed as `const void*` / `void*`.
 *   - Returned status codes are below; NVFP4_ERR_CUDA means a launch failed
 *     (cudaGetLastError() holds the CUDA error).
 *   - Device-side waits are bounded (1 s); a wait that expires makes its kernel
 *     stop early and sets a device error word, read by nvfp4_last_device_error.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside what the kernels handle */
    NVFP4_ERR_MISALIGNED = 3,        /* a pointer breaks the stated alignment */
    NVFP4_ERR_WORKSPACE = 4,         /* workspace too small */
    NVFP4_ERR_CUDA = 5,              /* a CUDA launch failed */
    NVFP4_ERR_TIMEOUT = 6            /* a bounded device wait expired */
} nvfp4_status;

typedef enum {
    NVFP4_GLOBAL_PER_TENSOR = 0, /* one global for the whole tensor (weights)   */
    NVFP4_GLOBAL_PER_ROW = 1,    /* one global per row (dynamic activations)    */
    NVFP4_GLOBAL_GIVEN = 2       /* global supplied by the caller               */
} nvfp4_global_mode;

typedef enum {
    NVFP4_W4A16 = 0, /* weights NVFP4, activations bf16 ([worklog] Step 1)        */
    NVFP4_W4A4 = 1   /* weights and activations NVFP4 ([worklog] Step 3)          */
} nvfp4_act_mode;

/* One NVFP4 matrix in the canonical layout; all three pointers are device
 * pointers; codes and scales 16-byte aligned. */
typedef struct {
    const uint8_t* codes;        /* [n][k/2]  */
    const uint8_t* scales;       /* [n][k/16] */
    const float* global_scale;   /* [1]       */
    int64_t n, k;
} nvfp4_matrix;

/* The weights of one MoE layer ([card-int4] "Checkpoint layout": routed experts
 * have up_proj [inter][hidden] and down_proj [hidden][inter], no gate_proj;
 * one shared expert). Routed expert tensors are stacked along a leading
 * expert axis; each expert matrix has its own per-tensor global. Device
 * pointers, codes/scales 16-byte aligned. */
typedef struct {
    int32_t num_experts;          /* E (128 in the pages' model)         */
    int32_t hidden;               /* H (2688)                            */
    int32_t inter;                /* I, routed intermediate (1856)       */
    int32_t shared_inter;         /* S, shared intermediate              */
    const uint8_t* up_codes;      /* [E][I][H/2]   */
    const uint8_t* up_scales;     /* [E][I][H/16]  */
    const float* up_global;       /* [E]           */
    const uint8_t* down_codes;    /* [E][H][I/2]   */
    const uint8_t* down_scales;   /* [E][H][I/16]  */
    const float* down_global;     /* [E]           */
    nvfp4_matrix shared_up;       /* [S][H] */
    nvfp4_matrix shared_down;     /* [H][S] */
} moe_layer_weights;

/*
 * nvfp4_quantize - NVFP4 quantisation of a row-major matrix x[rows][cols]
 * ([worklog] Step 1 format; per-row dynamic mode = [worklog] Step 3
 * "nvfp4_dynamic" activations). Used for weight registration (per tensor) and
 * for activations (per row).
 *   x            device, [rows][cols] bf16 (x_is_bf16 = 1) or float32 (0),
 *                16-byte aligned
 *   rows, cols   rows >= 0, cols > 0, cols % 16 == 0
 *   mode         PER_TENSOR: writes global_scale[0]; PER_ROW: writes
 *                global_scale[rows]; GIVEN: reads global_scale[0]
 *   codes        device out, [rows][cols/2], 8-byte aligned
 *   scales       device out, [rows][cols/16]
 * PER_TENSOR uses global_scale[0] as reduction scratch while it runs.
 * Codes and scales are bit-exact with the rule in the file header.
 */
nvfp4_status nvfp4_quantize(const void* x, int x_is_bf16, int64_t rows, int64_t cols,
                            nvfp4_global_mode mode, float* global_scale, uint8_t* codes,
                            uint8_t* scales, cudaStream_t stream);

/*
 * moe_route_topk - sigmoid router with correction bias ([card-int4] "Left at
 * bfloat16": .gate and fp32 e_score_correction_bias; [super-q] router compute
 * FP32), for T tokens:
 *   z_e = sum_i h_i Wg[e][i] (FP32); sigma_e = 1 / (1 + exp(-z_e));
 *   select the k largest sigma_e + bias_e (an exact tie goes to the lower
 *   index), in descending order;
 *   topk_w[j] = sigma_{e_j} / sum_l sigma_{e_l}.
 * h is the hidden row itself, or its RMS norm when rms_eps > 0 (see
 * moe_expert_forward).
 *   hidden    device bf16 [T][H], 16-byte aligned
 *   router_w  device float [E][H], 16-byte aligned
 *   bias      device float [E]
 *   T >= 1, H % 16 == 0, 1 <= k <= E <= 256, k <= 32
 *   rms_eps   > 0: normalise each hidden row first; <= 0: use it as is
 *   topk_idx  device out int32 [T][k];  topk_w device out float [T][k]
 */
nvfp4_status moe_route_topk(const void* hidden, const float* router_w, const float* bias,
                            int32_t T, int32_t H, int32_t E, int32_t k, float rms_eps,
                            int32_t* topk_idx, float* topk_w, cudaStream_t stream);

/*
 * moe_expert_forward_workspace_size - bytes of device workspace that
 * moe_expert_forward needs for these weights, T tokens, top-k and mode.
 */
size_t moe_expert_forward_workspace_size(const moe_layer_weights* w, int32_t T, int32_t k,
                                         nvfp4_act_mode mode);

/*
 * moe_expert_forward_workspace_init - zero a workspace before its first use.
 * moe_expert_forward keeps a small region of counters in the workspace and
 * leaves it zeroed when a call completes normally; after a call that reported
 * NVFP4_ERR_TIMEOUT, initialise the workspace again.
 */
nvfp4_status moe_expert_forward_workspace_init(void* workspace, size_t workspace_bytes,
                                               cudaStream_t stream);

/*
 * moe_expert_forward - routed experts + shared expert + combine of one MoE
 * layer for T tokens, given the routing:
 *   per token t, choice j, expert e = topk_idx[t][j]:
 *     u = up_e . x_t            (x_t: bf16 hidden row, or its per-row NVFP4
 *                                quantisation in W4A4)
 *     a = bf16(max(u, 0)^2)     (relu^2; bf16 intermediate)
 *     y = down_e . a'           (a': a, or its per-row NVFP4 quantisation)
 *   out_t = bf16( shared(x_t) + sum_j topk_w[t][j] * y_{t,j} [+ residual_t] )
 * with FP32 accumulation and one bf16 rounding at the end ([card-int4]
 * "Checkpoint layout" for the non-gated MLP; [super-q] for NVFP4 on the
 * shared expert too). x_t is the hidden row, or, when rms_eps > 0, its
 * unit-weight RMS norm bf16(h / sqrt(mean(h^2) + rms_eps)) -- the block input
 * norm of the pre-norm model the pages serve, whose norms stay in bf16
 * ([card-int4] "Left at bfloat16"); the residual is added un-normalised.
 *   w          weights (host struct holding device pointers); shapes must
 *              satisfy hidden, inter, shared_inter % 16 == 0 (the NVFP4
 *              block); widths that are not all multiples of 64 take the
 *              generic kernels (below), every other call here needs % 64
 *   hidden     device bf16 [T][H], 16-byte aligned
 *   topk_idx   device int32 [T][k], entries in [0, E) and distinct per token
 *   topk_w     device float [T][k]
 *   T >= 1, 1 <= k <= E (k <= 16 for T <= 4), E <= 256
 *   rms_eps    > 0: normalise each hidden row first; <= 0: use it as is
 *   residual   device bf16 [T][H] or NULL
 *   out        device bf16 [T][H]; may alias residual, must not alias hidden
 *              unless hidden == residual
 *   workspace  device, >= moe_expert_forward_workspace_size() bytes,
 *              256-byte aligned, zeroed once by
 *              moe_expert_forward_workspace_init; calls that share a
 *              workspace must not overlap in time
 */
/* Paths: T <= 4 streams the weight tiles of the step's unique experts through
 * persistent GEMV kernels (batch-1 decode and the 4-token verify, [worklog]
 * Interlude and Step 5); T > 4 groups the (token, choice) pairs by expert
 * (moe_permute) and runs the experts as one ragged grouped GEMM ([worklog]
 * Step 3). Widths off the 64 grid (any T) take generic kernels: one CTA per
 * (token, choice) and per token for the shared expert, a warp per output
 * row, then a combine kernel; the workspace is the T <= 4 path's. All paths
 * compute the same arithmetic; their FP32 summation orders differ. */
nvfp4_status moe_expert_forward(const moe_layer_weights* w, const void* hidden,
                                const int32_t* topk_idx, const float* topk_w, int32_t T,
                                int32_t k, nvfp4_act_mode mode, float rms_eps, const void* residual,
                                void* out, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * moe_permute - the token permutation of the grouped expert path ([worklog]
 * Step 3: the routed experts as a grouped GEMM over the tokens routed to
 * them). The T*k (token, choice) pairs p = t*k + j are grouped by expert
 * e = topk_idx[p], keeping pair order inside each expert:
 *   offsets[e] = number of pairs routed to experts < e   (offsets[E] = T*k)
 *   perm[pos]  = the pair at position pos                (position order)
 *   inv[p]     = the position of pair p                  (perm[inv[p]] == p)
 *   tile_offsets (optional, may be NULL): tile_offsets[e] = sum over experts
 *              < e of ceil(count / 64), the first 64-position tile of e.
 *   topk_idx   device int32 [T][k], entries in [0, E) (an entry outside is
 *              counted as expert 0 and reported by nvfp4_last_device_error)
 *   offsets    device int32 [E+1]; perm, inv: device int32 [T*k];
 *              tile_offsets: device int32 [E+1] or NULL
 *   1 <= k <= E <= 256 (NVFP4_ERR_UNSUPPORTED_SHAPE above 256)
 */
nvfp4_status moe_permute(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t* offsets,
                         int32_t* perm, int32_t* inv, int32_t* tile_offsets, cudaStream_t stream);

/*
 * moe_layer_forward - one whole MoE layer for 1..4 tokens in one call:
 * moe_route_topk followed by moe_expert_forward (same arithmetic, same
 * results), run as three kernels that hand their prepared operands to each
 * other through the workspace (routing plan, quantised activations) and
 * overlap each launch with the previous kernel's tail. The routing result is
 * also returned in topk_idx / topk_w.
 *   w, hidden, T, k, mode, rms_eps, residual, out: as moe_expert_forward
 *   router_w, bias: as moe_route_topk (device float [E][H], [E])
 *   topk_idx, topk_w: device out [T][k]
 *   T <= 4, k <= 16, E <= 256 (NVFP4_ERR_UNSUPPORTED_SHAPE otherwise)
 *   workspace: device, >= moe_layer_forward_workspace_size() bytes,
 *              256-byte aligned, zeroed once by
 *              moe_expert_forward_workspace_init and left zeroed by every
 *              completed call; calls that share it must not overlap.
 */
size_t moe_layer_forward_workspace_size(const moe_layer_weights* w, int32_t T, int32_t k,
                                        nvfp4_act_mode mode);
nvfp4_status moe_layer_forward(const moe_layer_weights* w, const float* router_w, const float* bias,
                               const void* hidden, int32_t T, int32_t k, nvfp4_act_mode mode,
                               float rms_eps, const void* residual, void* out, int32_t* topk_idx,
                               float* topk_w, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * moe_stack_forward - L consecutive MoE decode layers for 1..4 tokens in one
 * call: the residual chain of the pre-norm model the pages serve,
 *   h_{l+1} = h_l + moe_l(x_l),  x_l = RMSNorm(h_l) (or h_l if rms_eps <= 0),
 * where moe_l is the layer of moe_layer_forward (sigmoid + bias top-k router,
 * routed experts up -> relu^2 -> down, shared expert, gate-weighted combine;
 * [card-int4] "Checkpoint layout", [worklog] Interlude and Step 5). The
 * pre-norm is this library's reading: the pages name the layers but not the
 * blocks between them, and the bare chain overflows bf16 within a few
 * layers at the pages' shapes. It
 * runs as one persistent cooperative kernel with one CTA per SM: the layers'
 * steps meet in the workspace instead of at kernel boundaries (the router
 * logits and each layer's output as words tagged with their layer, which a
 * reader polls directly; counters for the rest), and the next layer's router
 * rows and shared-expert tiles are staged while
 * the current layer still waits on its routing. Each CTA takes 16-row units
 * of one expert's intermediate dimension (the shared expert's units go to a
 * fixed set of CTAs, each routed expert's to its share of the others) and
 * computes, per unit, 16 rows of W_up and then the matching 16 columns of
 * W_down (a split-K partial of the expert's output); so the down weights are
 * read from a column-block copy (nvfp4_colblock_layout), and the per-CTA
 * partials are added in a fixed order.
 *   layers     host array [L] of per-layer device pointers (copied into the
 *              launch; not read after the call returns); every layer has the
 *              same E, H, I, S with H, I, S % 64 == 0, H <= 3072, E % 8 == 0
 *              and E <= 256; router_w, router_bias, up_global, down_global and
 *              the two column-block copies 16-byte aligned. The row-major
 *              down weights in moe are not read: down_colblock must hold
 *              nvfp4_colblock_layout of down_codes / down_scales (batch E,
 *              rows H, cols I) and shared_down_colblock that of shared_down
 *              (batch 1, rows H, cols S).
 *   L          1 .. NVFP4MOE_STACK_MAX_LAYERS
 *   hidden_in  device bf16 [T][H] h_0, 16-byte aligned
 *   T, k       1 <= T <= 4, 1 <= k <= min(E, 16)
 *   hidden_out device bf16 [L][T][H]: h_1 .. h_L, 16-byte aligned, must not
 *              overlap hidden_in
 *   topk_idx, topk_w: device out [L][T][k], each layer's routing
 *   workspace  device, >= moe_stack_forward_workspace_size() bytes, 256-byte
 *              aligned, zeroed once by moe_expert_forward_workspace_init;
 *              every completed call leaves it ready for the next (counters
 *              zeroed, a call count advanced so that no tagged word left by
 *              one call matches the next); calls that share it must not
 *              overlap.
 * Summation orders differ from moe_layer_forward's (router dot products, the
 * split of tile reductions, the down projection split over 16-column blocks),
 * so results agree with it to FP32 rounding, not bit for bit; repeated calls
 * give identical bits. Returns NVFP4_ERR_UNSUPPORTED_SHAPE for shapes outside
 * the limits above, when one CTA per SM does not fit, when the GPU has fewer
 * SMs than min(T k, E) + 1 or when a CTA's share of a layer exceeds 32 units,
 * NVFP4_ERR_CUDA if the
 * cooperative launch fails; a device wait that expires ends every CTA of the
 * call early and is reported by nvfp4_last_device_error (NVFP4_ERR_TIMEOUT).
 */
#define NVFP4MOE_STACK_MAX_LAYERS 32
typedef struct {
    moe_layer_weights moe;
    const float* router_w;    /* [E][H], 16-byte aligned */
    const float* router_bias; /* [E], 16-byte aligned */
    const uint8_t* down_colblock;        /* [E][I/16][9 H] (nvfp4_colblock_layout) */
    const uint8_t* shared_down_colblock; /* [S/16][9 H] */
} moe_stack_layer;

/*
 * nvfp4_colblock_layout - the column-block copy of a batch of NVFP4 matrices
 * that moe_stack_forward reads its down weights from. Not an operation of
 * the pages: a storage order of the same codes and scales (the NVFP4 tensor
 * above, [worklog] Step 1: group size 16), so that one scale block of every
 * row (16 consecutive columns) sits together with the next rows' blocks.
 *   codes   device [batch][rows][cols/2] (two E2M1 codes a byte, low nibble
 *           first), scales device [batch][rows][cols/16] (E4M3), as every
 *           NVFP4 matrix here
 *   out     device [batch][cols/16][9 rows] bytes, 16-byte aligned: block c
 *           of matrix b holds columns 16c .. 16c + 15 of every row, codes
 *           [rows/32][32][8], then scales [rows/32][8][4]. Pair p covers rows
 *           32p .. 32p + 31 as two 16-row tiles m = 0, 1; byte 8L + 4m + i of
 *           its codes, L = 4g + q, holds row 32p + 16m + g (i = 0, 1) or that
 *           row + 8 (i = 2, 3), columns 16c + 4q + 2 (i & 1) and the next one;
 *           byte 4g + 2m + j of its scales holds the block scale of row
 *           32p + 16m + g + 8 j.
 *   rows % 32 == 0, cols % 16 == 0, batch >= 1; out must not overlap the
 *   inputs. NVFP4_ERR_INVALID_ARG / NVFP4_ERR_UNSUPPORTED_SHAPE /
 *   NVFP4_ERR_MISALIGNED (out) before anything is launched.
 */
nvfp4_status nvfp4_colblock_layout(const uint8_t* codes, const uint8_t* scales, int64_t batch, int64_t rows,
                                   int64_t cols, uint8_t* out, cudaStream_t stream);

size_t moe_stack_forward_workspace_size(const moe_stack_layer* layers, int32_t L, int32_t T, int32_t k,
                                        nvfp4_act_mode mode);
nvfp4_status moe_stack_forward(const moe_stack_layer* layers, int32_t L, const void* hidden_in, int32_t T,
                               int32_t k, nvfp4_act_mode mode, float rms_eps, void* hidden_out,
                               int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * moe_expert_forward_noalloc - moe_expert_forward for callers that cannot
 * allocate device memory. The pages have no counterpart to this call.
 *
 * Some hosts embed this layer without being able to give it a workspace:
 * for example an operator plugin whose host passes only the operator's
 * inputs and outputs and owns every device allocation, so the operator may
 * neither call cudaMalloc nor receive an extra buffer. This variant takes
 * the same arguments as moe_expert_forward minus the workspace and uses a
 * fixed scratch array that the library itself holds in device memory.
 *
 *   - Limit: the scratch is NVFP4MOE_NOALLOC_SCRATCH_BYTES (1 MiB) per GPU,
 *     held from library load until process exit. A call whose
 *     moe_expert_forward_workspace_size exceeds it is rejected with
 *     NVFP4_ERR_WORKSPACE before anything is launched (at the pages' layer
 *     shape this admits 1-4 tokens with top-6).
 *   - The first call in each CUDA context (per device: the primary context,
 *     or one made with cuCtxCreate or after cudaDeviceReset) looks up the
 *     scratch array's device address in that context, with its device
 *     current, and caches it under the context's id; make that first call
 *     before any stream capture. A driver without context ids makes every
 *     call look the address up again.
 *   - The arguments are checked exactly as moe_expert_forward checks them,
 *     before the scratch size is derived from them.
 *   - Each call clears the scratch region it uses on `stream` and leaves its
 *     contents behind; all calls on a device share the one array, so calls
 *     that overlap on the GPU (other streams, other threads) race. Order
 *     them on one stream or otherwise serialise them.
 *   - Nothing is allocated or freed: no cudaMalloc, cudaFree or allocating
 *     library routine is called.
 * Returns the same codes as moe_expert_forward.
 */
#define NVFP4MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
nvfp4_status moe_expert_forward_noalloc(const moe_layer_weights* w, const void* hidden,
                                        const int32_t* topk_idx, const float* topk_w, int32_t T,
                                        int32_t k, nvfp4_act_mode mode, float rms_eps,
                                        const void* residual, void* out, cudaStream_t stream);

/*
 * lm_head_gemv - NVFP4 weight-only lm_head ([worklog] Step 4; [card-w4a4]
 * "lm_head NVFP4 weight-only (W4A16)"):
 *   logits[t][v] = sum_j W[v][j] * h[t][j], FP32 accumulation and output;
 *   h is the hidden row, or its unit-weight RMS norm (the final norm before
 *   the head) when rms_eps > 0.
 *   w        NVFP4 matrix [V][H] (device pointers), V % 16 == 0, H % 16 == 0
 *            (H % 64 != 0 runs a generic kernel: a CTA per 64 rows x 8
 *            tokens, a warp per row; correct, not fast)
 *   hidden   device bf16 [T][H], 16-byte aligned;  T >= 1
 *   rms_eps  > 0: normalise each hidden row first; <= 0: use it as is
 *   logits   device float [T][V]
 */
nvfp4_status lm_head_gemv(const nvfp4_matrix* w, const void* hidden, int32_t T, float rms_eps,
                          float* logits, cudaStream_t stream);

/*
 * lm_head_forward - lm_head_gemv's computation for any token count, with a
 * workspace: up to 8 tokens it is lm_head_gemv; above, the hidden rows are
 * prepared once (RMS norm when rms_eps > 0, exact f16) and the head runs as
 * a dense GEMM over 64-token tiles (the 256-sequence concurrent decode of
 * the [card-w4a4] serving numbers), reading each weight tile once per 64
 * tokens instead of once per 8.
 *   w, hidden, T, rms_eps, logits: as lm_head_gemv; for T > 8 and
 *              H % 64 == 0 also V % 64 == 0 and logits 16-byte aligned
 *              (H % 64 != 0: the generic kernel for every T)
 *   workspace  device, >= lm_head_forward_workspace_size(w, T) bytes,
 *              256-byte aligned (unused for T <= 8)
 */
size_t lm_head_forward_workspace_size(const nvfp4_matrix* w, int32_t T);
nvfp4_status lm_head_forward(const nvfp4_matrix* w, const void* hidden, int32_t T, float rms_eps, float* logits,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * nvfp4_fp4_mma_peak - measures this GPU's dense FP4 tensor-pipe throughput
 * (no operation of the pages: the denominator of the FP4 roofline fraction
 * reported for the grouped W4A4 path, [super-q] "Deployment" Blackwell W4A4).
 * One CTA per SM issues `iters` tcgen05.mma kind::mxf4nvf4 block-scaled MMAs
 * (M = 128, N = n, K = 64, E2M1 x E2M1 with E4M3 scales per 16 elements) from
 * shared-memory operands into `chains` tensor-memory accumulators; a warm-up
 * launch, then one launch timed with CUDA events on `stream`.
 *   n       32 .. 256, a multiple of 32;  chains >= 1 with chains * n <= 448
 *   iters   MMAs per CTA (>= 1; ~20000 keeps a launch near a millisecond)
 *   tflops  host out: 2 * 128 * n * 64 * iters * SMs / seconds / 1e12
 * Synchronises `stream`. Allocates no device memory (two CUDA events).
 * Returns NVFP4_ERR_INVALID_ARG for arguments outside these ranges,
 * NVFP4_ERR_CUDA if a launch or the timing fails.
 */
nvfp4_status nvfp4_fp4_mma_peak(int32_t n, int32_t chains, int32_t iters, double* tflops, cudaStream_t stream);

/* Backend choice by batch size ([super-q] "Deployment": per-quantization GEMM
 * backend selection at intermediate batch sizes): moe_expert_forward runs
 * 1 .. t tokens on the decode GEMV kernels (weights decoded in registers,
 * tokens as MMA columns) and more on the grouped tensor-core path (W4A4:
 * tcgen05 block-scaled MMA; W4A16: the f16 grouped GEMM). t in 0 .. 4,
 * default 4. Process-wide; moe_expert_forward_workspace_size follows it, so
 * size workspaces after setting it (a smaller workspace is rejected with
 * NVFP4_ERR_WORKSPACE). Returns NVFP4_ERR_INVALID_ARG for t outside 0 .. 4. */
nvfp4_status nvfp4_set_decode_max_tokens(int32_t t);

/* Sets, on the current device, the limit of the device waits of one CTA on
 * another CTA's progress (moe_stack_forward's polls of its tagged words):
 * `ns` nanoseconds, or the default 1 s when ns is 0. A wait that runs out
 * ends every CTA of its call early, and the next nvfp4_last_device_error
 * returns NVFP4_ERR_TIMEOUT; the context stays usable, and a workspace
 * re-initialised with moe_expert_forward_workspace_init serves the next call.
 * Waits on a CTA's own staging copies keep 1 s. Not an operation of the
 * pages: a watchdog setting (a short limit makes the failure path testable).
 * Synchronous; affects calls launched afterwards. Returns NVFP4_ERR_CUDA if
 * the device copy fails. */
nvfp4_status nvfp4_set_peer_wait_limit(uint64_t ns);

/* Inspection of the activation rows a call leaves in its workspace (no
 * operation of the pages: it lets a test compare the NVFP4 activation rows
 * the kernels build in flight, [worklog] Step 3 "W4A4", with a reference
 * quantiser bit for bit). After moe_expert_forward (call 0) or
 * moe_layer_forward (call 1) with the same w, T, k and mode, `view` gets the
 * place of region `region` in the workspace:
 *   NVFP4_WS_X        the layer input rows as the up GEMMs take them [T][H]
 *                     (after the RMS norm when rms_eps > 0)
 *   NVFP4_WS_ACT      the routed intermediate relu(up)^2 in bf16 [T*k][I]
 *   NVFP4_WS_ACT_Q    the same rows quantised, as the down GEMMs take them
 *   NVFP4_WS_SH_ACT   the shared expert's intermediate in bf16 [T][S]
 *   NVFP4_WS_SH_ACT_Q the same rows quantised
 * format NVFP4_WS_BF16: bf16 values. NVFP4_WS_CODES: E2M1 codes [rows][cols/2]
 * (low nibble = even element) with E4M3 scales at scales_offset, scales_pitch
 * bytes per row, and per-row FP32 globals at global_offset (W4A4).
 * NVFP4_WS_F16_DEQUANT: per element the f16 value E2M1 code x E4M3 scale (exact),
 * per-row globals at global_offset. Rows are in (token, choice) order, or
 * in the permuted position order (grouped by expert) when position_order = 1;
 * row p of ACT and of ACT_Q are the same row either way.
 * Regions a path keeps only in shared memory (the decode GEMV path's
 * quantised rows; every quantised row of a W4A16 call; the W4A16 grouped
 * path) give NVFP4_ERR_UNSUPPORTED_SHAPE. Host only; reads no device memory.
 * Returns NVFP4_ERR_INVALID_ARG for a null w or view or an unknown call,
 * mode or region. */
typedef enum {
    NVFP4_WS_X = 0,
    NVFP4_WS_ACT = 1,
    NVFP4_WS_ACT_Q = 2,
    NVFP4_WS_SH_ACT = 3,
    NVFP4_WS_SH_ACT_Q = 4
} nvfp4_ws_region;

typedef enum { NVFP4_WS_BF16 = 0, NVFP4_WS_CODES = 1, NVFP4_WS_F16_DEQUANT = 2 } nvfp4_ws_format;

typedef struct {
    uint64_t offset;         /* byte offset of row 0 */
    int64_t rows, cols;      /* elements */
    int64_t pitch;           /* bytes between rows */
    uint64_t scales_offset;  /* NVFP4_WS_CODES: E4M3 scales of row 0 */
    int64_t scales_pitch;    /* bytes between scale rows */
    uint64_t global_offset;  /* FP32 [rows] per-row globals when has_global */
    int32_t format;          /* nvfp4_ws_format */
    int32_t has_global;
    int32_t position_order;
    int32_t reserved;
} nvfp4_ws_view;

nvfp4_status nvfp4_workspace_view(int32_t call, const moe_layer_weights* w, int32_t T, int32_t k,
                                  nvfp4_act_mode mode, int32_t region, nvfp4_ws_view* view);

/* ---------------------------------------------------------------- FP8 W8A8
 * The shared expert in FP8 per-tensor W8A8, the precision the W4A4 card's
 * table gives the shared experts ([card-w4a4] precision table: "Mamba
 * in_proj / out_proj, shared experts: FP8 per-tensor W8A8"; [worklog] Step 3
 * quant config: shared experts "num_bits: e4m3").
 *
 * FP8 tensor: codes uint8 [n][k] E4M3 (OCP "FN"), one FP32 scale;
 * value(r, c) = E4M3(code) * scale. Quantisation (this library's reading,
 * binary32, ties to even):
 *   scale = amax / 448;   code_i = E4M3_rn_satfinite( x_i / scale )
 * a scale of 0 (an all-zero tensor or row) gives codes 0 with the sign kept.
 */
typedef struct {
    const uint8_t* codes;      /* [n][k] E4M3 */
    const float* global_scale; /* [1] */
    int64_t n, k;
} fp8_matrix;

/* fp8_quantize - x [rows][cols] (bf16 if x_is_bf16, else fp32; device,
 * 16-byte aligned, cols % 16 == 0) to E4M3 codes [rows][cols] (device,
 * 16-byte aligned) with the scale of `mode`: NVFP4_GLOBAL_PER_TENSOR writes
 * amax / 448 to global_scale[0]; PER_ROW writes one per row to
 * global_scale[r]; GIVEN reads global_scale[0]. Asynchronous on `stream`.
 * Returns NVFP4_ERR_UNSUPPORTED_SHAPE for cols % 16, NVFP4_ERR_MISALIGNED,
 * NVFP4_ERR_INVALID_ARG for null pointers or an unknown mode. */
nvfp4_status fp8_quantize(const void* x, int x_is_bf16, int64_t rows, int64_t cols, nvfp4_global_mode mode,
                          float* global_scale, uint8_t* codes, cudaStream_t stream);

/* moe_shared_fp8_forward - the shared expert in FP8 W8A8 for T tokens:
 *   x   = RMSNorm(hidden) when rms_eps > 0 (the same unit-weight norm as the
 *         other calls), else hidden
 *   x_q = FP8(x) per token row;   u = up . x_q  (scales applied in FP32)
 *   a   = bf16(relu(u)^2);        a_q = FP8(a) per token row
 *   out = bf16(down . a_q + residual)   (residual may be null)
 * A layer whose shared expert is FP8 adds it to the routed experts' output by
 * passing that output as `residual` (two bf16 roundings: this library's
 * reading of a separately launched FP8 GEMM).
 *   up        fp8_matrix [S][H];  down fp8_matrix [H][S]; H, S % 64 == 0,
 *             H, S <= 2^20; 8 * H and 8 * S bytes within a CTA's shared
 *             memory (each CTA quantises the token rows its GEMV needs
 *             itself)
 *   hidden    device bf16 [T][H], 16-byte aligned; residual, out bf16 [T][H]
 *   workspace device, >= moe_shared_fp8_workspace_size(up, T) bytes,
 *             256-byte aligned (the bf16 intermediate; no zeroing needed)
 * Tokens run in chunks of 8 (the MMA's columns), two launches per chunk.
 * Asynchronous on `stream`.
 * Returns NVFP4_ERR_INVALID_ARG / _UNSUPPORTED_SHAPE / _MISALIGNED /
 * _WORKSPACE on bad arguments, before any launch. */
size_t moe_shared_fp8_workspace_size(const fp8_matrix* up, int32_t T);
nvfp4_status moe_shared_fp8_forward(const fp8_matrix* up, const fp8_matrix* down, const void* hidden, int32_t T,
                                    float rms_eps, const void* residual, void* out, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* nvfp4_status_string(nvfp4_status status);

/* Synchronises `stream`, then reads and clears the device error word: returns
 * NVFP4_ERR_TIMEOUT if a bounded device wait expired since the last read,
 * NVFP4_ERR_INVALID_ARG if a kernel met an invalid device-side input (an
 * expert index outside [0, E)), NVFP4_ERR_CUDA if the synchronisation itself
 * failed, else NVFP4_OK. */
nvfp4_status nvfp4_last_device_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
