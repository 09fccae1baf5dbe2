// nvfp4moe.cu - the C ABI of libnvfp4moe.so (declared in include/nvfp4moe.h):
// argument checks on the host, launch configuration, and dispatch to the
// kernels in the headers below. One translation unit, so that the device
// error word is a single object.
#include "nvfp4moe.h"
#if defined(NVFP4MOE_TRACE)
#include "nvfp4moe_trace.h"
#endif

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "fp4_peak.cuh"
#include "fp8.cuh"
#include "lm_head.cuh"
#include "lm_head_tc.cuh"
#include "moe_decode.cuh"
#include "moe_grouped.cuh"
#include "moe_generic.cuh"
#include "moe_grouped_tc.cuh"
#include "moe_layer.cuh"
#include "moe_stack.cuh"
#include "quantize.cuh"
#include "route.cuh"

using namespace nvfp4moe;

namespace {

constexpr int kMaxDevices = 64;

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

// The host-side caches below are shared by every thread that calls the
// library; each is read and filled under its own mutex.
int num_sms() {
    static int cache[kMaxDevices] = {0};
    static std::mutex mu;
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[d] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
        cache[d] = v > 0 ? v : 1;
    }
    return cache[d];
}

int smem_optin() {
    static int cache[kMaxDevices] = {0};
    static std::mutex mu;
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return 48 * 1024;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[d] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
        cache[d] = v > 0 ? v : 48 * 1024;
    }
    return cache[d];
}

// Unique id of the calling thread's current CUDA context (never reused
// within the process), from the driver; 0 if the driver does not provide it.
unsigned long long current_context_id() {
    using CtxGetCurrentFn = CUresult (*)(CUcontext*);
    using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Largest dynamic shared memory a kernel may use (opt-in limit minus its
// static shared memory); raises the kernel's limit to that value once per
// (kernel, device, context): a kernel's attributes belong to the module
// loaded in one context. Kernels are told apart by address: template
// instances with one signature share a type.
int dyn_smem_limit(const void* kernel) {
    struct Entry {
        const void* fn;
        unsigned long long ctx;
        int dev, lim;
    };
    static Entry table[256];
    static int used = 0;
    static std::mutex mu;
    const int d = current_device();
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (ctx != 0)
        for (int i = 0; i < used; ++i)
            if (table[i].fn == kernel && table[i].dev == d && table[i].ctx == ctx) return table[i].lim;
    cudaFuncAttributes at;
    if (cudaFuncGetAttributes(&at, kernel) != cudaSuccess) return 0;
    const int lim = smem_optin() - static_cast<int>(at.sharedSizeBytes) - 64;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim) != cudaSuccess)
        return 0;
    if (ctx != 0) {
        if (used < 256) table[used++] = Entry{kernel, ctx, d, lim};
        else table[ctx % 256] = Entry{kernel, ctx, d, lim};
    }
    return lim;
}

template <typename Kernel>
int dyn_smem_limit(Kernel k) {
    return dyn_smem_limit(reinterpret_cast<const void*>(k));
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline nvfp4_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Launch with programmatic stream serialisation: the kernel may start while
// the previous one in the stream finishes (it calls pdl_wait() before reading
// that kernel's results).
template <typename... KArgs, typename... Args>
nvfp4_status launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t stream,
                        Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) return NVFP4_ERR_CUDA;
    return launch_status();
}

// ------------------------------------------------------------ workspace
struct DecodeWs {
    size_t act, act_sh, ypart, ysh, tilecnt, total;
};

DecodeWs decode_ws(int T, int k, int H, int I, int S) {
    DecodeWs w{};
    size_t off = 0;
    w.tilecnt = off;
    off += align256(sizeof(int) * (size_t)(H / 16));
    w.act = off;
    off += align256((size_t)T * k * I * 2);
    w.act_sh = off;
    off += align256((size_t)T * S * 2);
    w.ypart = off;
    off += align256((size_t)T * k * H * 4);
    w.ysh = off;
    off += align256((size_t)T * H * 4);
    w.total = off;
    return w;
}

// Widths that are multiples of 16 but not of 64 (moe_generic.cuh): up for
// every (token, slot) and the shared expert, then down, then the combine.
nvfp4_status generic_forward(const moe_layer_weights* w, const void* hidden, const int32_t* topk_idx,
                             const float* topk_w, int T, int k, bool w4a4, float rms_eps, const void* residual,
                             void* out, uint8_t* ws, cudaStream_t stream) {
    const int H = w->hidden, I = w->inter, S = w->shared_inter;
    const DecodeWs o = decode_ws(T, k, H, I, S);
    const size_t smem_up = ((2 * (size_t)H + 15) & ~size_t(15)) + 4 * (size_t)H;
    const size_t smem_dn = 4 * (size_t)std::max(I, S);
    if ((int64_t)smem_up > dyn_smem_limit(k_gen_up) || (int64_t)smem_dn > dyn_smem_limit(k_gen_down))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)T * (k + 1) > (1LL << 30) || (int64_t)T * H > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    GenArgs ua{};
    ua.codes = w->up_codes;
    ua.scales = w->up_scales;
    ua.global = w->up_global;
    ua.sh_codes = w->shared_up.codes;
    ua.sh_scales = w->shared_up.scales;
    ua.sh_global = w->shared_up.global_scale;
    ua.E = w->num_experts;
    ua.n = I;
    ua.K = H;
    ua.n_sh = S;
    ua.K_sh = H;
    ua.src = static_cast<const uint16_t*>(hidden);
    ua.rms_eps = rms_eps;
    ua.topk_idx = topk_idx;
    ua.topk_w = topk_w;
    ua.T = T;
    ua.k = k;
    ua.w4a4 = w4a4;
    ua.act = reinterpret_cast<uint16_t*>(ws + o.act);
    ua.act_sh = reinterpret_cast<uint16_t*>(ws + o.act_sh);
    k_gen_up<<<T * (k + 1), kGenThreads, smem_up, stream>>>(ua);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    GenArgs da = ua;
    da.codes = w->down_codes;
    da.scales = w->down_scales;
    da.global = w->down_global;
    da.sh_codes = w->shared_down.codes;
    da.sh_scales = w->shared_down.scales;
    da.sh_global = w->shared_down.global_scale;
    da.n = H;
    da.K = I;
    da.n_sh = H;
    da.K_sh = S;
    da.src = ua.act;
    da.src_sh = ua.act_sh;
    da.rms_eps = 0.0f;
    da.ypart = reinterpret_cast<float*>(ws + o.ypart);
    da.ysh = reinterpret_cast<float*>(ws + o.ysh);
    k_gen_down<<<T * (k + 1), kGenThreads, smem_dn, stream>>>(da);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    k_gen_combine<<<(T * H + kGenThreads - 1) / kGenThreads, kGenThreads, 0, stream>>>(
        da.ypart, da.ysh, T, k, H, static_cast<const uint16_t*>(residual), static_cast<uint16_t*>(out));
    return launch_status();
}

// The grouped path (T > 4, moe_grouped.cuh), defined below.
size_t grouped_ws_total(int T, int k, int E, int H, int I, int S);
nvfp4_status grouped_forward(const moe_layer_weights* w, const void* hidden, const int32_t* topk_idx,
                             const float* topk_w, int T, int k, bool w4a4, float rms_eps, const void* residual,
                             void* out, uint8_t* ws, cudaStream_t stream);

// The largest token count moe_expert_forward runs on the decode GEMV kernels
// (nvfp4_set_decode_max_tokens); more tokens take the grouped path.
std::atomic<int> g_decode_max_t{kDecodeMaxT};

bool decode_path(const moe_layer_weights* w, int T, int k) {
    return T >= 1 && T <= g_decode_max_t.load(std::memory_order_relaxed) && k <= kDecodeMaxK && w->num_experts <= 256;
}

nvfp4_status check_matrix(const nvfp4_matrix& m, int64_t n, int64_t k) {
    if (!m.codes || !m.scales || !m.global_scale) return NVFP4_ERR_INVALID_ARG;
    if (m.n != n || m.k != k) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(m.codes, 16) || !aligned(m.scales, 16)) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

// A layer whose widths are multiples of 16 but not all of 64: only
// moe_expert_forward takes it (the generic kernels); every other layer call
// needs multiples of 64.
bool generic_shape(const moe_layer_weights* w) { return w->hidden % 64 || w->inter % 64 || w->shared_inter % 64; }

// kmod: the multiple the widths must be (64; 16 for moe_expert_forward)
nvfp4_status check_layer(const moe_layer_weights* w, int kmod = 64) {
    if (!w) return NVFP4_ERR_INVALID_ARG;
    if (w->num_experts < 1 || w->hidden < 1 || w->inter < 1 || w->shared_inter < 1)
        return NVFP4_ERR_INVALID_ARG;
    if (!w->up_codes || !w->up_scales || !w->up_global || !w->down_codes || !w->down_scales ||
        !w->down_global)
        return NVFP4_ERR_INVALID_ARG;
    if (w->hidden % kmod || w->inter % kmod || w->shared_inter % kmod) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w->up_codes, 16) || !aligned(w->up_scales, 16) || !aligned(w->down_codes, 16) ||
        !aligned(w->down_scales, 16))
        return NVFP4_ERR_MISALIGNED;
    nvfp4_status s = check_matrix(w->shared_up, w->shared_inter, w->hidden);
    if (s != NVFP4_OK) return s;
    return check_matrix(w->shared_down, w->hidden, w->shared_inter);
}

}  // namespace

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_INVALID_ARG: return "invalid argument";
        case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case NVFP4_ERR_MISALIGNED: return "misaligned pointer";
        case NVFP4_ERR_WORKSPACE: return "workspace too small";
        case NVFP4_ERR_CUDA: return "CUDA error";
        case NVFP4_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

nvfp4_status nvfp4_set_decode_max_tokens(int32_t t) {
    if (t < 0 || t > kDecodeMaxT) return NVFP4_ERR_INVALID_ARG;
    g_decode_max_t.store(t, std::memory_order_relaxed);
    return NVFP4_OK;
}

nvfp4_status nvfp4_set_peer_wait_limit(uint64_t ns) {
    const unsigned long long v = ns == 0 ? kWaitTimeoutNs : static_cast<unsigned long long>(ns);
    return cudaMemcpyToSymbol(g_peer_wait_ns, &v, sizeof(v)) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_last_device_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(v)) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero)) != cudaSuccess) return NVFP4_ERR_CUDA;
        return (v & (kErrWaitFull | kErrWaitEmpty | kErrWaitDrain | kErrWaitPeer)) ? NVFP4_ERR_TIMEOUT
                                                                      : NVFP4_ERR_INVALID_ARG;
    }
    return NVFP4_OK;
}

#if defined(NVFP4MOE_TRACE)
nvfp4_status nvfp4moe_stack_trace_read(void* dst, size_t bytes) {
    if (!dst) return NVFP4_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
    const size_t n = std::min(bytes, sizeof(g_stack_trace));
    return cudaMemcpyFromSymbol(dst, g_stack_trace, n) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4moe_tc_trace_read(int32_t kernel, void* dst, size_t bytes) {
    if (!dst || kernel < 0 || kernel > 2) return NVFP4_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
    const size_t one = sizeof(g_tc_trace) / 3;
    const size_t n = std::min(bytes, one);
    if (cudaMemcpyFromSymbol(dst, g_tc_trace, n, one * kernel) != cudaSuccess) return NVFP4_ERR_CUDA;
    void* base = nullptr;  // cleared, so that the next read holds only the next launch's entries
    if (cudaGetSymbolAddress(&base, g_tc_trace) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (cudaMemset(static_cast<uint8_t*>(base) + one * kernel, 0, one) != cudaSuccess) return NVFP4_ERR_CUDA;
    return cudaDeviceSynchronize() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
#endif

nvfp4_status nvfp4_quantize(const void* x, int x_is_bf16, int64_t rows, int64_t cols,
                            nvfp4_global_mode mode, float* global_scale, uint8_t* codes,
                            uint8_t* scales, cudaStream_t stream) {
    if (!global_scale || rows < 0 || cols <= 0) return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_GLOBAL_PER_TENSOR && mode != NVFP4_GLOBAL_PER_ROW && mode != NVFP4_GLOBAL_GIVEN)
        return NVFP4_ERR_INVALID_ARG;
    if (cols % 16) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) {
        if (mode == NVFP4_GLOBAL_PER_TENSOR) {
            if (cudaMemsetAsync(global_scale, 0, sizeof(float), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
        }
        return NVFP4_OK;
    }
    if (!x || !codes || !scales) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(codes, 8)) return NVFP4_ERR_MISALIGNED;
    const int64_t nblocks = rows * (cols / 16);
    const int maxg = num_sms() * 8;
    const int grid = static_cast<int>(std::min<int64_t>((nblocks + 255) / 256, maxg));
    const bool bf16 = x_is_bf16 != 0;
    if (mode == NVFP4_GLOBAL_PER_ROW) {
        const int rgrid = static_cast<int>(std::min<int64_t>((rows + 7) / 8, maxg));
        if (bf16) k_quantize_rows<true><<<rgrid, 256, 0, stream>>>(x, rows, cols, global_scale, codes, scales);
        else k_quantize_rows<false><<<rgrid, 256, 0, stream>>>(x, rows, cols, global_scale, codes, scales);
        return launch_status();
    }
    if (mode == NVFP4_GLOBAL_PER_TENSOR) {
        if (cudaMemsetAsync(global_scale, 0, sizeof(float), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
        unsigned int* bits = reinterpret_cast<unsigned int*>(global_scale);
        if (bf16) k_amax<true><<<grid, 256, 0, stream>>>(x, nblocks, bits);
        else k_amax<false><<<grid, 256, 0, stream>>>(x, nblocks, bits);
    }
    const int from_amax = mode == NVFP4_GLOBAL_PER_TENSOR ? 1 : 0;
    if (bf16) k_quantize_global<true><<<grid, 256, 0, stream>>>(x, nblocks, global_scale, from_amax, codes, scales);
    else k_quantize_global<false><<<grid, 256, 0, stream>>>(x, nblocks, global_scale, from_amax, codes, scales);
    if (mode == NVFP4_GLOBAL_PER_TENSOR) k_finalize_global<<<1, 1, 0, stream>>>(global_scale);
    return launch_status();
}

// From this many tokens on the router runs as k_route_rows (one CTA per 8
// tokens and every expert: a single wave of T / 8 CTAs that read the gate
// rows from L2) instead of clusters that split the experts (T / 8 x 8 CTAs,
// several waves at prefill sizes).
constexpr int kRouteManyTokens = 512;

nvfp4_status moe_route_topk(const void* hidden, const float* router_w, const float* bias, int32_t T,
                            int32_t H, int32_t E, int32_t k, float rms_eps, int32_t* topk_idx,
                            float* topk_w, cudaStream_t stream) {
    if (!hidden || !router_w || !bias || !topk_idx || !topk_w) return NVFP4_ERR_INVALID_ARG;
    if (T < 1 || H < 16 || E < 1 || k < 1 || k > E) return NVFP4_ERR_INVALID_ARG;
    if (H % 16 || E > 256 || k > 32) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(hidden, 16) || !aligned(router_w, 16)) return NVFP4_ERR_MISALIGNED;
    // Small batches: the cluster's gate rows staged in shared memory. Large
    // batches: gate rows read from L2 (where the 1.4 MB matrix stays), so that
    // a CTA needs shared memory only for its token rows and many fit per SM.
    auto launch = [&](auto kernel, int TT) {
        const int lim = dyn_smem_limit(kernel);
        const int hbytes = TT * H * 2;
        const int nj = (E + kRouteCluster - 1) / kRouteCluster;  // gate rows of CTA rank 0
        const int stage_w = T < 64 && hbytes + nj * H * 4 <= lim ? 1 : 0;
        const int smem = hbytes + (stage_w ? nj * H * 4 : 0);
        if (smem > lim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        const int tiles = (T + TT - 1) / TT;
        return launch_pdl(kernel, tiles * kRouteCluster, kRouteWarps * 32, smem, stream,
                          static_cast<const uint16_t*>(hidden), router_w, bias, T, H, E, k, rms_eps, stage_w,
                          topk_idx, topk_w, static_cast<DecodePlan*>(nullptr), static_cast<__half*>(nullptr),
                          static_cast<float*>(nullptr), 0);
    };
    if (T >= kRouteManyTokens) {  // many tokens: one CTA per 8 tokens and every expert
        const int smem = kRouteRowsTile * H * 2;
        if (smem > dyn_smem_limit(k_route_rows)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        return launch_pdl(k_route_rows, (T + kRouteRowsTile - 1) / kRouteRowsTile, kConsumerThreads, smem, stream,
                          static_cast<const uint16_t*>(hidden), router_w, bias, T, H, E, k, rms_eps, topk_idx,
                          topk_w);
    }
    return launch(k_route<8>, 8);
}

size_t moe_expert_forward_workspace_size(const moe_layer_weights* w, int32_t T, int32_t k,
                                         nvfp4_act_mode mode) {
    (void)mode;
    if (!w || T < 1 || k < 1) return 0;
    if (decode_path(w, T, k) || generic_shape(w)) return decode_ws(T, k, w->hidden, w->inter, w->shared_inter).total;
    return grouped_ws_total(T, k, w->num_experts, w->hidden, w->inter, w->shared_inter);
}

nvfp4_status moe_expert_forward_workspace_init(void* workspace, size_t workspace_bytes,
                                               cudaStream_t stream) {
    if (!workspace) return NVFP4_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, stream) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status moe_expert_forward(const moe_layer_weights* w, const void* hidden,
                                const int32_t* topk_idx, const float* topk_w, int32_t T, int32_t k,
                                nvfp4_act_mode mode, float rms_eps, const void* residual, void* out,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    nvfp4_status st = check_layer(w, 16);
    if (st != NVFP4_OK) return st;
    if (!hidden || !topk_idx || !topk_w || !out || !workspace) return NVFP4_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || k > w->num_experts) return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_W4A16 && mode != NVFP4_W4A4) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(out, 4) || !aligned(workspace, 256) ||
        (residual && !aligned(residual, 4)))
        return NVFP4_ERR_MISALIGNED;
    if (hidden == out && residual != hidden) return NVFP4_ERR_INVALID_ARG;
    if (generic_shape(w)) {
        if (workspace_bytes < decode_ws(T, k, w->hidden, w->inter, w->shared_inter).total)
            return NVFP4_ERR_WORKSPACE;
        return generic_forward(w, hidden, topk_idx, topk_w, T, k, mode == NVFP4_W4A4, rms_eps, residual, out,
                               static_cast<uint8_t*>(workspace), stream);
    }
    if (!decode_path(w, T, k)) {
        // more than 4 tokens: grouped GEMM over the tokens each expert received
        if (w->num_experts > 256) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        if (workspace_bytes < grouped_ws_total(T, k, w->num_experts, w->hidden, w->inter, w->shared_inter))
            return NVFP4_ERR_WORKSPACE;
        return grouped_forward(w, hidden, topk_idx, topk_w, T, k, mode == NVFP4_W4A4, rms_eps, residual, out,
                               static_cast<uint8_t*>(workspace), stream);
    }

    const int H = w->hidden, I = w->inter, S = w->shared_inter;
    const DecodeWs ws = decode_ws(T, k, H, I, S);
    if (workspace_bytes < ws.total) return NVFP4_ERR_WORKSPACE;
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    const bool w4a4 = mode == NVFP4_W4A4;
    const int nsm = num_sms();
    // enough CTAs that each one's item range spans at most two routed experts
    const int grid = std::max(nsm, 2 * (T * k + (S + I - 1) / I) + 4);

    UpArgs ua{};
    ua.codes = w->up_codes;
    ua.scales = w->up_scales;
    ua.global = w->up_global;
    ua.sh_codes = w->shared_up.codes;
    ua.sh_scales = w->shared_up.scales;
    ua.sh_global = w->shared_up.global_scale;
    ua.E = w->num_experts;
    ua.H = H;
    ua.I = I;
    ua.S = S;
    ua.hidden = static_cast<const uint16_t*>(hidden);
    ua.rms_eps = rms_eps;
    ua.topk_idx = topk_idx;
    ua.topk_w = topk_w;
    ua.T = T;
    ua.k = k;
    ua.act = reinterpret_cast<uint16_t*>(wsb + ws.act);
    ua.act_sh = reinterpret_cast<uint16_t*>(wsb + ws.act_sh);
    {
        const int lim = w4a4 ? dyn_smem_limit(k_moe_up_decode<true>) : dyn_smem_limit(k_moe_up_decode<false>);
        const int bbytes = 2 * T * H * 2;  // f16 B rows + normalised bf16 rows
        const int stage = 9 * H;
        ua.ring_bytes = std::min(kMaxStages * stage, ((lim - bbytes) / 128) * 128);
        if (ua.ring_bytes < 2 * stage) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        const int smem = ua.ring_bytes + bbytes;
        st = w4a4 ? launch_pdl(k_moe_up_decode<true>, grid, kThreads, smem, stream, ua)
                  : launch_pdl(k_moe_up_decode<false>, grid, kThreads, smem, stream, ua);
        if (st != NVFP4_OK) return st;
    }

    DownArgs da{};
    da.codes = w->down_codes;
    da.scales = w->down_scales;
    da.global = w->down_global;
    da.sh_codes = w->shared_down.codes;
    da.sh_scales = w->shared_down.scales;
    da.sh_global = w->shared_down.global_scale;
    da.E = w->num_experts;
    da.H = H;
    da.I = I;
    da.S = S;
    da.topk_idx = topk_idx;
    da.topk_w = topk_w;
    da.T = T;
    da.k = k;
    da.act = ua.act;
    da.act_sh = ua.act_sh;
    da.residual = static_cast<const uint16_t*>(residual);
    da.out = static_cast<uint16_t*>(out);
    da.ypart = reinterpret_cast<float*>(wsb + ws.ypart);
    da.ysh = reinterpret_cast<float*>(wsb + ws.ysh);
    da.tilecnt = reinterpret_cast<int*>(wsb + ws.tilecnt);
    {
        const int lim = w4a4 ? dyn_smem_limit(k_moe_down_decode<true>) : dyn_smem_limit(k_moe_down_decode<false>);
        const int bbytes = (2 * T * I + T * S) * 2;
        const int stage = 9 * std::max(I, S);
        da.ring_bytes = std::min(kMaxStages * stage, ((lim - bbytes) / 128) * 128);
        if (da.ring_bytes < 2 * stage) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        const int smem = da.ring_bytes + bbytes;
        st = w4a4 ? launch_pdl(k_moe_down_decode<true>, grid, kThreads, smem, stream, da)
                  : launch_pdl(k_moe_down_decode<false>, grid, kThreads, smem, stream, da);
    }
    return st;
}

// The lm_head for a hidden width that is a multiple of 16 but not of 64
// (moe_generic.cuh), any token count.
nvfp4_status lm_head_generic(const nvfp4_matrix* w, const void* hidden, int32_t T, float rms_eps, float* logits,
                             cudaStream_t stream) {
    const int H = static_cast<int>(w->k), V = static_cast<int>(w->n);
    const size_t smem = (size_t)kGenLmTok * H * 6;
    if ((int64_t)smem > dyn_smem_limit(k_gen_lm_head) || w->n > (1 << 30) || (T + kGenLmTok - 1) / kGenLmTok > 65535)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const dim3 grid((V + kGenLmRows - 1) / kGenLmRows, (T + kGenLmTok - 1) / kGenLmTok);
    k_gen_lm_head<<<grid, kGenThreads, smem, stream>>>(w->codes, w->scales, w->global_scale, V, H,
                                                       static_cast<const uint16_t*>(hidden), T, rms_eps, logits, V);
    return launch_status();
}

nvfp4_status lm_head_gemv(const nvfp4_matrix* w, const void* hidden, int32_t T, float rms_eps,
                          float* logits, cudaStream_t stream) {
    if (!w || !hidden || !logits || T < 1) return NVFP4_ERR_INVALID_ARG;
    if (!w->codes || !w->scales || !w->global_scale || w->n < 16 || w->k < 16)
        return NVFP4_ERR_INVALID_ARG;
    if (w->n % 16 || w->k % 16 || w->k > (1 << 20)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w->codes, 16) || !aligned(w->scales, 16) || !aligned(hidden, 16) || !aligned(logits, 4))
        return NVFP4_ERR_MISALIGNED;
    if (w->k % 64) return lm_head_generic(w, hidden, T, rms_eps, logits, stream);
    const int H = static_cast<int>(w->k);
    LmArgs la{};
    la.codes = w->codes;
    la.scales = w->scales;
    la.global = w->global_scale;
    la.V = w->n;
    la.H = H;
    la.ld = w->n;
    la.rms_eps = rms_eps;
    // two CTAs per SM (24 decoding warps) when half of the SM's shared
    // memory (less the static part and the per-CTA reserve) still holds three
    // stages besides the token rows, else one
    const int bbytes = 2 * std::min(T, kLmMaxT) * H * 2;  // f16 B rows + normalised bf16 rows
    const int stage = 9 * H;
    const int lim1 = dyn_smem_limit(k_lm_head);
    const int lim2 = std::min(lim1, smem_optin() / 2 - kLmStaticSmem - 1024);
    const bool two = lim2 - bbytes >= 3 * stage;
    const int lim = two ? lim2 : lim1;
    la.ring_bytes = std::min(kMaxStages * stage, ((lim - bbytes) / 128) * 128);
    if (la.ring_bytes < 2 * stage) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    la.groups = std::min(kMaxStages, la.ring_bytes / stage);
    const int smem = la.ring_bytes + bbytes;
    const int64_t tiles = w->n / 16;
    const int grid = static_cast<int>(std::min<int64_t>((two ? 2 : 1) * num_sms(), tiles));
    for (int t0 = 0; t0 < T; t0 += kLmMaxT) {
        la.T = std::min(kLmMaxT, T - t0);
        la.hidden = static_cast<const uint16_t*>(hidden) + (size_t)t0 * H;
        la.logits = logits + (size_t)t0 * w->n;
        const nvfp4_status st = launch_pdl(k_lm_head, grid, kThreads, smem, stream, la);
        if (st != NVFP4_OK) return st;
    }
    return NVFP4_OK;
}

}  // extern "C"

// ------------------------------------------------------------ grouped path (T > 4)
namespace {

struct GroupedWsOffsets {
    size_t offsets, tiles, perm, inv, xq, gx, act, amax, act_sh, amax_sh, aq, ga, aq_sh, gsh, ypart, ysh;
    // tensor-core path (W4A4): 128-position chunk prefix, NVFP4 B rows
    // (codes, then scales with a 16-byte pitch) in token and position order
    size_t chunks, tq_c, tq_s, xp_c, xp_s, gxp, aq_c, aq_s, as_c, as_s;
    size_t total;
};
inline int spitch16(int K) { return ((K / 16) + 15) & ~15; }

GroupedWsOffsets grouped_ws(int T, int k, int E, int H, int I, int S) {
    GroupedWsOffsets o{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    const size_t P = (size_t)T * k;
    o.offsets = take(4 * (size_t)(E + 1));
    o.tiles = take(4 * (size_t)(E + 1));
    o.perm = take(4 * P);
    o.inv = take(4 * P);
    o.amax = take(4 * P);
    o.amax_sh = take(4 * (size_t)T);
    o.xq = take(2 * (size_t)T * H);
    o.gx = take(4 * (size_t)T);
    o.act = take(2 * P * I);
    o.act_sh = take(2 * (size_t)T * S);
    o.aq = take(2 * P * I);
    o.ga = take(4 * P);
    o.aq_sh = take(2 * (size_t)T * S);
    o.gsh = take(4 * (size_t)T);
    o.ypart = take(4 * P * H);
    o.ysh = take(4 * (size_t)T * H);
    o.chunks = take(4 * (size_t)(E + 1));
    o.tq_c = take((size_t)T * H / 2);
    o.tq_s = take((size_t)T * spitch16(H));
    o.xp_c = take(P * H / 2);
    o.xp_s = take(P * spitch16(H));
    o.gxp = take(4 * P);
    o.aq_c = take(P * I / 2);
    o.aq_s = take(P * spitch16(I));
    o.as_c = take((size_t)T * S / 2);
    o.as_s = take((size_t)T * spitch16(S));
    o.total = off;
    return o;
}

size_t grouped_ws_total(int T, int k, int E, int H, int I, int S) { return grouped_ws(T, k, E, H, I, S).total; }

template <typename Kernel>
nvfp4_status launch_plain(Kernel kernel, int grid, int block, size_t smem, cudaStream_t stream,
                          const GroupedArgs& ga) {
    kernel<<<grid, block, smem, stream>>>(ga);
    return launch_status();
}

// cuTensorMapEncodeTiled from the driver (no link-time dependency on libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A row-major matrix of `rows` rows of `row_bytes` bytes as a 2-D byte
// tensor, boxes of {box_bytes, box_rows}.
bool byte_map(CUtensorMap* m, const void* base, int64_t row_bytes, int64_t rows, int box_bytes, int box_rows,
              CUtensorMapSwizzle swz) {
    const EncodeTiledFn enc = encode_tiled();
    if (!enc || !aligned(base, 16) || row_bytes % 16 || rows < 1) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows][K/2] NVFP4 code matrix as a 2-D byte tensor; a box
// {128 bytes, box_rows} with the 128-byte swizzle lands in the K-major
// swizzled layout tcgen05.mma reads (256 k per box).
bool code_map(CUtensorMap* m, const void* codes, int64_t rows, int K, int box_rows) {
    const EncodeTiledFn enc = encode_tiled();
    if (!enc || !aligned(codes, 16) || (K % 64) != 0 || rows < 1) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool seg_maps(TcArgs& ta, int s, const void* a_codes, int64_t a_rows, const void* b_codes, int64_t b_rows, int K) {
    if (!code_map(&ta.a_map[s], a_codes, a_rows, K, kTcRows)) return false;
    for (int g = 0; g < 4; ++g)
        if (!code_map(&ta.b_map[s][g], b_codes, b_rows, K, 32 * (g + 1))) return false;
    return true;
}

// Stage-ring bytes of k_grouped_tc: the shared memory the two scale blocks leave.
int tc_ring_cap() {
    const int lim = std::min(dyn_smem_limit(k_grouped_tc<kGroupedUp>), dyn_smem_limit(k_grouped_tc<kGroupedDown>));
    return ((lim - kTcOffRing - kTcSmemSlack) / 1024) * 1024;
}

// W4A4 grouped path on the tensor cores (tcgen05 kind::mxf4nvf4).
bool tc_path_ok(const moe_layer_weights* w) {
    const int H = w->hidden, I = w->inter, S = w->shared_inter;
    if (H % 64 || I % 64 || S % 64 || w->num_experts > kTcMaxExperts) return false;
    const void* p[] = {w->up_codes, w->down_codes, w->shared_up.codes, w->shared_down.codes};
    for (const void* q : p)
        if (!aligned(q, 16)) return false;
    const void* sc[] = {w->up_scales, w->down_scales, w->shared_up.scales, w->shared_down.scales};
    for (const void* q : sc)
        if (!aligned(q, 16)) return false;
    // one item's weight scales (128 rows x K/16 bytes) plus slack fit a block
    for (int K : {H, I, S})
        if (kTcRows * (K / 16) + 16 > kTcScBlk) return false;
    return encode_tiled() != nullptr && tc_ring_cap() >= 2 * tc_stage_bytes(4);
}

nvfp4_status grouped_forward_tc(const moe_layer_weights* w, const void* hidden, const int32_t* topk_idx,
                                const float* topk_w, int T, int k, float rms_eps, const void* residual, void* out,
                                uint8_t* ws, cudaStream_t stream) {
    const int E = w->num_experts, H = w->hidden, I = w->inter, S = w->shared_inter;
    const int P = T * k;
    const GroupedWsOffsets o = grouped_ws(T, k, E, H, I, S);
    auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    auto b16 = [&](size_t off) { return reinterpret_cast<uint16_t*>(ws + off); };
    auto u32 = [&](size_t off) { return reinterpret_cast<unsigned int*>(ws + off); };
    auto u8 = [&](size_t off) { return ws + off; };

    k_permute<<<1, kPermThreads, 0, stream>>>(topk_idx, P, E, i32(o.offsets), nullptr, i32(o.chunks), i32(o.perm),
                                              i32(o.inv));
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    if (cudaMemsetAsync(ws + o.amax, 0, o.xq - o.amax, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    // a1: token rows -> NVFP4 B rows, in token order and once per (token, choice) in position order
    k_quant_rows_tc<<<T, kGThreads, (size_t)H * 2, stream>>>(static_cast<const uint16_t*>(hidden), H, T, rms_eps,
                                                             nullptr, u8(o.tq_c), u8(o.tq_s), spitch16(H), f32(o.gx),
                                                             i32(o.inv), k, u8(o.xp_c), u8(o.xp_s), f32(o.gxp));
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;

    const int grid = num_sms();
    // a3 + a5 (up): routed experts over their positions, the shared expert over all tokens
    TcArgs ta{};
    ta.nseg = 2;
    TcSeg& ru = ta.seg[0];
    ru.nexp = E;
    ru.M = I;
    ru.K = H;
    ru.offsets = i32(o.offsets);
    ru.chunks = i32(o.chunks);
    ru.a_scales = w->up_scales;
    ru.a_global = w->up_global;
    ru.b_scales = u8(o.xp_s);
    ru.b_spitch = spitch16(H);
    ru.b_rows = P;
    ru.b_global = f32(o.gxp);
    ru.act = b16(o.act);
    ru.amax = u32(o.amax);
    TcSeg& su = ta.seg[1];
    su.nexp = 1;
    su.M = S;
    su.K = H;
    su.npos = T;
    su.a_scales = w->shared_up.scales;
    su.a_global = w->shared_up.global_scale;
    su.b_scales = u8(o.tq_s);
    su.b_spitch = spitch16(H);
    su.b_rows = T;
    su.b_global = f32(o.gx);
    su.act = b16(o.act_sh);
    su.amax = u32(o.amax_sh);
    if (!seg_maps(ta, 0, w->up_codes, (int64_t)E * I, u8(o.xp_c), P, H) ||
        !seg_maps(ta, 1, w->shared_up.codes, S, u8(o.tq_c), T, H))
        return NVFP4_ERR_CUDA;
    ta.ring_cap = tc_ring_cap();
    k_grouped_tc<kGroupedUp><<<grid, kTcThreads, kTcSmemSlack + kTcOffRing + ta.ring_cap, stream>>>(ta);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    // a1 on the intermediate rows (row amax from the up epilogue)
    k_quant_rows_tc<<<P, kGThreads, (size_t)I * 2, stream>>>(b16(o.act), I, P, 0.0f, u32(o.amax), u8(o.aq_c),
                                                             u8(o.aq_s), spitch16(I), f32(o.ga), nullptr, 0, nullptr,
                                                             nullptr, nullptr);
    k_quant_rows_tc<<<T, kGThreads, (size_t)S * 2, stream>>>(b16(o.act_sh), S, T, 0.0f, u32(o.amax_sh),
                                                             u8(o.as_c), u8(o.as_s), spitch16(S), f32(o.gsh), nullptr,
                                                             0, nullptr, nullptr, nullptr);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    // a4 + a5 (down): gate-weighted rows per position, shared rows per token
    TcArgs td{};
    td.nseg = 2;
    TcSeg& rd = td.seg[0];
    rd.nexp = E;
    rd.M = H;
    rd.K = I;
    rd.offsets = i32(o.offsets);
    rd.chunks = i32(o.chunks);
    rd.a_scales = w->down_scales;
    rd.a_global = w->down_global;
    rd.b_scales = u8(o.aq_s);
    rd.b_spitch = spitch16(I);
    rd.b_rows = P;
    rd.b_global = f32(o.ga);
    rd.y = f32(o.ypart);
    rd.gate = topk_w;
    rd.perm = i32(o.perm);
    TcSeg& sd = td.seg[1];
    sd.nexp = 1;
    sd.M = H;
    sd.K = S;
    sd.npos = T;
    sd.a_scales = w->shared_down.scales;
    sd.a_global = w->shared_down.global_scale;
    sd.b_scales = u8(o.as_s);
    sd.b_spitch = spitch16(S);
    sd.b_rows = T;
    sd.b_global = f32(o.gsh);
    sd.y = f32(o.ysh);
    if (!seg_maps(td, 0, w->down_codes, (int64_t)E * H, u8(o.aq_c), P, I) ||
        !seg_maps(td, 1, w->shared_down.codes, H, u8(o.as_c), T, S))
        return NVFP4_ERR_CUDA;
    td.ring_cap = tc_ring_cap();
    k_grouped_tc<kGroupedDown><<<grid, kTcThreads, kTcSmemSlack + kTcOffRing + td.ring_cap, stream>>>(td);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    // a6: combine + residual
    const int n4 = T * (H / 4);
    const int cgrid = std::min((n4 + 255) / 256, num_sms() * 8);
    k_combine<<<cgrid, 256, 0, stream>>>(f32(o.ysh), f32(o.ypart), i32(o.inv), static_cast<const uint16_t*>(residual),
                                         static_cast<uint16_t*>(out), T, H, k);
    return launch_status();
}

nvfp4_status grouped_forward(const moe_layer_weights* w, const void* hidden, const int32_t* topk_idx,
                             const float* topk_w, int T, int k, bool w4a4, float rms_eps, const void* residual,
                             void* out, uint8_t* ws, cudaStream_t stream) {
    const int E = w->num_experts, H = w->hidden, I = w->inter, S = w->shared_inter;
    if (w4a4 && k <= kDecodeMaxK && tc_path_ok(w)) return grouped_forward_tc(w, hidden, topk_idx, topk_w, T, k, rms_eps, residual, out, ws,
                                                         stream);
    const int P = T * k;
    const GroupedWsOffsets o = grouped_ws(T, k, E, H, I, S);
    auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    auto h16 = [&](size_t off) { return reinterpret_cast<__half*>(ws + off); };
    auto b16 = [&](size_t off) { return reinterpret_cast<uint16_t*>(ws + off); };
    auto u32 = [&](size_t off) { return reinterpret_cast<unsigned int*>(ws + off); };

    // a7: pairs grouped by expert
    k_permute<<<1, kPermThreads, 0, stream>>>(topk_idx, P, E, i32(o.offsets), i32(o.tiles), nullptr, i32(o.perm),
                                              i32(o.inv));
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    // amax words start at zero (amax and amax_sh are adjacent)
    if (cudaMemsetAsync(ws + o.amax, 0, o.xq - o.amax, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    // a1: token rows (normalised when rms_eps > 0) -> B operand
    if (w4a4) k_prep_rows<true><<<T, kGThreads, (size_t)H * 2, stream>>>(
        static_cast<const uint16_t*>(hidden), H, T, rms_eps, nullptr, h16(o.xq), f32(o.gx));
    else k_prep_rows<false><<<T, kGThreads, (size_t)H * 2, stream>>>(
        static_cast<const uint16_t*>(hidden), H, T, rms_eps, nullptr, h16(o.xq), f32(o.gx));
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;

    const size_t gsmem = (size_t)kGStages * kGStageBytes;
    GroupedArgs ga{};
    ga.E = E;
    ga.T = T;
    ga.k = k;
    ga.offsets = i32(o.offsets);
    ga.tiles = i32(o.tiles);
    ga.perm = i32(o.perm);
    ga.topk_w = topk_w;
    // a3 + a5 (up): routed over the grouped token rows, shared over all tokens
    ga.codes = w->up_codes;
    ga.scales = w->up_scales;
    ga.global = w->up_global;
    ga.sh_codes = w->shared_up.codes;
    ga.sh_scales = w->shared_up.scales;
    ga.sh_global = w->shared_up.global_scale;
    ga.M = I;
    ga.K = H;
    ga.MS = S;
    ga.KS = H;
    ga.b_routed = h16(o.xq);
    ga.g_routed = f32(o.gx);
    ga.b_shared = h16(o.xq);
    ga.g_shared = f32(o.gx);
    ga.act = b16(o.act);
    ga.act_sh = b16(o.act_sh);
    ga.amax = u32(o.amax);
    ga.amax_sh = u32(o.amax_sh);
    const int ggrid = num_sms() * 2;
    nvfp4_status st;
    if (w4a4) {
        if (dyn_smem_limit(k_grouped<true, kGroupedUp>) < (int)gsmem) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        st = launch_plain(k_grouped<true, kGroupedUp>, ggrid, kGThreads, gsmem, stream, ga);
    } else {
        if (dyn_smem_limit(k_grouped<false, kGroupedUp>) < (int)gsmem) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        st = launch_plain(k_grouped<false, kGroupedUp>, ggrid, kGThreads, gsmem, stream, ga);
    }
    if (st != NVFP4_OK) return st;
    // a1 on the intermediate rows (row amax from the up epilogue)
    if (w4a4) {
        k_prep_rows<true><<<P, kGThreads, (size_t)I * 2, stream>>>(b16(o.act), I, P, 0.0f, u32(o.amax), h16(o.aq),
                                                                    f32(o.ga));
        k_prep_rows<true><<<T, kGThreads, (size_t)S * 2, stream>>>(b16(o.act_sh), S, T, 0.0f, u32(o.amax_sh),
                                                                    h16(o.aq_sh), f32(o.gsh));
    } else {
        k_prep_rows<false><<<P, kGThreads, (size_t)I * 2, stream>>>(b16(o.act), I, P, 0.0f, nullptr, h16(o.aq),
                                                                     f32(o.ga));
        k_prep_rows<false><<<T, kGThreads, (size_t)S * 2, stream>>>(b16(o.act_sh), S, T, 0.0f, nullptr,
                                                                     h16(o.aq_sh), f32(o.gsh));
    }
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    // a4 + a5 (down): gate-weighted partial rows per position, shared rows per token
    ga.codes = w->down_codes;
    ga.scales = w->down_scales;
    ga.global = w->down_global;
    ga.sh_codes = w->shared_down.codes;
    ga.sh_scales = w->shared_down.scales;
    ga.sh_global = w->shared_down.global_scale;
    ga.M = H;
    ga.K = I;
    ga.MS = H;
    ga.KS = S;
    ga.b_routed = h16(o.aq);
    ga.g_routed = f32(o.ga);
    ga.b_shared = h16(o.aq_sh);
    ga.g_shared = f32(o.gsh);
    ga.ypart = f32(o.ypart);
    ga.ysh = f32(o.ysh);
    if (w4a4) {
        if (dyn_smem_limit(k_grouped<true, kGroupedDown>) < (int)gsmem) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        st = launch_plain(k_grouped<true, kGroupedDown>, ggrid, kGThreads, gsmem, stream, ga);
    } else {
        if (dyn_smem_limit(k_grouped<false, kGroupedDown>) < (int)gsmem) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        st = launch_plain(k_grouped<false, kGroupedDown>, ggrid, kGThreads, gsmem, stream, ga);
    }
    if (st != NVFP4_OK) return st;
    // a6: combine + residual
    const int n4 = T * (H / 4);
    const int cgrid = std::min((n4 + 255) / 256, num_sms() * 8);
    k_combine<<<cgrid, 256, 0, stream>>>(f32(o.ysh), f32(o.ypart), i32(o.inv), static_cast<const uint16_t*>(residual),
                                         static_cast<uint16_t*>(out), T, H, k);
    return launch_status();
}

}  // namespace

extern "C" nvfp4_status moe_permute(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t* offsets,
                                    int32_t* perm, int32_t* inv, int32_t* tile_offsets, cudaStream_t stream) {
    if (!topk_idx || !offsets || !perm || !inv) return NVFP4_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || E < 1 || k > E) return NVFP4_ERR_INVALID_ARG;
    if (E > 256 || (int64_t)T * k > (int64_t)1 << 28) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    k_permute<<<1, kPermThreads, 0, stream>>>(topk_idx, T * k, E, offsets, tile_offsets, nullptr, perm, inv);
    return launch_status();
}

// ------------------------------------------------------------ fused layer
namespace {

struct LayerWsOffsets {
    size_t plan, xq, gx, act, act_sh, aq, ga, aq_sh, gsh, ypart, ysh, ecnt, tilecnt, total;
};

LayerWsOffsets layer_ws(int T, int k, int H, int I, int S) {
    LayerWsOffsets o{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    o.ecnt = take(sizeof(int) * (kDecodeMaxU + 1));
    o.tilecnt = take(sizeof(int) * (size_t)(H / 16));
    o.plan = take(sizeof(DecodePlan));
    o.xq = take((size_t)T * H * 2);
    o.gx = take((size_t)T * 4);
    o.act = take((size_t)T * k * I * 2);
    o.act_sh = take((size_t)T * S * 2);
    o.aq = take((size_t)T * k * I * 2);
    o.ga = take((size_t)T * k * 4);
    o.aq_sh = take((size_t)T * S * 2);
    o.gsh = take((size_t)T * 4);
    o.ypart = take((size_t)T * k * H * 4);
    o.ysh = take((size_t)T * H * 4);
    o.total = off;
    return o;
}

LayerWs layer_ws_ptrs(const LayerWsOffsets& o, uint8_t* base) {
    LayerWs w{};
    w.plan = reinterpret_cast<DecodePlan*>(base + o.plan);
    w.xq = reinterpret_cast<__half*>(base + o.xq);
    w.gx = reinterpret_cast<float*>(base + o.gx);
    w.act = reinterpret_cast<uint16_t*>(base + o.act);
    w.act_sh = reinterpret_cast<uint16_t*>(base + o.act_sh);
    w.aq = reinterpret_cast<__half*>(base + o.aq);
    w.ga = reinterpret_cast<float*>(base + o.ga);
    w.aq_sh = reinterpret_cast<__half*>(base + o.aq_sh);
    w.gsh = reinterpret_cast<float*>(base + o.gsh);
    w.ypart = reinterpret_cast<float*>(base + o.ypart);
    w.ysh = reinterpret_cast<float*>(base + o.ysh);
    w.ecnt = reinterpret_cast<int*>(base + o.ecnt);
    w.tilecnt = reinterpret_cast<int*>(base + o.tilecnt);
    return w;
}

}  // namespace

extern "C" size_t moe_layer_forward_workspace_size(const moe_layer_weights* w, int32_t T, int32_t k,
                                                   nvfp4_act_mode mode) {
    (void)mode;
    if (!w || T < 1 || k < 1) return 0;
    return layer_ws(T, k, w->hidden, w->inter, w->shared_inter).total;
}

extern "C" nvfp4_status moe_layer_forward(const moe_layer_weights* w, const float* router_w, const float* bias,
                                          const void* hidden, int32_t T, int32_t k, nvfp4_act_mode mode,
                                          float rms_eps, const void* residual, void* out, int32_t* topk_idx,
                                          float* topk_w, void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream) {
    nvfp4_status st = check_layer(w);
    if (st != NVFP4_OK) return st;
    if (!router_w || !bias || !hidden || !out || !topk_idx || !topk_w || !workspace) return NVFP4_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || k > w->num_experts) return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_W4A16 && mode != NVFP4_W4A4) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(router_w, 16) || !aligned(out, 4) || !aligned(workspace, 256) ||
        (residual && !aligned(residual, 4)))
        return NVFP4_ERR_MISALIGNED;
    if (hidden == out && residual != hidden) return NVFP4_ERR_INVALID_ARG;
    if (T > kDecodeMaxT || k > kDecodeMaxK || k > 32 || w->num_experts > 256) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const int H = w->hidden, I = w->inter, S = w->shared_inter, E = w->num_experts;
    const LayerWsOffsets o = layer_ws(T, k, H, I, S);
    if (workspace_bytes < o.total) return NVFP4_ERR_WORKSPACE;
    const LayerWs ws = layer_ws_ptrs(o, static_cast<uint8_t*>(workspace));
    const bool w4a4 = mode == NVFP4_W4A4;

    {  // route + plan + up-B rows (one cluster)
        constexpr int TT = 8;
        const int lim = dyn_smem_limit(k_route<TT>);
        const int hbytes = TT * H * 2;
        const int nj = (E + kRouteCluster - 1) / kRouteCluster;
        const int stage_w = hbytes + nj * H * 4 <= lim ? 1 : 0;
        const int smem = hbytes + (stage_w ? nj * H * 4 : 0);
        if (smem > lim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        st = launch_pdl(k_route<TT>, kRouteCluster, kRouteWarps * 32, smem, stream,
                        static_cast<const uint16_t*>(hidden), router_w, bias, T, H, E, k, rms_eps, stage_w, topk_idx,
                        topk_w, ws.plan, ws.xq, ws.gx, w4a4 ? 1 : 0);
        if (st != NVFP4_OK) return st;
    }
    const int grid = std::max(num_sms(), 2 * (T * k + (S + I - 1) / I) + 4);
    {
        LayerUpArgs ua{};
        ua.codes = w->up_codes;
        ua.scales = w->up_scales;
        ua.global = w->up_global;
        ua.sh_codes = w->shared_up.codes;
        ua.sh_scales = w->shared_up.scales;
        ua.sh_global = w->shared_up.global_scale;
        ua.E = E;
        ua.H = H;
        ua.I = I;
        ua.S = S;
        ua.T = T;
        ua.k = k;
        ua.ws = ws;
        const int lim = w4a4 ? dyn_smem_limit(k_layer_up<true>) : dyn_smem_limit(k_layer_up<false>);
        const int bbytes = T * H * 2;
        const int stage = 9 * H;
        ua.ring_bytes = std::min(kMaxStages * stage, ((lim - bbytes) / 128) * 128);
        if (ua.ring_bytes < 2 * stage) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        const int smem = ua.ring_bytes + bbytes;
        st = w4a4 ? launch_pdl(k_layer_up<true>, grid, kThreads, smem, stream, ua)
                  : launch_pdl(k_layer_up<false>, grid, kThreads, smem, stream, ua);
        if (st != NVFP4_OK) return st;
    }
    {
        LayerDownArgs da{};
        da.codes = w->down_codes;
        da.scales = w->down_scales;
        da.global = w->down_global;
        da.sh_codes = w->shared_down.codes;
        da.sh_scales = w->shared_down.scales;
        da.sh_global = w->shared_down.global_scale;
        da.E = E;
        da.H = H;
        da.I = I;
        da.S = S;
        da.T = T;
        da.k = k;
        da.ws = ws;
        da.residual = static_cast<const uint16_t*>(residual);
        da.out = static_cast<uint16_t*>(out);
        const int lim = w4a4 ? dyn_smem_limit(k_layer_down<true>) : dyn_smem_limit(k_layer_down<false>);
        const int bbytes = (2 * T * I + T * S) * 2;
        const int stage = 9 * std::max(I, S);
        da.ring_bytes = std::min(kMaxStages * stage, ((lim - bbytes) / 128) * 128);
        if (da.ring_bytes < 2 * stage) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        const int smem = da.ring_bytes + bbytes;
        st = w4a4 ? launch_pdl(k_layer_down<true>, grid, kThreads, smem, stream, da)
                  : launch_pdl(k_layer_down<false>, grid, kThreads, smem, stream, da);
    }
    return st;
}

// ------------------------------------------------ allocation-free variant
// moe_expert_forward_noalloc: the same computation as moe_expert_forward for
// callers that cannot allocate device memory. Its scratch is this file-scope
// device array; the library holds it on every GPU that loads it until the
// process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NVFP4MOE_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch in the current context. In host code
// the symbol is only a host-side handle; its device address is looked up with
// cudaGetSymbolAddress once per (device, context) and cached under that
// context's id, so that a context made later (after cudaDeviceReset, or with
// cuCtxCreate) gets its own lookup. Without a context id every call looks it
// up again.
void* noalloc_scratch(nvfp4_status* st) {
    struct Entry {
        unsigned long long ctx;
        int dev;
        void* p;
    };
    static Entry table[64];
    static int used = 0;
    static std::mutex mu;
    const int d = current_device();
    // 0 before the runtime has made a context current (the lookup below does)
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (ctx != 0)
        for (int i = 0; i < used; ++i)
            if (table[i].ctx == ctx && table[i].dev == d) return table[i].p;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        *st = NVFP4_ERR_CUDA;
        return nullptr;
    }
    if (ctx != 0) {
        if (used < 64) table[used++] = Entry{ctx, d, p};
        else table[ctx % 64] = Entry{ctx, d, p};
    }
    return p;
}

}  // namespace

extern "C" nvfp4_status moe_expert_forward_noalloc(const moe_layer_weights* w, const void* hidden,
                                                   const int32_t* topk_idx, const float* topk_w,
                                                   int32_t T, int32_t k, nvfp4_act_mode mode,
                                                   float rms_eps, const void* residual, void* out,
                                                   cudaStream_t stream) {
    // the same argument checks as moe_expert_forward, before the size is derived from them
    nvfp4_status cs = check_layer(w);
    if (cs != NVFP4_OK) return cs;
    if (!hidden || !topk_idx || !topk_w || !out || T < 1 || k < 1 || k > w->num_experts)
        return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_W4A16 && mode != NVFP4_W4A4) return NVFP4_ERR_INVALID_ARG;
    const size_t need = moe_expert_forward_workspace_size(w, T, k, mode);
    if (need == 0) return NVFP4_ERR_INVALID_ARG;
    if (need > NVFP4MOE_NOALLOC_SCRATCH_BYTES) return NVFP4_ERR_WORKSPACE;  // beyond the fixed scratch
    nvfp4_status st = NVFP4_OK;
    void* scratch = noalloc_scratch(&st);
    if (scratch == nullptr) return st;
    // the previous call's contents remain: clear the region (its counters must start at zero)
    if (cudaMemsetAsync(scratch, 0, need, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    return moe_expert_forward(w, hidden, topk_idx, topk_w, T, k, mode, rms_eps, residual, out, scratch,
                              need, stream);
}

// ------------------------------------------------ column-block copy
namespace {

// One warp per (matrix, 16-column block, 32-row pair): lane L = 4g + q writes
// its 8 code bytes, lanes 0..7 the 4 scale bytes of group g = L (the layout
// in the header).
__global__ void k_colblock_layout(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                  int64_t pairs_total, int rows, int cols, uint8_t* __restrict__ out) {
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= pairs_total) return;
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int P = rows >> 5, C = cols >> 4;
    const int p = static_cast<int>(w % P);
    const int64_t bc = w / P;  // matrix * C + block
    const int c = static_cast<int>(bc % C);
    const int64_t mat = bc / C;
    const uint8_t* mc = codes + mat * rows * (int64_t)(cols >> 1);
    const uint8_t* ms = scales + mat * rows * (int64_t)C;
    uint8_t* blk = out + bc * 9 * (int64_t)rows;
    uint8_t v[8];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 32 * p + 16 * mt + g + 8 * (i >> 1);
            v[4 * mt + i] = mc[(int64_t)row * (cols >> 1) + 8 * c + 2 * q + (i & 1)];
        }
    uint2 o;
    o.x = v[0] | (v[1] << 8) | (v[2] << 16) | ((uint32_t)v[3] << 24);
    o.y = v[4] | (v[5] << 8) | (v[6] << 16) | ((uint32_t)v[7] << 24);
    *reinterpret_cast<uint2*>(blk + (int64_t)p * 256 + lane * 8) = o;
    if (lane < 8) {
        uint32_t s = 0;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                s |= (uint32_t)ms[(int64_t)(32 * p + 16 * mt + lane + 8 * j) * C + c] << (8 * (2 * mt + j));
        *reinterpret_cast<uint32_t*>(blk + 8 * (int64_t)rows + (int64_t)p * 32 + lane * 4) = s;
    }
}

}  // namespace

extern "C" nvfp4_status nvfp4_colblock_layout(const uint8_t* codes, const uint8_t* scales, int64_t batch,
                                              int64_t rows, int64_t cols, uint8_t* out, cudaStream_t stream) {
    if (!codes || !scales || !out || batch < 1 || rows < 1 || cols < 1) return NVFP4_ERR_INVALID_ARG;
    if (rows % 32 || cols % 16 || rows > (1 << 24) || cols > (1 << 24)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16)) return NVFP4_ERR_MISALIGNED;
    const int64_t pairs = batch * (cols / 16) * (rows / 32);
    const int wpb = 8;  // warps per block
    k_colblock_layout<<<(unsigned)((pairs + wpb - 1) / wpb), 32 * wpb, 0, stream>>>(
        codes, scales, pairs, static_cast<int>(rows), static_cast<int>(cols), out);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}

// ------------------------------------------------ persistent layer stack
namespace {

struct StackWsOffsets {
    size_t cnt, z, hx, amx, part, total;
};

// G: the grid (one CTA per SM), whose partials of each layer output meet in
// the workspace.
StackWsOffsets stack_ws(int L, int T, int k, int E, int H, int G) {
    StackWsOffsets o{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    o.cnt = take(sizeof(int) * kCtlWords);  // exit count, abort flag, epoch
    o.amx = take(sizeof(unsigned long long) * (size_t)G * T);
    o.z = take(sizeof(unsigned long long) * (size_t)L * T * E);
    o.hx = take(sizeof(unsigned int) * (size_t)T * H);
    o.part = take(sizeof(unsigned long long) * (size_t)G * T * H);
    o.total = off;
    return o;
}

// Units (16 intermediate rows of one expert) a CTA holds in one layer at
// most, under the kernel's split (stack_units): the shared expert's S/16 over
// cs CTAs, each routed expert's I/16 over at least (G - cs) / Umax CTAs,
// Umax = min(T k, E); 0 if some expert would get no CTA (G <= Umax).
int stack_max_units(int T, int k, int E, int I, int S, int G) {
    const int Umax = std::min(T * k, E), RS = S / 16, RI = I / 16;
    if (G <= Umax) return 0;
    const int cs = stack_shared_ctas(G, RS, RI, Umax);
    const int per_routed = (G - cs) / Umax;
    if (per_routed < 1) return 0;
    return std::max((RS + cs - 1) / cs, (RI + per_routed - 1) / per_routed);
}

// Dynamic shared memory of the stack kernel: the ring, then the router rows,
// the operand union (layer input and up B operand; later the layer output
// partial), the top-k scores, the units' intermediate values and down B
// operands.
struct StackSmem {
    int ring_cap, off_gate, off_uni, off_tk, off_uact, off_ubq, total;
};

// The staging ring takes whatever the rest leaves, and must hold at least two
// items (9 H bytes each).
bool stack_smem(int lim, int E, int G, int T, int H, int units, StackSmem* out) {
    auto a128 = [](size_t x) { return static_cast<int>((x + 127) & ~size_t(127)); };
    const int item = 9 * H;
    const int ng = (E + G - 1) / G;
    const int gate = a128((size_t)ng * H * 4);
    const int uni = a128((size_t)T * H * 4);
    const int tk = a128((size_t)T * E * 8);
    const int ua = a128((size_t)units * T * kUnitRows * 2);
    const int rest = gate + uni + tk + 2 * ua;
    const int ring = ((lim - rest) / 128) * 128;
    if (ring < 2 * item) return false;
    out->ring_cap = ring;
    out->off_gate = ring;
    out->off_uni = out->off_gate + gate;
    out->off_tk = out->off_uni + uni;
    out->off_uact = out->off_tk + tk;
    out->off_ubq = out->off_uact + ua;
    out->total = out->off_ubq + ua;
    return true;
}

nvfp4_status check_stack(const moe_stack_layer* layers, int32_t L, int32_t T, int32_t k) {
    if (!layers || L < 1 || T < 1 || k < 1) return NVFP4_ERR_INVALID_ARG;
    if (L > NVFP4MOE_STACK_MAX_LAYERS || L > kStackMaxLayers) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const moe_layer_weights& w0 = layers[0].moe;
    for (int l = 0; l < L; ++l) {
        const moe_stack_layer& ly = layers[l];
        const nvfp4_status st = check_layer(&ly.moe);
        if (st != NVFP4_OK) return st;
        if (ly.moe.num_experts != w0.num_experts || ly.moe.hidden != w0.hidden || ly.moe.inter != w0.inter ||
            ly.moe.shared_inter != w0.shared_inter)
            return NVFP4_ERR_INVALID_ARG;
        if (!ly.router_w || !ly.router_bias || !ly.down_colblock || !ly.shared_down_colblock)
            return NVFP4_ERR_INVALID_ARG;
        if (!aligned(ly.router_w, 16) || !aligned(ly.router_bias, 16) || !aligned(ly.moe.up_global, 16) ||
            !aligned(ly.moe.down_global, 16) || !aligned(ly.down_colblock, 16) ||
            !aligned(ly.shared_down_colblock, 16))
            return NVFP4_ERR_MISALIGNED;
    }
    if (k > w0.num_experts) return NVFP4_ERR_INVALID_ARG;
    if (T > kDecodeMaxT || k > kDecodeMaxK || w0.num_experts > 256 || w0.num_experts % 8) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    // the down step's warps hold at most kDownMaxPairs 32-row pairs each
    if (w0.hidden > 32 * kDownMaxPairs * kConsumerWarps) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const int mu = stack_max_units(T, k, w0.num_experts, w0.inter, w0.shared_inter, num_sms());
    if (mu < 1 || mu > kMaxUnits) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    return NVFP4_OK;
}

}  // namespace

extern "C" size_t moe_stack_forward_workspace_size(const moe_stack_layer* layers, int32_t L, int32_t T, int32_t k,
                                                   nvfp4_act_mode mode) {
    (void)mode;
    if (check_stack(layers, L, T, k) != NVFP4_OK) return 0;
    const moe_layer_weights& w = layers[0].moe;
    return stack_ws(L, T, k, w.num_experts, w.hidden, num_sms()).total;
}

extern "C" nvfp4_status moe_stack_forward(const moe_stack_layer* layers, int32_t L, const void* hidden_in, int32_t T,
                                          int32_t k, nvfp4_act_mode mode, float rms_eps, void* hidden_out,
                                          int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream) {
    nvfp4_status st = check_stack(layers, L, T, k);
    if (st != NVFP4_OK) return st;
    if (!hidden_in || !hidden_out || !topk_idx || !topk_w || !workspace) return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_W4A16 && mode != NVFP4_W4A4) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(hidden_in, 16) || !aligned(hidden_out, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
        !aligned(workspace, 256))
        return NVFP4_ERR_MISALIGNED;
    const moe_layer_weights& w0 = layers[0].moe;
    const int E = w0.num_experts, H = w0.hidden, I = w0.inter, S = w0.shared_inter;
    {  // hidden_out must not overlap hidden_in
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(hidden_in), a1 = a0 + (size_t)T * H * 2;
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(hidden_out), b1 = b0 + (size_t)L * T * H * 2;
        if (a0 < b1 && b0 < a1) return NVFP4_ERR_INVALID_ARG;
    }
    const int G = num_sms();
    const StackWsOffsets o = stack_ws(L, T, k, E, H, G);
    if (workspace_bytes < o.total) return NVFP4_ERR_WORKSPACE;
    const bool w4a4 = mode == NVFP4_W4A4;
    const void* kfn = w4a4 ? reinterpret_cast<const void*>(k_moe_stack<true>)
                           : reinterpret_cast<const void*>(k_moe_stack<false>);
    const int lim = dyn_smem_limit(kfn);
    StackSmem sm{};
    if (lim <= 0 || !stack_smem(lim, E, G, T, H, stack_max_units(T, k, E, I, S, G), &sm))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, kThreads, sm.total) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (per_sm < 1) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // one CTA per SM must fit for the cooperative grid

    StackArgs a{};
    for (int l = 0; l < L; ++l) {
        const moe_stack_layer& ly = layers[l];
        StackLayer& d = a.layer[l];
        d.up_codes = ly.moe.up_codes;
        d.up_scales = ly.moe.up_scales;
        d.up_global = ly.moe.up_global;
        d.down_cb = ly.down_colblock;
        d.down_global = ly.moe.down_global;
        d.shu_codes = ly.moe.shared_up.codes;
        d.shu_scales = ly.moe.shared_up.scales;
        d.shu_global = ly.moe.shared_up.global_scale;
        d.shd_cb = ly.shared_down_colblock;
        d.shd_global = ly.moe.shared_down.global_scale;
        d.router_w = ly.router_w;
        d.router_b = ly.router_bias;
    }
    a.L = L;
    a.E = E;
    a.H = H;
    a.I = I;
    a.S = S;
    a.T = T;
    a.k = k;
    a.rms_eps = rms_eps;
    a.hidden_in = static_cast<const uint16_t*>(hidden_in);
    a.hidden_out = static_cast<uint16_t*>(hidden_out);
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    a.ws.cnt = reinterpret_cast<int*>(base + o.cnt);
    a.ws.zt = reinterpret_cast<unsigned long long*>(base + o.z);
    a.ws.hx = reinterpret_cast<unsigned int*>(base + o.hx);
    a.ws.amx = reinterpret_cast<unsigned long long*>(base + o.amx);
    a.ws.part = reinterpret_cast<unsigned long long*>(base + o.part);
    a.ring_cap = sm.ring_cap;
    a.off_gate = sm.off_gate;
    a.off_uni = sm.off_uni;
    a.off_tk = sm.off_tk;
    a.off_uact = sm.off_uact;
    a.off_ubq = sm.off_ubq;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sm.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = w4a4 ? cudaLaunchKernelEx(&cfg, k_moe_stack<true>, a)
                               : cudaLaunchKernelEx(&cfg, k_moe_stack<false>, a);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    return launch_status();
}

// ------------------------------------------------ lm_head with a workspace
// Up to kLmMaxT tokens the GEMV kernel; above, the grouped GEMM kernel as one
// dense group (all tokens, 64-token tiles, each weight tile read once per
// 64 tokens and shared through L2 by the CTAs of one row tile).
namespace {

struct LmWsOffsets {
    size_t zero, xq, gx, total;
};

LmWsOffsets lm_ws(int T, int H) {
    LmWsOffsets o{};
    size_t off = 0;
    o.zero = off;
    off += 256;
    o.xq = off;  // rows padded to a multiple of 16: the tensor-core GEMM reads whole 16-row groups
    off += align256((size_t)((T + 15) & ~15) * H * 2);
    o.gx = off;  // per token: the W4A16 row prescale (1 unless the row's amax reaches 2^15)
    off += align256((size_t)T * 4);
    o.total = off;
    return o;
}

}  // namespace

extern "C" size_t lm_head_forward_workspace_size(const nvfp4_matrix* w, int32_t T) {
    if (!w || T < 1 || w->k < 16) return 0;
    if (T <= kLmMaxT || w->k % 64) return 256;
    return lm_ws(T, static_cast<int>(w->k)).total;
}

extern "C" nvfp4_status lm_head_forward(const nvfp4_matrix* w, const void* hidden, int32_t T, float rms_eps,
                                        float* logits, void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
    if (!w || !hidden || !logits || T < 1) return NVFP4_ERR_INVALID_ARG;
    if (T <= kLmMaxT || (w->k % 64 && w->k % 16 == 0)) return lm_head_gemv(w, hidden, T, rms_eps, logits, stream);
    if (!workspace) return NVFP4_ERR_INVALID_ARG;
    if (!w->codes || !w->scales || !w->global_scale || w->n < 64 || w->k < 64) return NVFP4_ERR_INVALID_ARG;
    if (w->n % 64 || w->k % 64 || w->k > (1 << 20) || w->n > (1 << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w->codes, 16) || !aligned(w->scales, 16) || !aligned(hidden, 16) || !aligned(logits, 16) ||
        !aligned(workspace, 256))
        return NVFP4_ERR_MISALIGNED;
    const int H = static_cast<int>(w->k);
    const LmWsOffsets o = lm_ws(T, H);
    if (workspace_bytes < o.total) return NVFP4_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // no routed group: its tile count reads as 0
    if (cudaMemsetAsync(ws + o.zero, 0, 4, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    __half* xq = reinterpret_cast<__half*>(ws + o.xq);
    float* gx = reinterpret_cast<float*>(ws + o.gx);
    k_prep_rows<false><<<T, kGThreads, (size_t)H * 2, stream>>>(static_cast<const uint16_t*>(hidden), H, T, rms_eps,
                                                                 nullptr, xq, gx);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    // the tensor-core GEMM (tcgen05 kind::f16), up to 256 tokens per launch
    if (w->n % kLmTcRows == 0 && encode_tiled() != nullptr) {
        const int lim = dyn_smem_limit(k_lm_head_tc);
        const int V = static_cast<int>(w->n);
        bool ok = lim >= 1024 + kLmTcStages * lm_tc_stage_bytes(kLmTcMaxN);
        LmTcArgs la{};
        ok = ok && byte_map(&la.a_map, w->codes, H / 2, V, 32, kLmTcRows, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (ok) {
            la.scales = w->scales;
            la.global = w->global_scale;
            la.ld = V;
            la.V = V;
            la.H = H;
            for (int t0 = 0; t0 < T; t0 += kLmTcMaxN) {
                const int n = std::min(kLmTcMaxN, T - t0);
                la.T = n;
                la.N = (n + 15) & ~15;
                la.gx = gx + t0;
                la.logits = logits + (int64_t)t0 * V;
                // rows n .. N - 1 (padding) feed only the MMA columns that are not stored
                if (!byte_map(&la.b_map, xq + (size_t)t0 * H, 2 * H, la.N, 128, la.N, CU_TENSOR_MAP_SWIZZLE_128B))
                    return NVFP4_ERR_CUDA;
                const size_t smem = 1024 + (size_t)kLmTcStages * lm_tc_stage_bytes(la.N);
                k_lm_head_tc<<<std::min(num_sms(), V / kLmTcRows), kLmTcThreads, smem, stream>>>(la);
                if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
            }
            return NVFP4_OK;
        }
    }
    GroupedArgs ga{};
    ga.E = 0;
    ga.M = 0;
    ga.K = H;
    ga.tiles = reinterpret_cast<const int32_t*>(ws + o.zero);
    ga.sh_codes = w->codes;
    ga.sh_scales = w->scales;
    ga.sh_global = w->global_scale;
    ga.MS = static_cast<int>(w->n);
    ga.KS = H;
    ga.T = T;
    ga.k = 1;
    ga.b_shared = xq;
    ga.g_shared = gx;
    ga.ysh = logits;
    const size_t gsmem = (size_t)kGStages * kGStageBytes;
    if (dyn_smem_limit(k_grouped<false, kGroupedDown>) < (int)gsmem) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    k_grouped<false, kGroupedDown><<<num_sms() * 2, kGThreads, gsmem, stream>>>(ga);
    return launch_status();
}

// ------------------------------------------------ FP4 tensor-pipe peak
extern "C" nvfp4_status nvfp4_fp4_mma_peak(int32_t n, int32_t chains, int32_t iters, double* tflops,
                                           cudaStream_t stream) {
    if (!tflops || n < 32 || n > 256 || n % 32 || chains < 1 || chains * n > 448 || iters < 1)
        return NVFP4_ERR_INVALID_ARG;
    const size_t smem = 1024 + kPeakSmemA + kPeakSmemB;
    if (dyn_smem_limit(k_fp4_peak) < static_cast<int>(smem)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const int grid = num_sms();
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return NVFP4_ERR_CUDA;
    nvfp4_status st = NVFP4_OK;
    k_fp4_peak<<<grid, kPeakThreads, smem, stream>>>(n, chains, iters);  // warm-up
    cudaEventRecord(e0, stream);
    k_fp4_peak<<<grid, kPeakThreads, smem, stream>>>(n, chains, iters);
    cudaEventRecord(e1, stream);
    float ms = 0.0f;
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || ms <= 0.0f)
        st = NVFP4_ERR_CUDA;
    else
        *tflops = 2.0 * 128.0 * n * 64.0 * static_cast<double>(iters) * grid / (ms * 1e-3) / 1e12;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return st;
}

// ------------------------------------------------------------ workspace inspection
extern "C" nvfp4_status nvfp4_workspace_view(int32_t call, const moe_layer_weights* w, int32_t T, int32_t k,
                                             nvfp4_act_mode mode, int32_t region, nvfp4_ws_view* view) {
    nvfp4_status st = check_layer(w);
    if (st != NVFP4_OK) return st;
    if (!view || T < 1 || k < 1 || k > w->num_experts) return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_W4A16 && mode != NVFP4_W4A4) return NVFP4_ERR_INVALID_ARG;
    if (region < NVFP4_WS_X || region > NVFP4_WS_SH_ACT_Q) return NVFP4_ERR_INVALID_ARG;
    const int E = w->num_experts, H = w->hidden, I = w->inter, S = w->shared_inter;
    const int64_t P = (int64_t)T * k;
    const bool w4a4 = mode == NVFP4_W4A4;
    nvfp4_ws_view v{};
    auto rows_of = [&](int r) -> int64_t { return (r == NVFP4_WS_X || r >= NVFP4_WS_SH_ACT) ? T : P; };
    auto cols_of = [&](int r) -> int64_t {
        return r == NVFP4_WS_X ? H : (r >= NVFP4_WS_SH_ACT ? S : I);
    };
    v.rows = rows_of(region);
    v.cols = cols_of(region);
    if (call == 1) {  // moe_layer_forward
        if (T > kDecodeMaxT || k > kDecodeMaxK || E > 256) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        const LayerWsOffsets o = layer_ws(T, k, H, I, S);
        const bool quantised = region == NVFP4_WS_X || region == NVFP4_WS_ACT_Q || region == NVFP4_WS_SH_ACT_Q;
        if (quantised && !w4a4) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // W4A16 rows are prescaled, not quantised
        switch (region) {
            case NVFP4_WS_X: v.offset = o.xq; v.global_offset = o.gx; break;
            case NVFP4_WS_ACT: v.offset = o.act; break;
            case NVFP4_WS_ACT_Q: v.offset = o.aq; v.global_offset = o.ga; break;
            case NVFP4_WS_SH_ACT: v.offset = o.act_sh; break;
            default: v.offset = o.aq_sh; v.global_offset = o.gsh; break;
        }
        v.format = quantised ? NVFP4_WS_F16_DEQUANT : NVFP4_WS_BF16;
        v.pitch = 2 * v.cols;
        v.has_global = quantised ? 1 : 0;
    } else if (call == 0) {  // moe_expert_forward
        if (decode_path(w, T, k)) {
            if (region != NVFP4_WS_ACT && region != NVFP4_WS_SH_ACT) return NVFP4_ERR_UNSUPPORTED_SHAPE;
            const DecodeWs o = decode_ws(T, k, H, I, S);
            v.offset = region == NVFP4_WS_ACT ? o.act : o.act_sh;
            v.format = NVFP4_WS_BF16;
            v.pitch = 2 * v.cols;
        } else {
            if (!(w4a4 && k <= kDecodeMaxK && tc_path_ok(w)) || E > 256) return NVFP4_ERR_UNSUPPORTED_SHAPE;
            const GroupedWsOffsets o = grouped_ws(T, k, E, H, I, S);
            switch (region) {
                case NVFP4_WS_X: v.offset = o.tq_c; v.scales_offset = o.tq_s; v.global_offset = o.gx; break;
                case NVFP4_WS_ACT: v.offset = o.act; break;
                case NVFP4_WS_ACT_Q: v.offset = o.aq_c; v.scales_offset = o.aq_s; v.global_offset = o.ga; break;
                case NVFP4_WS_SH_ACT: v.offset = o.act_sh; break;
                default: v.offset = o.as_c; v.scales_offset = o.as_s; v.global_offset = o.gsh; break;
            }
            const bool quantised = region == NVFP4_WS_X || region == NVFP4_WS_ACT_Q || region == NVFP4_WS_SH_ACT_Q;
            v.format = quantised ? NVFP4_WS_CODES : NVFP4_WS_BF16;
            v.pitch = quantised ? v.cols / 2 : 2 * v.cols;
            v.scales_pitch = quantised ? spitch16((int)v.cols) : 0;
            v.has_global = quantised ? 1 : 0;
            v.position_order = region == NVFP4_WS_ACT || region == NVFP4_WS_ACT_Q ? 1 : 0;
        }
    } else {
        return NVFP4_ERR_INVALID_ARG;
    }
    *view = v;
    return NVFP4_OK;
}

// ------------------------------------------------------------ FP8 shared expert
namespace {

struct Fp8WsOffsets {
    size_t act, total;
};

Fp8WsOffsets fp8_ws(int T, int H, int S) {
    (void)H;
    Fp8WsOffsets o{};
    const int tc = std::min(T, kF8MaxT);  // tokens per chunk
    o.act = 0;
    o.total = align256((size_t)tc * S * 2);
    return o;
}

nvfp4_status check_fp8_matrix(const fp8_matrix* m, int64_t n, int64_t k) {
    if (!m || !m->codes || !m->global_scale) return NVFP4_ERR_INVALID_ARG;
    if (m->n != n || m->k != k) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(m->codes, 16)) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status fp8_quantize(const void* x, int x_is_bf16, int64_t rows, int64_t cols,
                                     nvfp4_global_mode mode, float* global_scale, uint8_t* codes,
                                     cudaStream_t stream) {
    if (!global_scale || rows < 0 || cols <= 0) return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_GLOBAL_PER_TENSOR && mode != NVFP4_GLOBAL_PER_ROW && mode != NVFP4_GLOBAL_GIVEN)
        return NVFP4_ERR_INVALID_ARG;
    if (cols % 16) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) {
        if (mode == NVFP4_GLOBAL_PER_TENSOR && cudaMemsetAsync(global_scale, 0, sizeof(float), stream) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        return NVFP4_OK;
    }
    if (!x || !codes) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(codes, 16)) return NVFP4_ERR_MISALIGNED;
    const int64_t nblocks = rows * (cols / 16);
    const int maxg = num_sms() * 8;
    const int grid = static_cast<int>(std::min<int64_t>((nblocks + 255) / 256, maxg));
    const bool bf16 = x_is_bf16 != 0;
    if (mode == NVFP4_GLOBAL_PER_ROW) {
        const int rgrid = static_cast<int>(std::min<int64_t>((rows + 7) / 8, maxg));
        if (bf16) k_fp8_quantize_rows<true><<<rgrid, 256, 0, stream>>>(x, rows, cols, global_scale, codes);
        else k_fp8_quantize_rows<false><<<rgrid, 256, 0, stream>>>(x, rows, cols, global_scale, codes);
        return launch_status();
    }
    if (mode == NVFP4_GLOBAL_PER_TENSOR) {
        if (cudaMemsetAsync(global_scale, 0, sizeof(float), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
        unsigned int* bits = reinterpret_cast<unsigned int*>(global_scale);
        if (bf16) k_amax<true><<<grid, 256, 0, stream>>>(x, nblocks, bits);
        else k_amax<false><<<grid, 256, 0, stream>>>(x, nblocks, bits);
    }
    const int from_amax = mode == NVFP4_GLOBAL_PER_TENSOR ? 1 : 0;
    if (bf16) k_fp8_quantize_global<true><<<grid, 256, 0, stream>>>(x, nblocks, global_scale, from_amax, codes);
    else k_fp8_quantize_global<false><<<grid, 256, 0, stream>>>(x, nblocks, global_scale, from_amax, codes);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    if (from_amax) k_fp8_finalize_global<<<1, 1, 0, stream>>>(global_scale);
    return launch_status();
}

extern "C" size_t moe_shared_fp8_workspace_size(const fp8_matrix* up, int32_t T) {
    if (!up || T < 1) return 0;
    return fp8_ws(T, static_cast<int>(up->k), static_cast<int>(up->n)).total;
}

extern "C" nvfp4_status moe_shared_fp8_forward(const fp8_matrix* up, const fp8_matrix* down, const void* hidden,
                                               int32_t T, float rms_eps, const void* residual, void* out,
                                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!up || !down || !hidden || !out || !workspace || T < 1) return NVFP4_ERR_INVALID_ARG;
    const int64_t S = up->n, H = up->k;
    nvfp4_status st = check_fp8_matrix(up, S, H);
    if (st != NVFP4_OK) return st;
    if ((st = check_fp8_matrix(down, H, S)) != NVFP4_OK) return st;
    if (S < 1 || H < 1 || H % 64 || S % 64 || H > (1 << 20) || S > (1 << 20)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(hidden, 16) || !aligned(out, 4) || !aligned(workspace, 256) || (residual && !aligned(residual, 4)))
        return NVFP4_ERR_MISALIGNED;
    const Fp8WsOffsets o = fp8_ws(T, static_cast<int>(H), static_cast<int>(S));
    if (workspace_bytes < o.total) return NVFP4_ERR_WORKSPACE;
    const size_t smem_up = (size_t)kF8MaxT * H, smem_dn = (size_t)kF8MaxT * S;
    if ((int64_t)smem_up > dyn_smem_limit(k_fp8_gemv<kGroupedUp>) ||
        (int64_t)smem_dn > dyn_smem_limit(k_fp8_gemv<kGroupedDown>))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    uint16_t* act = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + o.act);
    for (int t0 = 0; t0 < T; t0 += kF8MaxT) {  // chunks of up to 8 tokens: the MMA's columns
        const int tc = std::min(kF8MaxT, T - t0);
        Fp8GemvArgs ua{};
        ua.w = up->codes;
        ua.gw = up->global_scale;
        ua.n = static_cast<int>(S);
        ua.K = static_cast<int>(H);
        ua.src = static_cast<const uint16_t*>(hidden) + (size_t)t0 * H;
        ua.rms_eps = rms_eps;
        ua.T = tc;
        ua.act = act;
        nvfp4_status st = launch_pdl(k_fp8_gemv<kGroupedUp>, static_cast<int>(S / 16), kF8Threads, (size_t)tc * H,
                                     stream, ua);
        if (st != NVFP4_OK) return st;
        Fp8GemvArgs da{};
        da.w = down->codes;
        da.gw = down->global_scale;
        da.n = static_cast<int>(H);
        da.K = static_cast<int>(S);
        da.src = act;
        da.T = tc;
        da.residual = residual ? static_cast<const uint16_t*>(residual) + (size_t)t0 * H : nullptr;
        da.out = static_cast<uint16_t*>(out) + (size_t)t0 * H;
        st = launch_pdl(k_fp8_gemv<kGroupedDown>, static_cast<int>(H / 16), kF8Threads, (size_t)tc * S, stream, da);
        if (st != NVFP4_OK) return st;
    }
    return launch_status();
}
