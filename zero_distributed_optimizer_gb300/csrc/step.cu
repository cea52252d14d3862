// Host side of the fused ZeRO-1 step: argument checks, run views, kernel
// choice and launches, and the extern "C" entry points of dopt.h.  The
// device code is in kernels.cuh.
#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "dopt_internal.h"

#include "kernels.cuh"
#include "probe.cuh"

namespace {

// A named range around each entry point for timeline profilers (a no-op
// when no profiler is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The run view of buckets [first, first + count) and the number of tiles a
// launch over it needs (0: nothing owned there).
RunView make_view(const dopt_layout *L, int32_t first, int32_t count, int64_t *tiles) {
    RunView v{};
    v.run_start = L->d_run_start;
    v.run_end = L->d_run_end;
    v.run_meta = L->d_run_meta;
    v.tile_run = L->d_tile_run;
    v.numel = L->numel;
    v.run_begin = L->bucket_run[size_t(first)];
    v.run_limit = L->bucket_run[size_t(first + count)];
    *tiles = 0;
    if (v.run_begin >= v.run_limit) return v;
    const int64_t lo = L->run_start[size_t(v.run_begin)];
    const int64_t hi = L->run_end[size_t(v.run_limit - 1)];
    v.lo = lo;
    v.hi = hi;
    v.tile0 = lo / kDoptTileElems;
    *tiles = (hi + kDoptTileElems - 1) / kDoptTileElems - v.tile0;
    return v;
}

RunView whole_view(const dopt_layout *L, int64_t *tiles) {
    return make_view(L, 0, int32_t(L->buckets.size()), tiles);
}

using StepKernel = void (*)(StepArgs);

// A launch that may start while the kernel before it on the stream is still
// running (programmatic dependent launch): the kernel waits for that one
// with griddepcontrol.wait before it touches what it wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                             Args... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = 0;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kernel, args...);
}
using NormKernel = void (*)(NormArgs);
using AllReduceKernel = void (*)(AllReduceArgs);

template <typename G, int MODE>
StepKernel pick_step_kernel(int D) {
    switch (D) {
        case 1: return dopt_step_kernel<G, 1, MODE>;
        case 2: return dopt_step_kernel<G, 2, MODE>;
        case 4: return dopt_step_kernel<G, 4, MODE>;
        case 8: return dopt_step_kernel<G, 8, MODE>;
        case 16: return dopt_step_kernel<G, 16, MODE>;
        default: return dopt_step_kernel<G, 0, MODE>;
    }
}

// The grouped kernels: D replicas in instances of R (1 < R < D); fp32
// grads at D = 16 take the run-time form.
template <typename G, int MODE>
StepKernel pick_step_kernel_grouped(int D, int R) {
    switch (D * 100 + R) {
        case 402: return dopt_step_kernel<G, 4, MODE, 2>;
        case 802: return dopt_step_kernel<G, 8, MODE, 2>;
        case 804: return dopt_step_kernel<G, 8, MODE, 4>;
        case 1602:
            if constexpr (sizeof(G) == 2) return dopt_step_kernel<G, 16, MODE, 2>;
            break;
        case 1604:
            if constexpr (sizeof(G) == 2) return dopt_step_kernel<G, 16, MODE, 4>;
            break;
        case 1608:
            if constexpr (sizeof(G) == 2) return dopt_step_kernel<G, 16, MODE, 8>;
            break;
        default: break;
    }
    return dopt_step_kernel<G, 0, MODE>;
}

// The kernels a layout takes.  D in {1, 2, 4, 8, 16} has compile-time
// forms.  With several optimizer instances of R ranks each, the step and
// all-reduce kernels have compile-time forms for every (D, R) with D in
// {4, 8, 16} (the grouped sum unrolled like the plain one, with the same
// registers); fp32 grads use them for D up to 8 (D = 16 as 2 instances ran
// 0.3 % slower than the run-time form).  Any other layout takes the
// run-time form.  Groups of one replica each (as many instances
// as ranks) add up exactly like one group, in rank order, so that layout
// takes the one-instance kernels; only the ranks' write-back stride (R = 1)
// differs, and the kernels read it at run time.
bool grouped(const dopt_layout *L) { return L->cfg.instances > 1 && L->cfg.instances < L->cfg.D; }
int group_size(const dopt_layout *L) { return L->cfg.D / L->cfg.instances; }
bool use_grouped_kernel(const dopt_layout *L, dopt_dtype grad_dtype) {
    const int D = L->cfg.D;
    return grouped(L) && (D == 4 || D == 8 || (D == 16 && grad_dtype != DOPT_FP32));
}
int kernel_D(const dopt_layout *L) { return grouped(L) ? 0 : L->cfg.D; }

template <int MODE>
StepKernel step_kernel_for(const dopt_layout *L, dopt_dtype grad_dtype) {
    const bool g = use_grouped_kernel(L, grad_dtype);
    switch (grad_dtype) {
        case DOPT_BF16:
            return g ? pick_step_kernel_grouped<__nv_bfloat16, MODE>(L->cfg.D, group_size(L))
                     : pick_step_kernel<__nv_bfloat16, MODE>(kernel_D(L));
        case DOPT_FP16:
            return g ? pick_step_kernel_grouped<__half, MODE>(L->cfg.D, group_size(L))
                     : pick_step_kernel<__half, MODE>(kernel_D(L));
        default:
            return g ? pick_step_kernel_grouped<float, MODE>(L->cfg.D, group_size(L))
                     : pick_step_kernel<float, MODE>(kernel_D(L));
    }
}

template <typename G>
NormKernel pick_norm_kernel(int D) {
    switch (D) {
        case 1: return dopt_rs_norm_kernel<G, 1>;
        case 2: return dopt_rs_norm_kernel<G, 2>;
        case 4: return dopt_rs_norm_kernel<G, 4>;
        case 8: return dopt_rs_norm_kernel<G, 8>;
        case 16: return dopt_rs_norm_kernel<G, 16>;
        default: return dopt_rs_norm_kernel<G, 0>;
    }
}

// The norm pass keeps the run-time form for several instances: its grouped
// compile-time forms (one per (D, R), 34-74 registers against 64-80 for the
// run-time form) made the clipped step 0.2 % slower at D = 8 as 2 instances
// and 6 % with fp32 grads, for 0.5 % at D = 8 as 4.
NormKernel norm_kernel_for(const dopt_layout *L, dopt_dtype grad_dtype) {
    switch (grad_dtype) {
        case DOPT_BF16: return pick_norm_kernel<__nv_bfloat16>(kernel_D(L));
        case DOPT_FP16: return pick_norm_kernel<__half>(kernel_D(L));
        default: return pick_norm_kernel<float>(kernel_D(L));
    }
}

template <typename G>
AllReduceKernel pick_allreduce_kernel(int D) {
    switch (D) {
        case 1: return dopt_allreduce_kernel<G, 1>;
        case 2: return dopt_allreduce_kernel<G, 2>;
        case 4: return dopt_allreduce_kernel<G, 4>;
        case 8: return dopt_allreduce_kernel<G, 8>;
        case 16: return dopt_allreduce_kernel<G, 16>;
        default: return dopt_allreduce_kernel<G, 0>;
    }
}

template <typename G>
AllReduceKernel pick_allreduce_kernel_grouped(int D, int R) {
    switch (D * 100 + R) {
        case 402: return dopt_allreduce_kernel<G, 4, 2>;
        case 802: return dopt_allreduce_kernel<G, 8, 2>;
        case 804: return dopt_allreduce_kernel<G, 8, 4>;
        case 1602:
            if constexpr (sizeof(G) == 2) return dopt_allreduce_kernel<G, 16, 2>;
            break;
        case 1604:
            if constexpr (sizeof(G) == 2) return dopt_allreduce_kernel<G, 16, 4>;
            break;
        case 1608:
            if constexpr (sizeof(G) == 2) return dopt_allreduce_kernel<G, 16, 8>;
            break;
        default: break;
    }
    return dopt_allreduce_kernel<G, 0>;
}

AllReduceKernel allreduce_kernel_for(const dopt_layout *L, dopt_dtype grad_dtype) {
    const bool g = use_grouped_kernel(L, grad_dtype);
    switch (grad_dtype) {
        case DOPT_BF16:
            return g ? pick_allreduce_kernel_grouped<__nv_bfloat16>(L->cfg.D, group_size(L))
                     : pick_allreduce_kernel<__nv_bfloat16>(kernel_D(L));
        case DOPT_FP16:
            return g ? pick_allreduce_kernel_grouped<__half>(L->cfg.D, group_size(L))
                     : pick_allreduce_kernel<__half>(kernel_D(L));
        default:
            return g ? pick_allreduce_kernel_grouped<float>(L->cfg.D, group_size(L))
                     : pick_allreduce_kernel<float>(kernel_D(L));
    }
}

// The staged kernels (DOPT_STEP_STAGE): one-instance layouts with D in
// {1, 2, 4, 8, 16}, plain or counted, and their shared-memory size.
template <typename G, int MODE>
StepKernel pick_staged_kernel(int D, size_t *smem) {
    switch (D) {
        case 1: *smem = staged_smem_bytes<G, 1>(); return dopt_step_staged_kernel<G, 1, MODE>;
        case 2: *smem = staged_smem_bytes<G, 2>(); return dopt_step_staged_kernel<G, 2, MODE>;
        case 4: *smem = staged_smem_bytes<G, 4>(); return dopt_step_staged_kernel<G, 4, MODE>;
        case 8: *smem = staged_smem_bytes<G, 8>(); return dopt_step_staged_kernel<G, 8, MODE>;
        case 16: *smem = staged_smem_bytes<G, 16>(); return dopt_step_staged_kernel<G, 16, MODE>;
        default: *smem = 0; return nullptr;
    }
}

template <int MODE>
StepKernel staged_kernel_for(const dopt_layout *L, dopt_dtype grad_dtype, size_t *smem) {
    if (L->cfg.instances > 1) {
        *smem = 0;
        return nullptr;
    }
    switch (grad_dtype) {
        case DOPT_BF16: return pick_staged_kernel<__nv_bfloat16, MODE>(L->cfg.D, smem);
        case DOPT_FP16: return pick_staged_kernel<__half, MODE>(L->cfg.D, smem);
        default: return pick_staged_kernel<float, MODE>(L->cfg.D, smem);
    }
}

// The staged kernels take more than the default 48 KB of dynamic shared
// memory; the limit is raised once per kernel and device.
std::mutex g_smem_mutex;
std::vector<std::pair<const void *, int>> g_smem_set;

int allow_smem(const char *who, const void *k, size_t bytes, int device) {
    std::lock_guard<std::mutex> lock(g_smem_mutex);
    for (const auto &e : g_smem_set)
        if (e.first == k && e.second == device) return DOPT_OK;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return dopt::fail(DOPT_E_CUDA, "%s: shared-memory limit: %s", who, cudaGetErrorString(e));
    }
    g_smem_set.emplace_back(k, device);
    return DOPT_OK;
}

// SMs and resident CTAs per SM of a kernel on a device, asked once.
struct GridInfo {
    const void *kernel;
    int device;
    int sms;
    int per_sm;
};
std::mutex g_grid_mutex;
std::vector<GridInfo> g_grid_info;

// (A kernel is always launched with the same block size and dynamic shared
// memory, so the kernel and the device are the key.)
void sm_occupancy(const void *k, int device, int *sms, int *per_sm, int threads = kThreads,
                  size_t smem = 0) {
    std::lock_guard<std::mutex> lock(g_grid_mutex);
    for (const GridInfo &g : g_grid_info)
        if (g.kernel == k && g.device == device) {
            *sms = g.sms;
            *per_sm = g.per_sm;
            return;
        }
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, k, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        *sms = 1;
        *per_sm = 1;
        return;  // not cached: asked again next time
    }
    g_grid_info.push_back(GridInfo{k, device, *sms, *per_sm});
}

// Launch the step kernel of a launch (or, with DOPT_STEP_STAGE, its staged
// form) over `tiles` tiles.
template <int MODE>
int launch_step_kernel(const char *who, const dopt_layout *L, dopt_dtype grad_dtype,
                       uint32_t flags, const StepArgs &a, int64_t tiles, cudaStream_t stream) {
    if constexpr (MODE == kPlain || MODE == kCounted) {
        if (flags & DOPT_STEP_STAGE) {
            size_t smem = 0;
            StepKernel k = staged_kernel_for<MODE>(L, grad_dtype, &smem);
            int rc = allow_smem(who, reinterpret_cast<const void *>(k), smem, L->device);
            if (rc != DOPT_OK) return rc;
            k<<<unsigned(tiles), kThreads, smem, stream>>>(a);
            return DOPT_OK;
        }
    }
    StepKernel k = step_kernel_for<MODE>(L, grad_dtype);
    cudaError_t e = launch_dependent(k, dim3(unsigned(tiles)), dim3(kThreads), stream, a);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return dopt::fail(DOPT_E_CUDA, "%s: step launch: %s", who, cudaGetErrorString(e));
    }
    return DOPT_OK;
}


// Grid of the norm pass.  For the compile-time kernels at D = 4, 8 and 16
// (one instance), 4 tiles per CTA: its CTAs leave the SMs one by one to the
// step pass that follows, as step kernels do.  Otherwise a persistent grid
// of at most 6 CTAs per SM: at D = 1 and 2, for the run-time-D kernel
// (other D, several instances) and with more CTAs per SM, the tiled grid
// measured slower.  The partials are summed exactly, so the grid changes
// nothing in the result.
constexpr int64_t kNormTilesPerCta = 4;
constexpr int kNormPersistentPerSm = 6;

int norm_grid(NormKernel k, const dopt_layout *L, int64_t n_tiles) {
    n_tiles = std::max<int64_t>(n_tiles, 1);
    if (L->cfg.instances == 1 && (L->cfg.D == 4 || L->cfg.D == 8 || L->cfg.D == 16))
        return int((n_tiles + kNormTilesPerCta - 1) / kNormTilesPerCta);
    int sms = 0, per_sm = 0;
    sm_occupancy(reinterpret_cast<const void *>(k), L->device, &sms, &per_sm);
    const int64_t g = int64_t(std::max(sms, 1)) * std::min(std::max(per_sm, 1), kNormPersistentPerSm);
    return int(std::min(g, n_tiles));
}

int check_device_tables(const dopt_layout *L, const char *who) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
    if (L->device != dev || !L->d_block)
        return dopt::fail(DOPT_E_STATE,
                          "%s: layout tables are not on device %d (call dopt_layout_to_device)",
                          who, dev);
    return DOPT_OK;
}

int check_replicas(const char *who, int D, const void *const *ptrs) {
    using dopt::fail;
    for (int r = 0; r < D; ++r) {
        if (!ptrs[r]) return fail(DOPT_E_ARG, "%s: replica %d pointer is NULL", who, r);
        if (!aligned16(ptrs[r]))
            return fail(DOPT_E_ALIGN, "%s: replica %d pointer is not 16-byte aligned", who, r);
    }
    return DOPT_OK;
}

// Host checks shared by the step entry points; nothing is queued before
// they pass.
int check_step_args(const char *who, const dopt_layout *L, const dopt_adam_cfg *cfg,
                    int64_t step, const void *const *grad_replicas, dopt_dtype grad_dtype,
                    const float *master, const float *exp_avg, const float *exp_avg_sq,
                    void *const *param_replicas, uint32_t flags, const float *main_grad,
                    uint32_t extra_flags = 0) {
    using dopt::fail;
    if (!L || !cfg || !grad_replicas || !param_replicas || !master || !exp_avg || !exp_avg_sq)
        return fail(DOPT_E_ARG, "%s: NULL argument", who);
    if (step < 1) return fail(DOPT_E_ARG, "%s: step=%lld < 1", who, (long long)step);
    if (grad_dtype != DOPT_BF16 && grad_dtype != DOPT_FP32 && grad_dtype != DOPT_FP16)
        return fail(DOPT_E_ARG, "%s: unknown grad dtype %d", who, int(grad_dtype));
    if (flags & ~(uint32_t(DOPT_STEP_GATHER | DOPT_STEP_HOST_GRADS | DOPT_STEP_ROUND_GRAD |
                           DOPT_STEP_PARAMS_FP16 | DOPT_STEP_HOST_PARAMS) |
                  extra_flags))
        return fail(DOPT_E_ARG, "%s: unknown flags 0x%x", who, flags);
    if (flags & DOPT_STEP_STAGE) {
        const int D = L->cfg.D;
        if (L->cfg.instances > 1 || (D != 1 && D != 2 && D != 4 && D != 8 && D != 16))
            return fail(DOPT_E_ARG, "%s: DOPT_STEP_STAGE needs one instance and D in {1, 2, 4, 8, 16}",
                        who);
        if (flags & (DOPT_STEP_HOST_GRADS | DOPT_STEP_HOST_PARAMS))
            return fail(DOPT_E_ARG, "%s: DOPT_STEP_STAGE takes device buffers only", who);
    }
    if (!(cfg->lr >= 0.0f) || !std::isfinite(cfg->lr) || !(cfg->beta1 >= 0.0f && cfg->beta1 < 1.0f) ||
        !(cfg->beta2 >= 0.0f && cfg->beta2 < 1.0f) || !(cfg->eps >= 0.0f) || !std::isfinite(cfg->eps) ||
        !(cfg->weight_decay >= 0.0f) || !std::isfinite(cfg->weight_decay) ||
        !std::isfinite(cfg->grad_scale))
        return fail(DOPT_E_ARG, "%s: hyper-parameter out of range", who);
    const int D = L->cfg.D;
    int rc = check_replicas(who, D, grad_replicas);
    if (rc != DOPT_OK) return rc;
    rc = check_replicas(who, D, const_cast<const void *const *>(param_replicas));
    if (rc != DOPT_OK) return rc;
    if (!aligned16(master) || !aligned16(exp_avg) || !aligned16(exp_avg_sq) ||
        (main_grad && !aligned16(main_grad)))
        return fail(DOPT_E_ALIGN, "%s: state pointer is not 16-byte aligned", who);
    return DOPT_OK;
}

// With DOPT_STEP_HOST_GRADS the grad pointers are pinned host buffers: each
// is replaced by the device's mapping of it, and anything else is refused.
int resolve_grads(const char *who, int D, const void *const *grad_replicas, uint32_t flags,
                  const void **out) {
    using dopt::fail;
    for (int r = 0; r < D; ++r) out[r] = grad_replicas[r];
    if (!(flags & DOPT_STEP_HOST_GRADS)) return DOPT_OK;
    for (int r = 0; r < D; ++r) {
        cudaPointerAttributes at{};
        cudaError_t e = cudaPointerGetAttributes(&at, grad_replicas[r]);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(DOPT_E_ARG, "%s: grad replica %d: cudaPointerGetAttributes: %s", who, r,
                        cudaGetErrorString(e));
        }
        if (at.type != cudaMemoryTypeHost || !at.devicePointer)
            return fail(DOPT_E_ARG, "%s: grad replica %d is not pinned host memory mapped to the "
                        "device", who, r);
        const char *base = static_cast<const char *>(at.devicePointer);
        out[r] = base + (static_cast<const char *>(grad_replicas[r]) -
                         static_cast<const char *>(at.hostPointer));
        if (!aligned16(out[r]))
            return fail(DOPT_E_ALIGN, "%s: grad replica %d mapping is not 16-byte aligned", who, r);
    }
    return DOPT_OK;
}

// With DOPT_STEP_HOST_PARAMS each param replica may be a pinned host buffer
// (replaced by the device's mapping of it) or device memory (kept);
// anything else is refused.
int resolve_params(const char *who, int D, void *const *param_replicas, uint32_t flags,
                   void **out) {
    using dopt::fail;
    for (int r = 0; r < D; ++r) out[r] = param_replicas[r];
    if (!(flags & DOPT_STEP_HOST_PARAMS)) return DOPT_OK;
    for (int r = 0; r < D; ++r) {
        cudaPointerAttributes at{};
        cudaError_t e = cudaPointerGetAttributes(&at, param_replicas[r]);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(DOPT_E_ARG, "%s: param replica %d: cudaPointerGetAttributes: %s", who, r,
                        cudaGetErrorString(e));
        }
        if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) continue;
        if (at.type != cudaMemoryTypeHost || !at.devicePointer)
            return fail(DOPT_E_ARG, "%s: param replica %d is neither device memory nor pinned "
                        "host memory mapped to the device", who, r);
        char *base = static_cast<char *>(at.devicePointer);
        out[r] = base + (static_cast<char *>(param_replicas[r]) - static_cast<char *>(at.hostPointer));
        if (!aligned16(out[r]))
            return fail(DOPT_E_ALIGN, "%s: param replica %d mapping is not 16-byte aligned", who, r);
    }
    return DOPT_OK;
}

void fill_step_args(StepArgs &a, const dopt_layout *L, const dopt_adam_cfg *cfg, int64_t step,
                    const void *const *grad_replicas, float *master, float *exp_avg,
                    float *exp_avg_sq, void *const *param_replicas, uint32_t flags) {
    const int D = L->cfg.D;
    for (int r = 0; r < D; ++r) {
        a.grads[r] = grad_replicas[r];
        a.params[r] = param_replicas[r];
    }
    a.master = master;
    a.exp_avg = exp_avg;
    a.exp_avg_sq = exp_avg_sq;
    a.D = D;
    a.R = L->R;
    a.gather = (flags & DOPT_STEP_GATHER) ? 1 : 0;
    a.round_grad = (flags & DOPT_STEP_ROUND_GRAD) ? 1 : 0;
    a.param_f16 = (flags & DOPT_STEP_PARAMS_FP16) ? 1 : 0;
    a.sc = scalars_for(*cfg, step);
}

int launch_error(const char *who, const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, "%s: %s launch: %s", who, what, cudaGetErrorString(e));
    return DOPT_OK;
}

// The arguments of one step launch over buckets [first, first+count);
// *tiles = 0 when nothing there is owned (then nothing else is checked).
int prepare_step(const char *who, const dopt_layout *L, const dopt_adam_cfg *cfg, int64_t step,
                 int32_t first, int32_t count, const void *const *grad_replicas,
                 float *master, float *exp_avg, float *exp_avg_sq, void *const *param_replicas,
                 uint32_t flags, float *main_grad_out, StepArgs &a, int64_t *tiles) {
    a.rv = make_view(L, first, count, tiles);
    if (*tiles == 0) return DOPT_OK;
    int rc = check_device_tables(L, who);
    if (rc != DOPT_OK) return rc;
    const void *grads[DOPT_MAX_D];
    rc = resolve_grads(who, L->cfg.D, grad_replicas, flags, grads);
    if (rc != DOPT_OK) return rc;
    void *params[DOPT_MAX_D];
    rc = resolve_params(who, L->cfg.D, param_replicas, flags, params);
    if (rc != DOPT_OK) return rc;
    fill_step_args(a, L, cfg, step, grads, master, exp_avg, exp_avg_sq, params, flags);
    a.main_grad_out = main_grad_out;
    return DOPT_OK;
}

// One step launch (plain or all-reduce mode) over buckets [first, first+count).
template <int MODE>
int launch_step(const char *who, const dopt_layout *L, const dopt_adam_cfg *cfg, int64_t step,
                int32_t first, int32_t count, const void *const *grad_replicas,
                dopt_dtype grad_dtype, float *master, float *exp_avg, float *exp_avg_sq,
                void *const *param_replicas, uint32_t flags, float *main_grad_out,
                cudaStream_t stream) {
    int64_t tiles = 0;
    StepArgs a{};
    int rc = prepare_step(who, L, cfg, step, first, count, grad_replicas, master, exp_avg,
                          exp_avg_sq, param_replicas, flags, main_grad_out, a, &tiles);
    if (rc != DOPT_OK || tiles == 0) return rc;
    rc = launch_step_kernel<MODE>(who, L, grad_dtype, flags, a, tiles, stream);
    if (rc != DOPT_OK) return rc;
    return launch_error(who, "step");
}

// The two launches of the clipped step, with the workspace given as a
// device address.
int launch_clipped(const char *who, const dopt_layout *L, const dopt_adam_cfg *cfg,
                   int64_t step, float max_norm, const void *const *grad_replicas,
                   dopt_dtype grad_dtype, float *master, float *exp_avg, float *exp_avg_sq,
                   void *const *param_replicas, uint32_t flags, float *main_grad,
                   ClipWorkspace *ws, float *norm_out, cudaStream_t stream,
                   const CounterBlock *counter = nullptr) {
    using dopt::fail;
    NormArgs na{};
    const int D = L->cfg.D;
    const void *grads[DOPT_MAX_D];
    int rc = resolve_grads(who, D, grad_replicas, flags, grads);
    if (rc != DOPT_OK) return rc;
    void *params[DOPT_MAX_D];
    rc = resolve_params(who, D, param_replicas, flags, params);
    if (rc != DOPT_OK) return rc;
    for (int r = 0; r < D; ++r) na.grads[r] = grads[r];
    na.main_grad = main_grad;
    na.ws = ws;
    na.norm_out = norm_out;
    na.rv = whole_view(L, &na.n_tiles);
    na.D = D;
    na.R = L->R;
    na.round_grad = (flags & DOPT_STEP_ROUND_GRAD) ? 1 : 0;
    na.skip_nonfinite = (flags & DOPT_STEP_SKIP_NONFINITE) ? 1 : 0;
    na.scale = cfg->grad_scale;
    na.max_norm = max_norm;
    na.counter = const_cast<CounterBlock *>(counter);
    NormKernel nk = norm_kernel_for(L, grad_dtype);
    const int grid_a = norm_grid(nk, L, na.n_tiles);
    dopt_clip_reset_kernel<<<1, kThreads, 0, stream>>>(ws);
    rc = launch_error(who, "workspace reset");
    if (rc != DOPT_OK) return rc;
    cudaError_t e = launch_dependent(nk, dim3(unsigned(grid_a)), dim3(kThreads), stream, na);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DOPT_E_CUDA, "%s: norm launch: %s", who, cudaGetErrorString(e));
    }
    rc = launch_error(who, "norm");
    if (rc != DOPT_OK) return rc;
    e = launch_dependent(dopt_clip_finalize_kernel, dim3(1), dim3(kThreads), stream, na);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DOPT_E_CUDA, "%s: finalize launch: %s", who, cudaGetErrorString(e));
    }
    rc = launch_error(who, "finalize");
    if (rc != DOPT_OK) return rc;

    StepArgs a{};
    int64_t tiles = 0;
    a.rv = whole_view(L, &tiles);
    fill_step_args(a, L, cfg, step, grads, master, exp_avg, exp_avg_sq, params, flags);
    a.main_grad_in = main_grad;
    a.clip_coef = &ws->coef;
    a.skip_nonfinite = na.skip_nonfinite;
    a.counter = counter;  // the counted clipped step: scalars and status from the counter
    StepKernel k = pick_step_kernel<float, kFromMain>(kernel_D(L));
    // a programmatic dependent of the finalize kernel: its CTAs start as the
    // norm pass's CTAs leave, load master/m/v and wait for the finalize
    // kernel (and so the norm pass) to complete before they read the main
    // grads and the coefficient
    cudaError_t le = launch_dependent(k, dim3(unsigned(tiles)), dim3(kThreads), stream, a);
    if (le != cudaSuccess) {
        cudaGetLastError();
        return fail(DOPT_E_CUDA, "%s: step launch: %s", who, cudaGetErrorString(le));
    }
    return launch_error(who, "step");
}

// The counter kernel of a counted step, launched as a programmatic dependent
// of the kernel before it on the stream (see dopt_count_step_kernel).
int launch_counter(const char *who, CounterBlock *c, const dopt_adam_cfg *cfg,
                   cudaStream_t stream) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(1);
    lc.blockDim = dim3(4);
    lc.dynamicSmemBytes = 0;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const dopt_adam_cfg cfg_copy = *cfg;
    cudaError_t le = cudaLaunchKernelEx(&lc, dopt_count_step_kernel, c, cfg_copy);
    if (le != cudaSuccess) {
        cudaGetLastError();
        return dopt::fail(DOPT_E_CUDA, "%s: counter launch: %s", who, cudaGetErrorString(le));
    }
    return launch_error(who, "counter");
}

// Checks of a step counter argument.
int check_counter(const char *who, const dopt_step_counter *counter) {
    if (!counter) return dopt::fail(DOPT_E_ARG, "%s: counter is NULL", who);
    if (!aligned16(counter))
        return dopt::fail(DOPT_E_ALIGN, "%s: counter is not 16-byte aligned", who);
    return DOPT_OK;
}

// Checks of the clipped entry points beyond the step's own.
int check_clip_args(const char *who, const float *main_grad, const float *norm_out,
                    float max_norm) {
    using dopt::fail;
    if (!main_grad) return fail(DOPT_E_ARG, "%s: main_grad is required", who);
    if (norm_out && (reinterpret_cast<uintptr_t>(norm_out) & 7u))
        return fail(DOPT_E_ALIGN, "%s: norm_out misaligned", who);
    if (!(max_norm > 0.0f) || !std::isfinite(max_norm))
        return fail(DOPT_E_ARG, "%s: max_norm must be positive and finite", who);
    return DOPT_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Entry points
// ---------------------------------------------------------------------------

extern "C" int dopt_device_checks(int reset, uint32_t *flags, int64_t *first_bad) {
    using dopt::fail;
    if (!flags || !first_bad) return fail(DOPT_E_ARG, "dopt_device_checks: NULL output");
#ifdef DOPT_DEVICE_CHECKS
    unsigned int f = 0;
    unsigned long long first = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&f, g_check_flags, sizeof f);
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&first, g_check_first, sizeof first);
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        const unsigned long long none = ~0ull;
        e = cudaMemcpyToSymbol(g_check_flags, &zero, sizeof zero);
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_first, &none, sizeof none);
    }
    if (e != cudaSuccess)
        return fail(DOPT_E_CUDA, "dopt_device_checks: %s", cudaGetErrorString(e));
    *flags = f;
    *first_bad = static_cast<int64_t>(first);
    return DOPT_OK;
#else
    (void)reset;
    return fail(DOPT_E_STATE, "dopt_device_checks: this library was built without DOPT_DEVICE_CHECKS");
#endif
}

extern "C" int dopt_stream_probe(int32_t reads, int32_t writes, const void *const *read_buffers,
                                 void *const *write_buffers, int64_t n_vectors,
                                 cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_stream_probe";
    if (reads < 0 || writes < 0 || reads > kMaxProbeStreams || writes > kMaxProbeStreams ||
        reads + writes == 0)
        return fail(DOPT_E_ARG, "%s: %d read and %d write streams (0..%d each, not both 0)", who,
                    reads, writes, kMaxProbeStreams);
    if (n_vectors < 0 || n_vectors > (int64_t(1) << 40))
        return fail(DOPT_E_ARG, "%s: n_vectors out of range", who);
    if ((reads && !read_buffers) || (writes && !write_buffers))
        return fail(DOPT_E_ARG, "%s: NULL buffer array", who);
    ProbeArgs a{};
    for (int r = 0; r < reads; ++r) {
        if (!read_buffers[r]) return fail(DOPT_E_ARG, "%s: read buffer %d is NULL", who, r);
        if (!aligned16(read_buffers[r])) return fail(DOPT_E_ALIGN, "%s: read buffer %d misaligned", who, r);
        a.in[r] = static_cast<const uint4 *>(read_buffers[r]);
    }
    for (int w = 0; w < writes; ++w) {
        if (!write_buffers[w]) return fail(DOPT_E_ARG, "%s: write buffer %d is NULL", who, w);
        if (!aligned16(write_buffers[w])) return fail(DOPT_E_ALIGN, "%s: write buffer %d misaligned", who, w);
        a.out[w] = static_cast<uint4 *>(write_buffers[w]);
    }
    a.n = n_vectors;
    a.reads = reads;
    a.writes = writes;
    if (n_vectors == 0) return DOPT_OK;
    const int64_t blocks = (n_vectors + kThreads - 1) / kThreads;
    if (blocks >= (int64_t(1) << 31)) return fail(DOPT_E_ARG, "%s: too many vectors", who);
    void (*k)(ProbeArgs) = reads <= 1   ? dopt_stream_probe_kernel<1>
                           : reads <= 2 ? dopt_stream_probe_kernel<2>
                           : reads <= 4 ? dopt_stream_probe_kernel<4>
                           : reads <= 8 ? dopt_stream_probe_kernel<8>
                                        : dopt_stream_probe_kernel<16>;
    k<<<unsigned(blocks), kThreads, 0, stream>>>(a);
    return launch_error(who, "probe");
}

extern "C" int dopt_stage_timeouts(int reset, uint32_t *count) {
    using dopt::fail;
    dopt::clear_error();
    if (!count) return fail(DOPT_E_ARG, "dopt_stage_timeouts: NULL output");
    unsigned int c = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&c, g_stage_timeouts, sizeof c);
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_stage_timeouts, &zero, sizeof zero);
    }
    if (e != cudaSuccess) return fail(DOPT_E_CUDA, "dopt_stage_timeouts: %s", cudaGetErrorString(e));
    *count = c;
    return DOPT_OK;
}

extern "C" int dopt_stage_wait_test(uint32_t extra_bytes) {
    using dopt::fail;
    dopt::clear_error();
#ifdef DOPT_DEVICE_CHECKS
    // the largest phantom count taken: well inside an mbarrier's
    // transaction-count range with the largest staged tile (D = 16 fp32)
    constexpr uint32_t kMaxStagePhantomBytes = 1u << 16;
    if (extra_bytes > kMaxStagePhantomBytes)
        return fail(DOPT_E_ARG, "dopt_stage_wait_test: extra_bytes above %u", kMaxStagePhantomBytes);
    const unsigned int v = extra_bytes;
    const cudaError_t e = cudaMemcpyToSymbol(g_stage_phantom_bytes, &v, sizeof v);
    if (e != cudaSuccess) return fail(DOPT_E_CUDA, "dopt_stage_wait_test: %s", cudaGetErrorString(e));
    return DOPT_OK;
#else
    (void)extra_bytes;
    return fail(DOPT_E_STATE, "dopt_stage_wait_test: this library was built without DOPT_DEVICE_CHECKS");
#endif
}

extern "C" int dopt_step(const dopt_layout *L, const dopt_adam_cfg *cfg, int64_t step,
                         const void *const *grad_replicas, dopt_dtype grad_dtype, float *master,
                         float *exp_avg, float *exp_avg_sq, void *const *param_replicas,
                         uint32_t flags, float *main_grad_out, cudaStream_t stream) {
    dopt::clear_error();
    const char *who = "dopt_step";
    NvtxRange range(who);
    int rc = check_step_args(who, L, cfg, step, grad_replicas, grad_dtype, master, exp_avg,
                             exp_avg_sq, param_replicas, flags, main_grad_out, DOPT_STEP_STAGE);
    if (rc != DOPT_OK) return rc;
    return launch_step<kPlain>(who, L, cfg, step, 0, int32_t(L->buckets.size()), grad_replicas,
                               grad_dtype, master, exp_avg, exp_avg_sq, param_replicas, flags,
                               main_grad_out, stream);
}

extern "C" int dopt_step_buckets(const dopt_layout *L, const dopt_adam_cfg *cfg, int64_t step,
                                 int32_t first_bucket, int32_t n_buckets,
                                 const void *const *grad_replicas, dopt_dtype grad_dtype,
                                 float *master, float *exp_avg, float *exp_avg_sq,
                                 void *const *param_replicas, uint32_t flags,
                                 float *main_grad_out, cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_step_buckets";
    NvtxRange range(who);
    int rc = check_step_args(who, L, cfg, step, grad_replicas, grad_dtype, master, exp_avg,
                             exp_avg_sq, param_replicas, flags, main_grad_out, DOPT_STEP_STAGE);
    if (rc != DOPT_OK) return rc;
    const int32_t nb = int32_t(L->buckets.size());
    if (first_bucket < 0 || n_buckets < 0 || first_bucket > nb || n_buckets > nb - first_bucket)
        return fail(DOPT_E_ARG, "%s: buckets [%d, %d+%d) outside 0..%d", who, first_bucket,
                    first_bucket, n_buckets, nb);
    return launch_step<kPlain>(who, L, cfg, step, first_bucket, n_buckets, grad_replicas,
                               grad_dtype, master, exp_avg, exp_avg_sq, param_replicas, flags,
                               main_grad_out, stream);
}

extern "C" int dopt_step_counted(const dopt_layout *L, const dopt_adam_cfg *cfg,
                                 dopt_step_counter *counter, const void *const *grad_replicas,
                                 dopt_dtype grad_dtype, float *master, float *exp_avg,
                                 float *exp_avg_sq, void *const *param_replicas, uint32_t flags,
                                 float *main_grad_out, cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_step_counted";
    NvtxRange range(who);
    int rc = check_step_args(who, L, cfg, 1, grad_replicas, grad_dtype, master, exp_avg,
                             exp_avg_sq, param_replicas, flags, main_grad_out, DOPT_STEP_STAGE);
    if (rc != DOPT_OK) return rc;
    rc = check_counter(who, counter);
    if (rc != DOPT_OK) return rc;
    // every check before the first launch: the counter advances only
    // together with the step it counts
    int64_t tiles = 0;
    StepArgs a{};
    rc = prepare_step(who, L, cfg, 1, 0, int32_t(L->buckets.size()), grad_replicas, master,
                      exp_avg, exp_avg_sq, param_replicas, flags, main_grad_out, a, &tiles);
    if (rc != DOPT_OK) return rc;
    CounterBlock *c = reinterpret_cast<CounterBlock *>(counter);
    rc = launch_counter(who, c, cfg, stream);
    if (rc != DOPT_OK || tiles == 0) return rc;
    a.counter = c;
    rc = launch_step_kernel<kCounted>(who, L, grad_dtype, flags, a, tiles, stream);
    if (rc != DOPT_OK) return rc;
    return launch_error(who, "step");
}

extern "C" int dopt_step_allreduce(const dopt_layout *L, const dopt_adam_cfg *cfg, int64_t step,
                                   void *const *grad_replicas, dopt_dtype grad_dtype,
                                   float *master, float *exp_avg, float *exp_avg_sq,
                                   void *const *param_replicas, uint32_t flags,
                                   float *main_grad_out, cudaStream_t stream) {
    dopt::clear_error();
    const char *who = "dopt_step_allreduce";
    NvtxRange range(who);
    const void *const *grads = const_cast<const void *const *>(grad_replicas);
    int rc = check_step_args(who, L, cfg, step, grads, grad_dtype, master, exp_avg, exp_avg_sq,
                             param_replicas, flags, main_grad_out);
    if (rc != DOPT_OK) return rc;
    return launch_step<kWriteGrads>(who, L, cfg, step, 0, int32_t(L->buckets.size()), grads,
                                    grad_dtype, master, exp_avg, exp_avg_sq, param_replicas,
                                    flags, main_grad_out, stream);
}

extern "C" int dopt_allreduce(const dopt_layout *L, void *const *grad_replicas,
                              dopt_dtype grad_dtype, float grad_scale, cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_allreduce";
    NvtxRange range(who);
    if (!L || !grad_replicas) return fail(DOPT_E_ARG, "%s: NULL argument", who);
    if (grad_dtype != DOPT_BF16 && grad_dtype != DOPT_FP32 && grad_dtype != DOPT_FP16)
        return fail(DOPT_E_ARG, "%s: unknown grad dtype %d", who, int(grad_dtype));
    if (!std::isfinite(grad_scale)) return fail(DOPT_E_ARG, "%s: grad_scale not finite", who);
    const int D = L->cfg.D;
    int rc = check_replicas(who, D, const_cast<const void *const *>(grad_replicas));
    if (rc != DOPT_OK) return rc;
    AllReduceArgs a{};
    int64_t tiles = 0;
    a.rv = whole_view(L, &tiles);
    if (tiles == 0) return DOPT_OK;
    rc = check_device_tables(L, who);
    if (rc != DOPT_OK) return rc;
    for (int r = 0; r < D; ++r) a.grads[r] = grad_replicas[r];
    a.D = D;
    a.R = L->R;
    a.scale = grad_scale;
    AllReduceKernel k = allreduce_kernel_for(L, grad_dtype);
    cudaError_t e = launch_dependent(k, dim3(unsigned(tiles)), dim3(kThreads), stream, a);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DOPT_E_CUDA, "%s: all-reduce launch: %s", who, cudaGetErrorString(e));
    }
    return launch_error(who, "all-reduce");
}

extern "C" int dopt_step_clipped(const dopt_layout *L, const dopt_adam_cfg *cfg, int64_t step,
                                 float max_norm, const void *const *grad_replicas,
                                 dopt_dtype grad_dtype, float *master, float *exp_avg,
                                 float *exp_avg_sq, void *const *param_replicas, uint32_t flags,
                                 float *main_grad, void *workspace, float *norm_out,
                                 cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_step_clipped";
    NvtxRange range(who);
    int rc = check_step_args(who, L, cfg, step, grad_replicas, grad_dtype, master, exp_avg,
                             exp_avg_sq, param_replicas, flags, main_grad,
                             DOPT_STEP_SKIP_NONFINITE);
    if (rc != DOPT_OK) return rc;
    rc = check_clip_args(who, main_grad, norm_out, max_norm);
    if (rc != DOPT_OK) return rc;
    if (!workspace) return fail(DOPT_E_ARG, "%s: workspace is required", who);
    if (!aligned16(workspace)) return fail(DOPT_E_ALIGN, "%s: workspace misaligned", who);
    if (L->run_start.empty()) return DOPT_OK;
    rc = check_device_tables(L, who);
    if (rc != DOPT_OK) return rc;
    return launch_clipped(who, L, cfg, step, max_norm, grad_replicas, grad_dtype, master,
                          exp_avg, exp_avg_sq, param_replicas, flags, main_grad,
                          static_cast<ClipWorkspace *>(workspace), norm_out, stream);
}

extern "C" int dopt_step_clipped_counted(const dopt_layout *L, const dopt_adam_cfg *cfg,
                                         dopt_step_counter *counter, float max_norm,
                                         const void *const *grad_replicas, dopt_dtype grad_dtype,
                                         float *master, float *exp_avg, float *exp_avg_sq,
                                         void *const *param_replicas, uint32_t flags,
                                         float *main_grad, void *workspace, float *norm_out,
                                         cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_step_clipped_counted";
    NvtxRange range(who);
    int rc = check_step_args(who, L, cfg, 1, grad_replicas, grad_dtype, master, exp_avg,
                             exp_avg_sq, param_replicas, flags, main_grad,
                             DOPT_STEP_SKIP_NONFINITE);
    if (rc != DOPT_OK) return rc;
    rc = check_clip_args(who, main_grad, norm_out, max_norm);
    if (rc != DOPT_OK) return rc;
    rc = check_counter(who, counter);
    if (rc != DOPT_OK) return rc;
    if (!workspace) return fail(DOPT_E_ARG, "%s: workspace is required", who);
    if (!aligned16(workspace)) return fail(DOPT_E_ALIGN, "%s: workspace misaligned", who);
    const bool empty = L->run_start.empty();
    if (!empty) {
        rc = check_device_tables(L, who);
        if (rc != DOPT_OK) return rc;
        const void *grads[DOPT_MAX_D];
        rc = resolve_grads(who, L->cfg.D, grad_replicas, flags, grads);
        if (rc != DOPT_OK) return rc;
        void *params[DOPT_MAX_D];
        rc = resolve_params(who, L->cfg.D, param_replicas, flags, params);
        if (rc != DOPT_OK) return rc;
    }
    // every check before the first launch: the counter advances only
    // together with the step it counts
    CounterBlock *c = reinterpret_cast<CounterBlock *>(counter);
    rc = launch_counter(who, c, cfg, stream);
    if (rc != DOPT_OK || empty) return rc;
    return launch_clipped(who, L, cfg, 1, max_norm, grad_replicas, grad_dtype, master, exp_avg,
                          exp_avg_sq, param_replicas, flags, main_grad,
                          static_cast<ClipWorkspace *>(workspace), norm_out, stream, c);
}

// ---------------------------------------------------------------------------
// dopt_step_clipped_noalloc: the same two launches with the scratch in a
// static device array instead of a caller workspace (see dopt.h).
// ---------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_noalloc_scratch[DOPT_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_address[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device.  In host code the array's name only stands for the symbol; the
// kernels must get this address.
int noalloc_scratch(int device, void **out) {
    using dopt::fail;
    if (device < 0 || device >= kMaxDevices)
        return fail(DOPT_E_ARG, "dopt_step_clipped_noalloc: device %d out of range", device);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_address[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(DOPT_E_CUDA, "dopt_step_clipped_noalloc: cudaGetSymbolAddress: %s",
                        cudaGetErrorString(e));
        g_scratch_address[device] = p;
    }
    *out = g_scratch_address[device];
    return DOPT_OK;
}

}  // namespace

extern "C" int dopt_step_clipped_noalloc(const dopt_layout *L, const dopt_adam_cfg *cfg,
                                         int64_t step, float max_norm,
                                         const void *const *grad_replicas, dopt_dtype grad_dtype,
                                         float *master, float *exp_avg, float *exp_avg_sq,
                                         void *const *param_replicas, uint32_t flags,
                                         float *main_grad, float *norm_out, cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_step_clipped_noalloc";
    NvtxRange range(who);
    int rc = check_step_args(who, L, cfg, step, grad_replicas, grad_dtype, master, exp_avg,
                             exp_avg_sq, param_replicas, flags, main_grad);
    if (rc != DOPT_OK) return rc;
    rc = check_clip_args(who, main_grad, norm_out, max_norm);
    if (rc != DOPT_OK) return rc;
    if (L->run_start.empty()) return DOPT_OK;
    rc = check_device_tables(L, who);
    if (rc != DOPT_OK) return rc;
    static_assert(sizeof(ClipWorkspace) <= sizeof(g_noalloc_scratch), "scratch size");
    void *scratch = nullptr;
    rc = noalloc_scratch(L->device, &scratch);
    if (rc != DOPT_OK) return rc;
    return launch_clipped(who, L, cfg, step, max_norm, grad_replicas, grad_dtype, master, exp_avg,
                          exp_avg_sq, param_replicas, flags, main_grad,
                          static_cast<ClipWorkspace *>(scratch), norm_out, stream);
}

extern "C" int dopt_gather(const dopt_layout *L, void *const *param_replicas, cudaStream_t stream) {
    using dopt::fail;
    dopt::clear_error();
    const char *who = "dopt_gather";
    NvtxRange range(who);
    if (!L || !param_replicas) return fail(DOPT_E_ARG, "%s: NULL argument", who);
    const int D = L->cfg.D;
    int rc = check_replicas(who, D, const_cast<const void *const *>(param_replicas));
    if (rc != DOPT_OK) return rc;
    if (L->R == 1) return DOPT_OK;  // every rank is alone in its instance
    GatherArgs a{};
    int64_t tiles = 0;
    a.rv = whole_view(L, &tiles);
    if (tiles == 0) return DOPT_OK;
    rc = check_device_tables(L, who);
    if (rc != DOPT_OK) return rc;
    for (int r = 0; r < D; ++r) a.params[r] = param_replicas[r];
    a.D = D;
    a.R = L->R;
    cudaError_t e = launch_dependent(dopt_gather_kernel, dim3(unsigned(tiles)), dim3(kThreads),
                                     stream, a);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DOPT_E_CUDA, "%s: gather launch: %s", who, cudaGetErrorString(e));
    }
    return launch_error(who, "gather");
}
