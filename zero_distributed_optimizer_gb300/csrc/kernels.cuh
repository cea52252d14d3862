#pragma once
// Device code of the fused ZeRO-1 distributed-optimizer step for sm_103a,
// the clipped step, the all-reduce and the standalone all-gather (Megatron-LM
// distributed-optimizer page, §4.2-§4.4 and §5; distributed-training
// tutorial, "AllReduce" and §8.3).  Included by step.cu only.
//
// Work split.  With all D ranks held on one device, every owned element i
// is independent: rank q's reduce-scatter reads the D replicas at i, its
// Adam reads and writes the fp32 master/m/v at i (the four-way range map
// composes to the identity on the buffer index, because main params are
// stored buffer-indexed), and the write-back plus all-gather writes the D
// param replicas at i.  So one launch covers any set of buckets (all of them
// for dopt_step), in tiles of 2048 elements (256 threads x 8 elements).
//
// Per element the only facts needed are "owned or padding", "decays or
// not" and the owner rank.  They come from the run table (maximal owned
// stretches of one bucket with one rank and one decay flag).  A launch
// covers a contiguous range of runs (a RunView); each CTA gets the first run
// of its tile from a host-built index, each warp finds the first run of its
// own 256 elements with one ballot over 32 run ends, and each thread walks
// forward to its 8 elements.  An 8-element vector inside one run goes
// through 128-bit loads and stores; a vector that straddles a run edge
// (param with another decay flag, a rank edge, padding, the edge of the
// launch's range) is done element by element and touches owned elements of
// the range only, the warp's such vectors shared out over its lanes.
//
// Arithmetic.  Every fp32 operation uses the round-to-nearest intrinsics
// (__fmul_rn, __fadd_rn, __fsub_rn, __fdiv_rn, __fsqrt_rn), so no multiply
// and add are fused and divide and square root are IEEE; the rank order of
// the reduction is the loop order.
#include <cmath>
#include <cstddef>
#include <cstdint>

#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dopt_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;
static_assert(kThreads * kVec == kDoptTileElems, "tile size must match the host table");

struct Scalars {
    float b1, b2, omb1, omb2, decay, step_size, bc2_sqrt, eps, scale;
};

// The two scalars that depend on the step number t: step_size =
// lr / (1 - beta1^t) and bc2_sqrt = sqrt(1 - beta2^t), the bias corrections
// of Adam.  Each is evaluated in double and rounded to float once, with
// beta^t = pow(beta, t): the host entry points call the C library's pow
// (step_size_host, bc2_sqrt_host), so their scalars are those of that
// definition, bit for bit.  The device (the counter kernel of the counted
// steps) has no such pow; counted_scalar below reaches the same floats.
inline float step_size_host(const dopt_adam_cfg &c, int64_t t) {
    return float(double(c.lr) / (1.0 - std::pow(double(c.beta1), double(t))));
}
inline float bc2_sqrt_host(const dopt_adam_cfg &c, int64_t t) {
    return float(std::sqrt(1.0 - std::pow(double(c.beta2), double(t))));
}

// The scalars that do not depend on the step number, each evaluated in
// double and rounded to float once.
__host__ __device__ inline Scalars scalars_for_fixed(const dopt_adam_cfg &c) {
    const double lr = c.lr, b1 = c.beta1, b2 = c.beta2, wd = c.weight_decay;
    Scalars s;
    s.b1 = c.beta1;
    s.b2 = c.beta2;
    s.omb1 = float(1.0 - b1);
    s.omb2 = float(1.0 - b2);
    s.decay = float(1.0 - lr * wd);
    s.step_size = 0.0f;
    s.bc2_sqrt = 0.0f;
    s.eps = c.eps;
    s.scale = c.grad_scale;
    return s;
}

// All the scalars of step t (host).
inline Scalars scalars_for(const dopt_adam_cfg &c, int64_t t) {
    Scalars s = scalars_for_fixed(c);
    s.step_size = step_size_host(c, t);
    s.bc2_sqrt = bc2_sqrt_host(c, t);
    return s;
}

// Device view of dopt_step_counter.  The step kernel reads the 16 bytes of
// `hot` (the two scalars that depend on the step number and a copy of the
// status) with one load per warp; everything else it takes from its launch
// arguments.
struct CounterHot {
    float step_size;
    float bc2_sqrt;
    int32_t status;
    int32_t unused;
};
struct CounterBlock {
    int64_t next_step;
    int32_t status;
    int32_t reserved;
    CounterHot hot;
    uint32_t exact_steps;      // steps whose scalars took the exact evaluation
    uint32_t undecided_steps;  // steps where even that left the float open
    uint32_t unused[6];
};
static_assert(sizeof(CounterBlock) == sizeof(dopt_step_counter), "counter layout");
static_assert(offsetof(CounterBlock, hot) % 16 == 0, "one 16-byte load");
static_assert(offsetof(CounterBlock, exact_steps) == offsetof(dopt_step_counter, exact_steps) &&
                  offsetof(CounterBlock, undecided_steps) ==
                      offsetof(dopt_step_counter, undecided_steps),
              "counter layout");
constexpr int64_t kMaxCountedStep = int64_t(1) << 62;

// The part of the run table one launch covers: runs [run_begin, run_limit)
// and tiles from tile0 on.  Elements outside those runs are left alone.
struct RunView {
    const int64_t *run_start;
    const int64_t *run_end;
    const int32_t *run_meta;
    const int32_t *tile_run;
    int64_t numel;
    int64_t tile0;
    int64_t lo, hi;  // [start of the first run, end of the last run) of the view
    int32_t run_begin;
    int32_t run_limit;
};

// What the step kernel does with the reduced grads.
enum StepMode : int {
    kPlain = 0,       // reduce the replicas, Adam
    kFromMain = 1,    // read main_grad_in times the clipping coefficient, Adam
    kWriteGrads = 2,  // reduce the replicas, write the reduced grads back into
                      // every replica (all-reduce), Adam
    kCounted = 3,     // as kPlain, with the scalars from a CounterBlock
};

struct StepArgs {
    const void *grads[DOPT_MAX_D];
    void *params[DOPT_MAX_D];
    float *master;
    float *exp_avg;
    float *exp_avg_sq;
    float *main_grad_out;
    const float *main_grad_in;  // kFromMain: the reduced grads
    const float *clip_coef;     // kFromMain: device scalar
    const CounterBlock *counter;  // kCounted, and kFromMain when not NULL: status and
                                  // t-dependent scalars
    RunView rv;
    int32_t D;
    int32_t R;  // ranks per instance (D with one instance)
    int32_t gather;
    int32_t round_grad;  // round the reduced grad to the grad type first
    int32_t skip_nonfinite;  // kFromMain: a NaN coefficient means store nothing
    int32_t param_f16;       // the param replicas hold fp16 (else bf16)
    Scalars sc;
};

// Workspace of the clipped step (device memory, DOPT_CLIP_WORKSPACE_BYTES).
// The norm pass adds its per-CTA partials exactly: every partial (a
// non-negative double, a multiple of 2^-149 because every square is an fp32
// product, or an fp64 one of a sum of 2^120 or more) is split into 32-bit
// digits of a fixed-point number whose lowest
// bit weighs 2^-149, and each digit is added to a 64-bit word with an
// integer atomic.  Integer sums do not depend on their order, so the norm
// is the same at every call whatever the grid and the order in which CTAs
// finish, and it is the exact sum of the partials rounded once.  kAccWords
// digits reach 2^(32 * kAccWords - 149) = 2^299, beyond any finite sum of
// fp32 squares of up to 2^40 elements; each word takes at most one digit
// (< 2^32) per CTA, so it cannot overflow before 2^32 CTAs.  kAccCopies
// copies, chosen by CTA index, spread the atomics over more addresses; the
// finalize kernel adds them.
constexpr int kAccWords = 14;
constexpr int kAccLsb = -149;
constexpr int kAccCopies = 16;

struct ClipWorkspace {
    unsigned int special;          // 1: some partial was +Inf, 2: NaN; zeroed before every launch
    unsigned int pad0;
    unsigned long long nonfinite;  // non-finite reduced grads; zeroed likewise
    double norm_sq;
    float norm;
    float coef;
    unsigned char pad1[32];
    unsigned long long acc[kAccCopies][kAccWords];  // zeroed likewise
};
static_assert(offsetof(ClipWorkspace, acc) == 64, "workspace header");
static_assert(sizeof(dopt_clip_report) == 16, "report layout");
static_assert(sizeof(ClipWorkspace) <= DOPT_CLIP_WORKSPACE_BYTES, "workspace size");
static_assert(sizeof(ClipWorkspace) <= DOPT_NOALLOC_SCRATCH_BYTES, "scratch size");

struct NormArgs {
    const void *grads[DOPT_MAX_D];
    float *main_grad;
    ClipWorkspace *ws;
    float *norm_out;
    RunView rv;
    int64_t n_tiles;
    int32_t D;
    int32_t R;
    int32_t round_grad;
    int32_t skip_nonfinite;  // report a NaN coefficient (skip) if any grad is Inf/NaN
    float scale;
    CounterBlock *counter;   // the counted clipped step: a skipped step gives its number back
    float max_norm;
};

struct GatherArgs {
    void *params[DOPT_MAX_D];
    RunView rv;
    int32_t D;
    int32_t R;
};

// The grads are read, reduced and written back in place (each element by
// the one thread that read it), so the pointers are stored as const and
// cast back for the stores.
struct AllReduceArgs {
    const void *grads[DOPT_MAX_D];
    RunView rv;
    int32_t D;
    int32_t R;
    float scale;
};

// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ void unpack_bf16x8(const uint4 &raw, float (&f)[8]) {
    f[0] = bf16_lo(raw.x);
    f[1] = bf16_hi(raw.x);
    f[2] = bf16_lo(raw.y);
    f[3] = bf16_hi(raw.y);
    f[4] = bf16_lo(raw.z);
    f[5] = bf16_hi(raw.z);
    f[6] = bf16_lo(raw.w);
    f[7] = bf16_hi(raw.w);
}

// Two floats to two bf16 (round to nearest even), element 0 in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
}

// IEEE fp16: conversions to and from fp32 (round to nearest even, Inf on
// overflow; widening is exact).
__device__ __forceinline__ uint16_t to_f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }
__device__ __forceinline__ float f16_to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ void unpack_f16x8(const uint4 &raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 p = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
        f[2 * k] = p.x;
        f[2 * k + 1] = p.y;
    }
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack_f16x8(const float (&f)[8]) {
    return make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                      pack_f16x2(f[6], f[7]));
}

// A reduced grad in the grad buffer's type: bf16 and fp16 round to nearest
// even, fp32 is already in its type.
template <typename G>
__device__ __forceinline__ float to_grad_type(float g) {
    if constexpr (std::is_same_v<G, __nv_bfloat16>)
        return __uint_as_float(uint32_t(to_bf16_bits(g)) << 16);
    else if constexpr (std::is_same_v<G, __half>)
        return f16_to_float(to_f16_bits(g));
    else
        return g;
}

template <typename G>
__device__ __forceinline__ void to_grad_type8(float (&acc)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = to_grad_type<G>(acc[k]);
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}
__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream_f4(float *p, const float4 &v) {
    __stcs(reinterpret_cast<float4 *>(p), v);
}

// The two scalars that depend on the step number, passed apart from the
// others: the counted step takes them from its counter and every other
// scalar from the constant bank, like the other steps.
struct StepDep {
    float step_size;
    float bc2_sqrt;
};

// One AdamW update of one element, each operation rounded on its own.
__device__ __forceinline__ void adamw(const Scalars &s, StepDep dep, float decay, float g,
                                      float &w, float &m, float &v) {
    m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    const float gg = __fmul_rn(g, g);
    v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, gg));
    w = __fmul_rn(w, decay);
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), dep.bc2_sqrt), s.eps);
    w = __fsub_rn(w, __fmul_rn(dep.step_size, __fdiv_rn(m, denom)));
}

// First run (index >= j, < limit) whose end lies beyond `pos`: one ballot
// over 32 consecutive run ends per iteration.  All 32 lanes must call it.
__device__ __forceinline__ int warp_first_run(const int64_t *run_end, int limit, int j,
                                              int64_t pos, int lane) {
    for (;;) {
        const int idx = j + lane;
        const bool ended = idx < limit && run_end[idx] <= pos;
        const unsigned mask = __ballot_sync(0xffffffffu, ended);
        j += __popc(mask);
        if (mask != 0xffffffffu) return j;
    }
}

// Where a thread's 8-element vector at e0 of `tile` stands in the view:
// kNone (nothing of the view in it), kFull (inside one run) or kMixed; `j`
// is the first run of the view ending after e0.  All lanes must call it.
enum VecKind : int { kNone = 0, kFull = 1, kMixed = 2 };

__device__ __forceinline__ VecKind locate(const RunView &v, int64_t tile, int64_t e0, int &j) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_begin = tile * kDoptTileElems + int64_t(threadIdx.x & ~31) * kVec;
    j = warp_first_run(v.run_end, v.run_limit, max(v.tile_run[tile], v.run_begin), warp_begin,
                       lane);
    if (e0 >= v.numel) return kNone;
    while (j < v.run_limit && v.run_end[j] <= e0) ++j;
    if (j >= v.run_limit) return kNone;
    const int64_t rs = v.run_start[j];
    if (rs >= e0 + kVec) return kNone;
    return (rs <= e0 && e0 + kVec <= v.run_end[j]) ? kFull : kMixed;
}

// For the element path: advance j to the run holding e; false if e is not
// owned in the view (padding, or outside its runs).  Sets `done` once no
// run of the view is left.
__device__ __forceinline__ bool owned_at(const RunView &v, int64_t e, int &j, bool &done) {
    if (e >= v.numel) {
        done = true;
        return false;
    }
    while (j < v.run_limit && v.run_end[j] <= e) ++j;
    if (j >= v.run_limit) {
        done = true;
        return false;
    }
    return v.run_start[j] <= e;
}

// Device-side checks, compiled in only with DOPT_DEVICE_CHECKS (a separate
// build of the library for testing): before a vector or element access each
// kernel checks the index against the buffer (every buffer of a launch is
// padded_numel long) and the vector's alignment; a failed check records its
// kind and the first bad index and skips the access.  In the product build
// both checks are constant true.
#ifdef DOPT_DEVICE_CHECKS
__device__ unsigned int g_check_flags;              // DOPT_CHECK_* bits
__device__ unsigned long long g_check_first = ~0ull;  // first bad index, ~0 if none

__device__ __noinline__ void record_check(unsigned int flag, int64_t index) {
    atomicOr(&g_check_flags, flag);
    atomicCAS(&g_check_first, ~0ull, static_cast<unsigned long long>(index));
}
#endif

__device__ __forceinline__ bool vector_in_buffer(const RunView &v, int64_t e0) {
#ifdef DOPT_DEVICE_CHECKS
    if (e0 < 0 || e0 + kVec > v.numel) {
        record_check(DOPT_CHECK_INDEX, e0);
        return false;
    }
    if (e0 % kVec != 0) {
        record_check(DOPT_CHECK_ALIGN, e0);
        return false;
    }
#endif
    return true;
}

__device__ __forceinline__ bool element_in_buffer(const RunView &v, int64_t e) {
#ifdef DOPT_DEVICE_CHECKS
    if (e < 0 || e >= v.numel) {
        record_check(DOPT_CHECK_INDEX, e);
        return false;
    }
#endif
    return true;
}

// The vectors of a warp that straddle a run edge (padding, another decay
// flag or owner in them), shared out over the warp's lanes: `mixed` holds
// the lanes whose vector straddles (the same in every lane, so every lane
// must call this); in each round the four octets of lanes take one such
// vector each, one element per lane, and f(e, run meta) runs for each owned
// element.  (One lane per vector, element after element with each
// element's loads waited on in turn, the step of a 1000-element layout took
// 11.3 us a step against 6.4 us.)  The warp's first run is looked up again
// here so that the vector path keeps no run index alive.
template <typename F>
__device__ __forceinline__ void for_straddling_elements(const RunView &v, int64_t tile, unsigned mixed,
                                                        F &&f) {
    const int lane = threadIdx.x & 31;
    const int octet = lane >> 3;
    const int64_t warp_e0 = tile * kDoptTileElems + int64_t(threadIdx.x & ~31) * kVec;
    const int jw = warp_first_run(v.run_end, v.run_limit, max(v.tile_run[tile], v.run_begin), warp_e0, lane);
    while (mixed != 0) {
        unsigned mine = mixed;  // this octet's vector: the octet-th lane left in `mixed`
        for (int s = 0; s < octet && mine != 0; ++s) mine &= mine - 1;
        for (int s = 0; s < 4 && mixed != 0; ++s) mixed &= mixed - 1;
        if (mine == 0) continue;
        const int64_t e = warp_e0 + int64_t(__ffs(mine) - 1) * kVec + (lane & 7);
        int j = jw;
        bool done = false;
        if (owned_at(v, e, j, done) && element_in_buffer(v, e)) f(e, v.run_meta[j]);
    }
}

template <typename G>
__device__ __forceinline__ float load_grad_scalar(const void *base, int64_t i) {
    if constexpr (std::is_same_v<G, __nv_bfloat16>)
        return __uint_as_float(uint32_t(__ldcs(static_cast<const unsigned short *>(base) + i)) << 16);
    else if constexpr (std::is_same_v<G, __half>)
        return f16_to_float(__ldcs(static_cast<const unsigned short *>(base) + i));
    else
        return __ldcs(static_cast<const float *>(base) + i);
}

template <typename G>
__device__ __forceinline__ void store_grad_scalar(const void *base, int64_t i, float g) {
    if constexpr (std::is_same_v<G, __nv_bfloat16>)
        static_cast<uint16_t *>(const_cast<void *>(base))[i] = to_bf16_bits(g);
    else if constexpr (std::is_same_v<G, __half>)
        static_cast<uint16_t *>(const_cast<void *>(base))[i] = to_f16_bits(g);
    else
        static_cast<float *>(const_cast<void *>(base))[i] = g;
}

// Load the 8 grads of replica r at e0 (16-bit types: one 16-byte load; fp32:
// two).
template <typename G>
struct GradVec;

template <>
struct GradVec<__half> {
    uint4 a;
    __device__ __forceinline__ void load(const void *base, int64_t e0) {
        a = ld_stream(static_cast<const __half *>(base) + e0);
    }
    __device__ __forceinline__ void get(float (&f)[8]) const { unpack_f16x8(a, f); }
    __device__ __forceinline__ static void store(const void *base, int64_t e0, const float (&f)[8]) {
        st_stream(static_cast<__half *>(const_cast<void *>(base)) + e0, pack_f16x8(f));
    }
};

template <>
struct GradVec<__nv_bfloat16> {
    uint4 a;
    __device__ __forceinline__ void load(const void *base, int64_t e0) {
        a = ld_stream(static_cast<const __nv_bfloat16 *>(base) + e0);
    }
    __device__ __forceinline__ void get(float (&f)[8]) const { unpack_bf16x8(a, f); }
    // the 8 reduced grads, rounded to bf16, into replica `base` at e0
    __device__ __forceinline__ static void store(const void *base, int64_t e0, const float (&f)[8]) {
        st_stream(static_cast<__nv_bfloat16 *>(const_cast<void *>(base)) + e0, pack_bf16x8(f));
    }
};

template <>
struct GradVec<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const void *base, int64_t e0) {
        const float *p = static_cast<const float *>(base) + e0;
        a = ld_stream_f4(p);
        b = ld_stream_f4(p + 4);
    }
    __device__ __forceinline__ void get(float (&f)[8]) const {
        f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w;
        f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
    }
    __device__ __forceinline__ static void store(const void *base, int64_t e0, const float (&f)[8]) {
        float *p = static_cast<float *>(const_cast<void *>(base)) + e0;
        st_stream_f4(p, make_float4(f[0], f[1], f[2], f[3]));
        st_stream_f4(p + 4, make_float4(f[4], f[5], f[6], f[7]));
    }
};

// The compile-time-D reduction of 8 elements from replicas already loaded:
// the rank-order sum (one instance, GR = DC), or each group of GR
// consecutive replicas in rank order and then the groups' sums in group
// order (DC / GR instances).  The group size is a template argument so that
// the grouped sum unrolls into the same straight-line code as the plain one.
// (With the group size read at run time, the branch at each group's end
// kept the state loads behind the whole reduction: 1.3 % slower at D = 8 as
// 2 instances and 8 % at D = 2 as 2.)
template <typename G, int DC, int GR>
__device__ __forceinline__ void reduce_loaded(const GradVec<G> (&g)[DC], float scale, float (&acc)[8]) {
    static_assert(GR > 0 && DC % GR == 0, "the group size divides the replica count");
    if constexpr (GR == DC) {
#pragma unroll
        for (int r = 0; r < DC; ++r) {
            float f[8];
            g[r].get(f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float x = __fmul_rn(scale, f[k]);
                acc[k] = r == 0 ? x : __fadd_rn(acc[k], x);
            }
        }
    } else {
        float part[8];
#pragma unroll
        for (int r = 0; r < DC; ++r) {
            float f[8];
            g[r].get(f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float x = __fmul_rn(scale, f[k]);
                part[k] = r % GR == 0 ? x : __fadd_rn(part[k], x);
                if (r % GR == GR - 1) acc[k] = r == GR - 1 ? part[k] : __fadd_rn(acc[k], part[k]);
            }
        }
    }
}

// Scaled rank-order fp32 reduction of 8 elements over the D replicas.  The
// compile-time-D form loads every replica first (one instance, or groups of
// GR); the run-time form loads 4 replicas at a time and reduces each
// group of R consecutive replicas in rank order, adding the groups' sums in
// group order (several optimizer instances; with R = D the last group's sum
// is copied, so the result is the plain rank-order sum).
template <typename G, int DC, int GR = DC, typename Args>
__device__ __forceinline__ void reduce_vec(const Args &a, float scale, int64_t e0,
                                           float (&acc)[8]) {
    if constexpr (DC > 0) {
        GradVec<G> g[DC];
#pragma unroll
        for (int r = 0; r < DC; ++r) g[r].load(a.grads[r], e0);
        reduce_loaded<G, DC, GR>(g, scale, acc);
    } else {
        constexpr int kBatch = 4;
        float part[8];
        int in_group = 0;  // position of the next replica inside its group
        for (int r0 = 0; r0 < a.D; r0 += kBatch) {
            GradVec<G> g[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (r0 + u < a.D) g[u].load(a.grads[r0 + u], e0);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int r = r0 + u;
                if (r >= a.D) break;
                float f[8];
                g[u].get(f);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float x = __fmul_rn(scale, f[k]);
                    part[k] = in_group == 0 ? x : __fadd_rn(part[k], x);
                }
                if (++in_group == a.R) {
                    in_group = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        acc[k] = r + 1 == a.R ? part[k] : __fadd_rn(acc[k], part[k]);
                }
            }
        }
    }
}

// The same reduction for one element: groups of R replicas in rank order,
// then the groups' sums in group order.
template <typename G>
__device__ __forceinline__ float reduce_scalar(const void *const *grads, int D, int R,
                                               float scale, int64_t e) {
    float g = 0.0f, part = 0.0f;
    for (int r = 0; r < D; ++r) {
        const float x = __fmul_rn(scale, load_grad_scalar<G>(grads[r], e));
        const int in_group = r % R;
        part = in_group == 0 ? x : __fadd_rn(part, x);
        if (in_group == R - 1) g = r + 1 == R ? part : __fadd_rn(g, part);
    }
    return g;
}

// The reduced grads of 8 elements written into every replica, rounded to
// the grad type (the all-reduce's all-gather half).
template <typename G, int DC>
__device__ __forceinline__ void write_grads_vec(const void *const *grads, int D_rt, int64_t e0,
                                                const float (&acc)[8]) {
    if constexpr (DC > 0) {
#pragma unroll
        for (int r = 0; r < DC; ++r) GradVec<G>::store(grads[r], e0, acc);
    } else {
        for (int r = 0; r < D_rt; ++r) GradVec<G>::store(grads[r], e0, acc);
    }
}

// ---------------------------------------------------------------------------
// The step kernel
// ---------------------------------------------------------------------------

// The Adam update of a vector of 8 owned elements of one run and all its
// stores, from its reduced grads and its loaded master/m/v.
template <typename G, int DC, int MODE>
__device__ __forceinline__ void update_and_store(const StepArgs &a, const Scalars &sc, StepDep dep,
                                                 int64_t e0,
                                                 int32_t meta, int32_t status, float (&acc)[8],
                                                 const float4 &w0, const float4 &w1,
                                                 const float4 &m0, const float4 &m1,
                                                 const float4 &v0, const float4 &v1) {
    float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const float decay = (meta & kRunDecays) ? sc.decay : 1.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) adamw(sc, dep, decay, acc[k], w[k], m[k], v[k]);
    if constexpr (MODE == kCounted || MODE == kFromMain) {
        if (status != 0) return;  // the counter launch found a bad step number
    }

    st_stream_f4(a.master + e0, make_float4(w[0], w[1], w[2], w[3]));
    st_stream_f4(a.master + e0 + 4, make_float4(w[4], w[5], w[6], w[7]));
    st_stream_f4(a.exp_avg + e0, make_float4(m[0], m[1], m[2], m[3]));
    st_stream_f4(a.exp_avg + e0 + 4, make_float4(m[4], m[5], m[6], m[7]));
    st_stream_f4(a.exp_avg_sq + e0, make_float4(v[0], v[1], v[2], v[3]));
    st_stream_f4(a.exp_avg_sq + e0 + 4, make_float4(v[4], v[5], v[6], v[7]));
    if (MODE != kFromMain && a.main_grad_out) {
        st_stream_f4(a.main_grad_out + e0, make_float4(acc[0], acc[1], acc[2], acc[3]));
        st_stream_f4(a.main_grad_out + e0 + 4, make_float4(acc[4], acc[5], acc[6], acc[7]));
    }

    const uint4 packed = a.param_f16 ? pack_f16x8(w) : pack_bf16x8(w);
    if (a.gather) {
        if constexpr (DC > 0) {
#pragma unroll
            for (int r = 0; r < DC; ++r)
                st_stream(static_cast<__nv_bfloat16 *>(a.params[r]) + e0, packed);
        } else {
            for (int r = 0; r < a.D; ++r)
                st_stream(static_cast<__nv_bfloat16 *>(a.params[r]) + e0, packed);
        }
    } else {
        const int q = meta >> kRunRankShift;
        for (int r = q; r < a.D; r += a.R)
            st_stream(static_cast<__nv_bfloat16 *>(a.params[r]) + e0, packed);
    }
}

// A vector of 8 owned elements of one run, loading as it goes.
template <typename G, int DC, int MODE, int GR>
__device__ __forceinline__ void full_vector(const StepArgs &a, const Scalars &sc, StepDep dep, int64_t e0,
                                            int32_t meta, int32_t status = 0) {
    static_assert(MODE != kFromMain, "the clipped step's vectors are done in step_vector");
    float acc[8];
    reduce_vec<G, DC, GR>(a, sc.scale, e0, acc);
    if (a.round_grad) to_grad_type8<G>(acc);
    if constexpr (MODE == kWriteGrads) write_grads_vec<G, DC>(a.grads, a.D, e0, acc);
    const float4 w0 = ld_stream_f4(a.master + e0), w1 = ld_stream_f4(a.master + e0 + 4);
    const float4 m0 = ld_stream_f4(a.exp_avg + e0), m1 = ld_stream_f4(a.exp_avg + e0 + 4);
    const float4 v0 = ld_stream_f4(a.exp_avg_sq + e0), v1 = ld_stream_f4(a.exp_avg_sq + e0 + 4);
    update_and_store<G, DC, MODE>(a, sc, dep, e0, meta, status, acc, w0, w1, m0, m1, v0, v1);
}

// The loads of a vector issued before the thread knows whether it is a
// whole vector of one run (its run lookup is a chain of dependent loads): the
// D grad replicas and master/m/v at e0, all inside the launch's own range.
template <typename G, int DC>
struct Preloaded {
    GradVec<G> g[DC];
    float4 w0, w1, m0, m1, v0, v1;
    __device__ __forceinline__ void load(const StepArgs &a, int64_t e0) {
#pragma unroll
        for (int r = 0; r < DC; ++r) g[r].load(a.grads[r], e0);
        w0 = ld_stream_f4(a.master + e0), w1 = ld_stream_f4(a.master + e0 + 4);
        m0 = ld_stream_f4(a.exp_avg + e0), m1 = ld_stream_f4(a.exp_avg + e0 + 4);
        v0 = ld_stream_f4(a.exp_avg_sq + e0), v1 = ld_stream_f4(a.exp_avg_sq + e0 + 4);
    }
};

// Which instantiations preload: D = 1 with 16-bit grads, where it made the
// 256 Mi sweep's step 1.8 % faster.  With more replicas enough other warps
// cover the lookup, and holding the preloaded vectors across it cost 0.5 %
// (D = 2) to 4.7 % (D = 8, 1 Mi buckets); they load as they go.
template <typename G, int DC, int MODE>
constexpr bool kPreload = DC == 1 && sizeof(G) == 2 && MODE != kFromMain;

// A whole vector of one run from its preloaded grads and state.
template <typename G, int DC, int MODE>
__device__ __forceinline__ void full_vector_preloaded(const StepArgs &a, const Scalars &sc, StepDep dep,
                                                      int64_t e0, int32_t meta, int32_t status,
                                                      const Preloaded<G, DC> &p) {
    float acc[8];
    reduce_loaded<G, DC, DC>(p.g, sc.scale, acc);
    if (a.round_grad) to_grad_type8<G>(acc);
    if constexpr (MODE == kWriteGrads) write_grads_vec<G, DC>(a.grads, a.D, e0, acc);
    update_and_store<G, DC, MODE>(a, sc, dep, e0, meta, status, acc, p.w0, p.w1, p.m0, p.m1,
                                  p.v0, p.v1);
}

// The step of the warp's vectors that straddle a run edge, element by
// element over the warp's lanes (for_straddling_elements).
template <typename G, int DC, int MODE>
__device__ __noinline__ void mixed_elements(const StepArgs &a, const Scalars &sc, StepDep dep,
                                            unsigned mixed, int64_t tile) {
    if constexpr (MODE == kFromMain) {
        if (a.skip_nonfinite && isnan(*a.clip_coef)) return;  // the step is skipped
    }
    const int D = DC > 0 ? DC : a.D;
    for_straddling_elements(a.rv, tile, mixed, [&](int64_t e, int32_t meta) {
        float g;
        if constexpr (MODE == kFromMain) {
            g = __fmul_rn(a.main_grad_in[e], *a.clip_coef);
        } else {
            g = reduce_scalar<G>(a.grads, D, a.R, sc.scale, e);
            if (a.round_grad) g = to_grad_type<G>(g);
        }
        if constexpr (MODE == kWriteGrads)
            for (int r = 0; r < D; ++r) store_grad_scalar<G>(a.grads[r], e, g);
        float w = a.master[e], m = a.exp_avg[e], v = a.exp_avg_sq[e];
        adamw(sc, dep, (meta & kRunDecays) ? sc.decay : 1.0f, g, w, m, v);
        a.master[e] = w;
        a.exp_avg[e] = m;
        a.exp_avg_sq[e] = v;
        if (MODE != kFromMain && a.main_grad_out) a.main_grad_out[e] = g;
        const uint16_t bits = a.param_f16 ? to_f16_bits(w) : to_bf16_bits(w);
        if (a.gather) {
            for (int r = 0; r < D; ++r) static_cast<uint16_t *>(a.params[r])[e] = bits;
        } else {
            for (int r = meta >> kRunRankShift; r < D; r += a.R)
                static_cast<uint16_t *>(a.params[r])[e] = bits;
        }
    });
}

// At least 3 CTAs per SM: this lets ptxas use up to 85 registers where it
// would otherwise stop near 56-64, and the extra registers keep more loads in
// flight per thread (D = 4: 2.5 % faster, D = 8 and 16: 0.2-0.4 %; forcing 6
// or 8 CTAs per SM spilled and lost 15-40 %).
// Where the two step-dependent scalars and the status come from: the
// launch's own scalars in the constant bank (a copy of them in registers
// cost the D = 2 step 4 %), or the counter of the counted steps, read with
// one 16-byte load per warp either before anything else (the counted step,
// right after its wait for the counter kernel) or after the wait that
// follows the run lookup (the counted clipped step).  Nothing waits for the counter's load until the
// Adam arithmetic, and the status is checked only before the first store.
// (Reading the whole counter through shared memory behind a CTA barrier
// cost 1.7 %; a persistent grid that reads it once per resident CTA cost
// 15 %; the counted step reading it after its run lookup, as a programmatic
// dependent of the counter kernel, cost 0.15 % on GPT-2 small and 1.2 µs a
// step on the 1000-element layout.)
enum ScalarSource : int { kFromArgs = 0, kFromCounterAfterWait = 1, kFromCounterEarly = 2 };

template <int SRC>
__device__ __forceinline__ void step_scalars(const StepArgs &a, const Scalars &sc, const uint4 &early,
                                             StepDep &dep, int32_t &status) {
    if constexpr (SRC == kFromArgs) {
        dep = StepDep{sc.step_size, sc.bc2_sqrt};
        status = 0;
    } else {
        const uint4 hot = SRC == kFromCounterEarly ? early
                                                   : *reinterpret_cast<const uint4 *>(&a.counter->hot);
        dep = StepDep{__uint_as_float(hot.x), __uint_as_float(hot.y)};
        status = int32_t(hot.z);
    }
}

// The wait for the launch before (see dopt_step_kernel), then the scalars;
// the counted step has waited and read its scalars at its start.
template <int SRC>
__device__ __forceinline__ void wait_then_scalars(const StepArgs &a, const Scalars &sc,
                                                  const uint4 &early, StepDep &dep,
                                                  int32_t &status) {
    if constexpr (SRC != kFromCounterEarly) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        step_scalars<SRC>(a, sc, early, dep, status);
    }
}

// One tile per CTA: this thread's vector of 8 elements.  `sc` is the
// launch's own scalars (read from the constant bank); the two
// step-dependent ones come from step_scalars.
template <typename G, int DC, int MODE, int GR, int SRC>
__device__ __forceinline__ void step_vector(const StepArgs &a, const Scalars &sc, const uint4 &early) {
    const int64_t tile = a.rv.tile0 + blockIdx.x;
    const int64_t e0 = tile * kDoptTileElems + int64_t(threadIdx.x) * kVec;
    int j;
    VecKind kind;
    StepDep dep;
    int32_t status;
    if constexpr (SRC == kFromCounterEarly) step_scalars<SRC>(a, sc, early, dep, status);
    if constexpr (kPreload<G, DC, MODE>) {
        // A whole vector of one run lies inside [lo, hi), so every vector
        // that turns out whole has its loads in flight before the lookup
        // (after the wait for the kernel before: see dopt_step_kernel).
        wait_then_scalars<SRC>(a, sc, early, dep, status);
        Preloaded<G, DC> p;
        const bool inside = e0 >= a.rv.lo && e0 + kVec <= a.rv.hi && vector_in_buffer(a.rv, e0);
        if (inside) p.load(a, e0);
        kind = locate(a.rv, tile, e0, j);
        if (kind == kFull && vector_in_buffer(a.rv, e0))
            full_vector_preloaded<G, DC, MODE>(a, sc, dep, e0, a.rv.run_meta[j], status, p);
    } else if constexpr (MODE == kFromMain) {
        // The second launch of the clipped step starts (programmatic
        // dependent launch) while the norm pass finishes: the run lookup and
        // the master/m/v loads, which do not depend on that pass, go first;
        // the main grads and the coefficient are read after the wait for
        // the norm pass to complete.
        kind = locate(a.rv, tile, e0, j);
        const bool full = kind == kFull && vector_in_buffer(a.rv, e0);
        float4 w0, w1, m0, m1, v0, v1;
        if (full) {
            w0 = ld_stream_f4(a.master + e0), w1 = ld_stream_f4(a.master + e0 + 4);
            m0 = ld_stream_f4(a.exp_avg + e0), m1 = ld_stream_f4(a.exp_avg + e0 + 4);
            v0 = ld_stream_f4(a.exp_avg_sq + e0), v1 = ld_stream_f4(a.exp_avg_sq + e0 + 4);
        }
        wait_then_scalars<SRC>(a, sc, early, dep, status);
        if (full) {
            const float coef = *a.clip_coef;
            if (!(a.skip_nonfinite && isnan(coef))) {  // else the step is skipped
                const float4 g0 = ld_stream_f4(a.main_grad_in + e0);
                const float4 g1 = ld_stream_f4(a.main_grad_in + e0 + 4);
                float acc[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] = __fmul_rn(acc[k], coef);
                update_and_store<G, DC, MODE>(a, sc, dep, e0, a.rv.run_meta[j], status, acc, w0, w1,
                                              m0, m1, v0, v1);
            }
        }
    } else {
        kind = locate(a.rv, tile, e0, j);
        // the run lookup reads only the layout's tables; grads and state
        // may still be written by the kernel before (see dopt_step_kernel)
        wait_then_scalars<SRC>(a, sc, early, dep, status);
        if (kind == kFull && vector_in_buffer(a.rv, e0))
            full_vector<G, DC, MODE, GR>(a, sc, dep, e0, a.rv.run_meta[j], status);
    }
    // every lane of the warp is here (no lane returns before this point)
    const unsigned mixed = __ballot_sync(0xffffffffu, kind == kMixed);
    if (mixed != 0 && status == 0) mixed_elements<G, DC, MODE>(a, sc, dep, mixed, tile);
}

// GR: the replicas of one optimizer instance (GR = DC: one instance).
//
// Every step kernel is launched as a programmatic dependent of the kernel
// before it on the stream, and lets its own dependent start as soon as all
// of its CTAs run: the next launch's first CTAs take the SMs that this
// grid's last wave leaves, look up their runs, and wait
// (griddepcontrol.wait: the grid before has completed and its writes are
// visible) before they read grads or state or store anything.  The counted
// step waits at its very start, before its run lookup: its counter kernel
// lets it start only once the step before has completed, and reading the
// counter after the lookup was slower.  Where the kernel before does not
// let its dependents start early, the wait returns at once and nothing
// changes.
//
// CTAs per SM that the kernel's registers must allow: 3 (at most 85
// registers), but 4 (64 registers, no spills) for the plain and counted
// steps with D = 4 and 16-bit grads, which run 2-5 % faster with the fourth
// CTA than with the 67-71 registers they take when allowed 3, and 5 (48
// registers; 32 bytes spilled) for the plain step with D = 1 and 16-bit
// grads: 0.6-1.7 % faster than 4 CTAs of 50 registers.  Measured slower:
// 4 CTAs at D = 8 (0.2-0.4 %), 4 with fp32 grads at D = 4 and 8 (0.4-12 %,
// spills), 5 for the counted D = 1 step (6 %, 76 bytes spilled).
template <typename G, int DC, int MODE>
constexpr int step_min_ctas() {
    if (sizeof(G) != 2) return 3;
    if (DC == 1 && MODE == kPlain) return 5;
    if (DC == 4 && (MODE == kPlain || MODE == kCounted)) return 4;
    return 3;
}

template <typename G, int DC, int MODE, int GR = DC>
__global__ void __launch_bounds__(kThreads, step_min_ctas<G, DC, MODE>())
    dopt_step_kernel(const __grid_constant__ StepArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint4 none = make_uint4(0, 0, 0, 0);
    if constexpr (MODE == kCounted) {
        // the counter kernel before it wrote the counter: wait for it first
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const uint4 hot = *reinterpret_cast<const uint4 *>(&a.counter->hot);
        step_vector<G, DC, MODE, GR, kFromCounterEarly>(a, a.sc, hot);
    } else if constexpr (MODE == kFromMain) {
        if (a.counter != nullptr)  // the counted clipped step
            step_vector<G, DC, MODE, GR, kFromCounterAfterWait>(a, a.sc, none);
        else
            step_vector<G, DC, MODE, GR, kFromArgs>(a, a.sc, none);
    } else {
        step_vector<G, DC, MODE, GR, kFromArgs>(a, a.sc, none);
    }
}

// ---------------------------------------------------------------------------
// The staged step kernel: each tile's grads and state moved into shared
// memory by bulk copies first (DOPT_STEP_STAGE)
// ---------------------------------------------------------------------------
//
// The same step as dopt_step_kernel (one-instance layouts, D in {1, 2, 4, 8,
// 16}, plain or counted), with a different way of reading: one thread of the
// CTA issues one 1-D bulk copy (cp.async.bulk, the TMA unit of the SM,
// global -> this CTA's shared memory, no cluster multicast) per grad replica
// and per state array for the tile's whole vectors, completing on an
// mbarrier, while the CTA looks up its runs; the threads then read their
// vectors from shared memory.  Stores go to global memory as in the plain
// kernel.  The plain kernel loads with 128-bit vector loads straight into
// registers; this one exists to measure the other design.

// Bulk-copy waits that ran past their time limit (the TMA unit never
// completed them); the CTA then skipped its tile.  Read by
// dopt_stage_timeouts.
__device__ unsigned int g_stage_timeouts;

constexpr unsigned long long kStageWaitNs = 2000000000ull;  // 2 s

#ifdef DOPT_DEVICE_CHECKS
// Test build only: bytes added to every staged CTA's expected transaction
// count that no copy delivers, so that its bounded wait runs out and the
// failure path runs without any fault (dopt_stage_wait_test).
__device__ unsigned int g_stage_phantom_bytes;
__device__ __forceinline__ uint32_t stage_phantom_bytes() { return g_stage_phantom_bytes; }
#else
__device__ __forceinline__ uint32_t stage_phantom_bytes() { return 0u; }
#endif

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Wait for phase `parity` of the mbarrier at `bar` for at most kStageWaitNs;
// false if the time ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (globaltimer_ns() - t0 > kStageWaitNs) return false;
    }
}

// One 1-D bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global memory into this CTA's shared memory, completing on
// the mbarrier at `bar`.
__device__ __forceinline__ void bulk_to_shared(uint32_t dst, const void *src, uint32_t bytes,
                                               uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :
        : "r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Shared-memory bytes of one staged tile: DC grad chunks and master/m/v.
template <typename G, int DC>
__host__ __device__ constexpr size_t staged_smem_bytes() {
    return size_t(DC) * kDoptTileElems * sizeof(G) + 3 * kDoptTileElems * sizeof(float);
}

template <typename G>
__device__ __forceinline__ void load_grad_shared(GradVec<G> &g, const unsigned char *p) {
    if constexpr (sizeof(G) == 2) {
        g.a = *reinterpret_cast<const uint4 *>(p);
    } else {
        g.a = *reinterpret_cast<const float4 *>(p);
        g.b = *reinterpret_cast<const float4 *>(p + 16);
    }
}

template <typename G, int DC, int MODE>
__device__ __forceinline__ void staged_tile(const StepArgs &a, const Scalars &sc, StepDep dep,
                                            int32_t status, unsigned char *stage,
                                            unsigned long long *bar_ptr) {
    constexpr int64_t kGradChunk = kDoptTileElems * int64_t(sizeof(G));
    const int64_t tile = a.rv.tile0 + blockIdx.x;
    const int64_t base = tile * kDoptTileElems;
    const int64_t e0 = base + int64_t(threadIdx.x) * kVec;
    // every whole vector of a run lies in [lo, hi) of the view: stage the
    // tile's part of that span, cut to whole vectors (so that sizes and
    // addresses are multiples of 16 bytes)
    const int64_t s0 = max(base, a.rv.lo & ~int64_t(kVec - 1));
    const int64_t s1 = min(base + kDoptTileElems, a.rv.hi & ~int64_t(kVec - 1));
    const int64_t n = s1 - s0;
    const uint32_t bar = smem_addr(bar_ptr);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && n > 0) {
        const uint32_t gbytes = uint32_t(n * int64_t(sizeof(G)));
        const uint32_t sbytes = uint32_t(n * 4);
        const uint32_t total = uint32_t(DC) * gbytes + 3 * sbytes + stage_phantom_bytes();
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(total)
                     : "memory");
        const uint32_t sm = smem_addr(stage);
        const int64_t goff = (s0 - base) * int64_t(sizeof(G)), soff = (s0 - base) * 4;
#pragma unroll
        for (int r = 0; r < DC; ++r)
            bulk_to_shared(sm + uint32_t(r * kGradChunk + goff),
                           static_cast<const G *>(a.grads[r]) + s0, gbytes, bar);
        const uint32_t st = sm + uint32_t(DC * kGradChunk);
        bulk_to_shared(st + uint32_t(soff), a.master + s0, sbytes, bar);
        bulk_to_shared(st + uint32_t(kDoptTileElems * 4 + soff), a.exp_avg + s0, sbytes, bar);
        bulk_to_shared(st + uint32_t(2 * kDoptTileElems * 4 + soff), a.exp_avg_sq + s0, sbytes, bar);
    }
    int j;
    const VecKind kind = locate(a.rv, tile, e0, j);  // while the copies fly
    const bool ok = n <= 0 || mbar_wait(bar, 0);
    if (__syncthreads_or(!ok)) {
        // the bulk copies did not complete in time (for some thread: the
        // whole CTA decides together): count it, give the copies one more
        // bounded wait (they write this CTA's shared memory), and leave the
        // tile alone
        if (threadIdx.x == 0) atomicAdd(&g_stage_timeouts, 1u);
        mbar_wait(bar, 0);
        return;
    }
    if (kind == kFull && vector_in_buffer(a.rv, e0)) {
        const int64_t off = e0 - base;
        GradVec<G> g[DC];
#pragma unroll
        for (int r = 0; r < DC; ++r) load_grad_shared<G>(g[r], stage + r * kGradChunk + off * int64_t(sizeof(G)));
        float acc[8];
        reduce_loaded<G, DC, DC>(g, sc.scale, acc);
        if (a.round_grad) to_grad_type8<G>(acc);
        const float *sw = reinterpret_cast<const float *>(stage + DC * kGradChunk) + off;
        const float *smv = sw + kDoptTileElems, *svv = sw + 2 * kDoptTileElems;
        const float4 w0 = *reinterpret_cast<const float4 *>(sw), w1 = *reinterpret_cast<const float4 *>(sw + 4);
        const float4 m0 = *reinterpret_cast<const float4 *>(smv), m1 = *reinterpret_cast<const float4 *>(smv + 4);
        const float4 v0 = *reinterpret_cast<const float4 *>(svv), v1 = *reinterpret_cast<const float4 *>(svv + 4);
        update_and_store<G, DC, MODE>(a, sc, dep, e0, a.rv.run_meta[j], status, acc, w0, w1, m0, m1,
                                      v0, v1);
    }
    const unsigned mixed = __ballot_sync(0xffffffffu, kind == kMixed);
    if (mixed != 0 && status == 0) mixed_elements<G, DC, MODE>(a, sc, dep, mixed, tile);
}

template <typename G, int DC, int MODE>
__global__ void __launch_bounds__(kThreads) dopt_step_staged_kernel(const __grid_constant__ StepArgs a) {
    static_assert(MODE == kPlain || MODE == kCounted, "the staged kernel has the plain and counted modes");
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ __align__(8) unsigned long long bar;
    if constexpr (MODE == kCounted) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        const uint4 hot = *reinterpret_cast<const uint4 *>(&a.counter->hot);
        staged_tile<G, DC, MODE>(a, a.sc, StepDep{__uint_as_float(hot.x), __uint_as_float(hot.y)},
                                 int32_t(hot.z), stage, &bar);
    } else {
        staged_tile<G, DC, MODE>(a, a.sc, StepDep{a.sc.step_size, a.sc.bc2_sqrt}, 0, stage, &bar);
    }
}

// ---------------------------------------------------------------------------
// The counter kernel of the counted steps: the step number and its two
// bias-correction scalars on the device
// ---------------------------------------------------------------------------
//
// The host entry points take beta^t from the C library's pow.  The device
// reaches the same floats as follows.  beta^t by binary powering in double
// (at most 2*63 multiplies: this GPU's double pipeline is slow, and a
// general pow costs far more) is within (t - 1) * 2^-53, relative, of the
// exact power (each product rounds once; a chain of multiplications that
// makes x^t lets at most t - 1 of those roundings count), unless it
// underflows.  A correct pow is within 0.52 units in the last place of the
// exact power (the C library's documented bound).  So pow's double lies in
// [p - B, p + B] with p the powering's result and B = p * (t + 2) * 2^-52
// (plus 2^-1000 for underflow).  Both scalars are monotone in beta^t (every
// IEEE operation on the way, 1 - x, lr / x, sqrt, the rounding to float, is
// monotone), so when the two ends of that interval give the same float, it
// is pow's float.  Two lanes evaluate the two ends of each scalar side by
// side.  Only when they differ (a float rounding boundary inside the
// interval: about 2^-20 of the steps where t is small enough for the power
// to matter) does the pair compute beta^t again in double-double, whose
// error is far below an ulp, and evaluate the scalar at the smallest and at
// the largest double within 0.52 ulp of it; the counter records such steps
// (exact_steps), and the ones where those two still differ
// (undecided_steps, which then take the double nearest the double-double
// value).

// beta^t by binary powering in double.
__device__ __forceinline__ double beta_pow_fast(double b, int64_t t) {
    double r = 1.0;
    double x = b;
    while (t > 0) {
        if (t & 1) r = __dmul_rn(r, x);
        t >>= 1;
        if (t > 0) x = __dmul_rn(x, x);
    }
    return r;
}

// A double-double number hi + lo with |lo| at most half an ulp of hi.
struct DoubleDouble {
    double hi, lo;
};

// Product of two double-double numbers: the leading product's rounding
// error exactly (fused multiply-add), the cross terms rounded, renormalised
// with a fast two-sum (|p| >= |e|).  Relative error about 2^-104 unless
// something underflows.
__device__ __forceinline__ DoubleDouble dd_mul(DoubleDouble a, DoubleDouble b) {
    const double p = __dmul_rn(a.hi, b.hi);
    double e = __fma_rn(a.hi, b.hi, -p);
    e = __dadd_rn(e, __dadd_rn(__dmul_rn(a.hi, b.lo), __dmul_rn(a.lo, b.hi)));
    const double s = __dadd_rn(p, e);
    return DoubleDouble{s, __dsub_rn(e, __dsub_rn(s, p))};
}

__device__ __noinline__ DoubleDouble beta_pow_dd(double b, int64_t t) {
    DoubleDouble r{1.0, 0.0};
    DoubleDouble x{b, 0.0};
    while (t > 0) {
        if (t & 1) r = dd_mul(r, x);
        t >>= 1;
        if (t > 0) x = dd_mul(x, x);
    }
    return r;
}

// Scalar `which` (0: lr / (1 - p), 1: sqrt(1 - p)) for beta^t = p: the
// operations of the host's evaluation, each an IEEE round-to-nearest.
__device__ __forceinline__ float scalar_at(const dopt_adam_cfg &cfg, int which, double p) {
    const double d = __dsub_rn(1.0, p);
    return which == 0 ? __double2float_rn(__ddiv_rn(double(cfg.lr), d))
                      : __double2float_rn(__dsqrt_rn(d));
}

struct CountedScalar {
    float x;
    bool exact;      // the double-double evaluation ran
    bool undecided;  // and the candidates still gave two floats
};

// The exact evaluation of a lane pair (side 0: smallest candidate double,
// side 1: largest): the doubles within 0.52 ulp of beta^t, found from its
// double-double value (whose own error, at most (t + 2) * 2^-100 of it, is
// added to the margin).
__device__ __noinline__ CountedScalar counted_scalar_exact(const dopt_adam_cfg &cfg, double b,
                                                           int64_t t, int which, int side,
                                                           unsigned pair) {
    const DoubleDouble q = beta_pow_dd(b, t);
    // the larger of the two ulps around hi: a conservative margin at a
    // binade edge
    const double up = __dsub_rn(nextafter(q.hi, 2.0), q.hi);
    const double down = __dsub_rn(q.hi, nextafter(q.hi, -1.0));
    const double ulp = fmax(up, down);
    const double err = __dadd_rn(__dmul_rn(__dmul_rn(fabs(q.hi), double(t) + 2.0), 0x1p-100),
                                 0x1p-1074);
    const double margin = __dadd_rn(__dmul_rn(0.52, ulp), err);
    const double lo_off = __dsub_rn(q.lo, margin);  // candidates d: lo_off <= d - hi <= hi_off
    const double hi_off = __dadd_rn(q.lo, margin);
    double d = q.hi;
    if (side == 0) {
        for (int k = 0; k < 4; ++k) {
            const double prev = nextafter(d, -1.0);
            if (prev < 0.0 || __dsub_rn(prev, q.hi) < lo_off) break;
            d = prev;
        }
    } else {
        for (int k = 0; k < 4; ++k) {
            const double next = nextafter(d, 2.0);
            if (__dsub_rn(next, q.hi) > hi_off) break;
            d = next;
        }
    }
    CountedScalar s{scalar_at(cfg, which, d), true, false};
    const float other = __shfl_xor_sync(pair, s.x, 1);
    if (other != s.x) {
        s.undecided = true;
        s.x = scalar_at(cfg, which, q.hi);  // the double nearest the double-double value
    }
    return s;
}

// Lane l of the counter kernel's four: scalar l >> 1 (0: step size, 1:
// bc2_sqrt) of step t, the pair l, l ^ 1 evaluating the two ends of pow's
// interval.  Every lane of the four must call it with the same t.
__device__ __forceinline__ CountedScalar counted_scalar(const dopt_adam_cfg &cfg, int64_t t,
                                                        int lane) {
    if (t < 1 || t > kMaxCountedStep) return CountedScalar{0.0f, false, false};
    const int which = lane >> 1, side = lane & 1;
    const double b = which == 0 ? double(cfg.beta1) : double(cfg.beta2);
    const double p = beta_pow_fast(b, t);
    const double B = __dadd_rn(__dmul_rn(__dmul_rn(p, double(t) + 2.0), 0x1p-52), 0x1p-1000);
    const double end = side == 0 ? fmax(__dsub_rn(p, B), 0.0) : __dadd_rn(p, B);
    const float x = scalar_at(cfg, which, end);
    const float other = __shfl_xor_sync(0xfu, x, 1);
    if (other == x) return CountedScalar{x, false, false};
    return counted_scalar_exact(cfg, b, t, which, side, 0x3u << (lane & 2));
}

// First launch of the counted steps, one warp of four lanes: the step
// number from the counter, its two scalars (see above), the counter
// advanced, or the bad number reported.  It is launched as a programmatic
// dependent of the previous kernel on the stream (the step kernel of the
// step before, which lets it start once all its CTAs run): it evaluates the
// scalars for the number it reads then, waits for the previous grid to
// complete, reads the number again and evaluates once more only if it
// changed, so the slow part overlaps the previous step's last wave.
__global__ void dopt_count_step_kernel(CounterBlock *c, const dopt_adam_cfg cfg) {
    const int lane = threadIdx.x;
    const int64_t guess = __ldcg(&c->next_step);
    CountedScalar s = counted_scalar(cfg, guess, lane);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the grids before: complete, visible
    // the step kernel after it may now take the SMs (it waits for this grid
    // before it reads the counter)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t t = __ldcg(&c->next_step);
    if (t != guess) s = counted_scalar(cfg, t, lane);
    const bool bad = t < 1 || t > kMaxCountedStep;
    const float bc2_sqrt = __shfl_sync(0xfu, s.x, 2);
    const unsigned exact = __ballot_sync(0xfu, s.exact);
    const unsigned undecided = __ballot_sync(0xfu, s.undecided);
    if (lane != 0) return;
    if (bad) {
        c->status = DOPT_COUNTER_BAD_STEP;
        c->hot.status = DOPT_COUNTER_BAD_STEP;
        return;
    }
    c->hot = CounterHot{s.x, bc2_sqrt, 0, 0};
    if (exact) c->exact_steps += 1;
    if (undecided) c->undecided_steps += 1;
    c->status = 0;
    c->next_step = t + 1;
}

// ---------------------------------------------------------------------------
// The all-reduce kernel: reduce, then write the reduced grads into every
// replica, rounded to the grad type.
// ---------------------------------------------------------------------------

// The all-reduce of the warp's vectors that straddle a run edge, element by
// element over the warp's lanes.
template <typename G, int DC>
__device__ __noinline__ void allreduce_mixed(const AllReduceArgs &a, unsigned mixed) {
    const int D = DC > 0 ? DC : a.D;
    for_straddling_elements(a.rv, a.rv.tile0 + blockIdx.x, mixed, [&](int64_t e, int32_t) {
        const float g = reduce_scalar<G>(a.grads, D, a.R, a.scale, e);
        for (int r = 0; r < D; ++r) store_grad_scalar<G>(a.grads[r], e, g);
    });
}

// The same launch bounds as the step kernel: 0.6 % faster at D = 8 and
// 0.3 % at D = 16.  (The gather kernel keeps the default: 3 CTAs per SM
// helped at D = 8 by 0.5 % and cost 4 % at D = 4.)
// Launched like the step kernels: a programmatic dependent of the kernel
// before it, reading and writing grads only after griddepcontrol.wait.
template <typename G, int DC, int GR = DC>
__global__ void __launch_bounds__(kThreads, 3) dopt_allreduce_kernel(const __grid_constant__ AllReduceArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t tile = a.rv.tile0 + blockIdx.x;
    const int64_t e0 = tile * kDoptTileElems + int64_t(threadIdx.x) * kVec;
    int j;
    const VecKind kind = locate(a.rv, tile, e0, j);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (kind == kFull && vector_in_buffer(a.rv, e0)) {
        float acc[8];
        reduce_vec<G, DC, GR>(a, a.scale, e0, acc);
        write_grads_vec<G, DC>(a.grads, a.D, e0, acc);
    }
    const unsigned mixed = __ballot_sync(0xffffffffu, kind == kMixed);
    if (mixed != 0) allreduce_mixed<G, DC>(a, mixed);
}

// ---------------------------------------------------------------------------
// Pass 1 of the clipped step
// ---------------------------------------------------------------------------

// The clipped step's first launch: zero the workspace's special-value bits,
// non-finite count and accumulator for the norm pass, which starts
// alongside it (a programmatic dependent) and waits for it only before it
// touches the workspace.  One CTA of kThreads threads.
__global__ void dopt_clip_reset_kernel(ClipWorkspace *ws) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int i = threadIdx.x;
    if (i < kAccCopies * kAccWords) (&ws->acc[0][0])[i] = 0ull;
    if (i == 0) {
        ws->special = 0;
        ws->nonfinite = 0;
    }
}

// Add a CTA's partial p (>= 0, or +Inf, or NaN) to accumulator copy `acc`
// exactly (see ClipWorkspace): p = m * 2^e with m < 2^53, and m shifted to
// its place above 2^-149 is at most three 32-bit digits.  The atomics
// return nothing (reductions), so no CTA waits for them.
__device__ __forceinline__ void acc_add(unsigned long long *acc, unsigned int *special, double p) {
    if (p == 0.0) return;
    if (isnan(p)) {
        atomicOr(special, 2u);
        return;
    }
    const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(p));
    const int bexp = int((bits >> 52) & 0x7ff);
    unsigned long long m = bits & ((1ull << 52) - 1);
    int e = -1074;
    if (bexp != 0) {
        m |= 1ull << 52;
        e = bexp - 1075;
    }
    int shift = e - kAccLsb;
    if (shift < 0) {  // m carries trailing zeros down to 2^-149
        m >>= -shift;
        shift = 0;
    }
    if (bexp == 0x7ff || shift + 53 > 32 * kAccWords) {  // +Inf, or beyond the range
        atomicOr(special, 1u);
        return;
    }
    const int w = shift >> 5;
    const unsigned __int128 v = static_cast<unsigned __int128>(m) << (shift & 31);
    const unsigned long long d0 = static_cast<unsigned long long>(v) & 0xffffffffull;
    const unsigned long long d1 = static_cast<unsigned long long>(v >> 32) & 0xffffffffull;
    const unsigned long long d2 = static_cast<unsigned long long>(v >> 64);
    if (d0) atomicAdd(&acc[w], d0);
    if (d1) atomicAdd(&acc[w + 1], d1);
    if (d2) atomicAdd(&acc[w + 2], d2);
}

// The exact sum held in kAccWords words (the copies already added), the
// carries propagated, rounded once to the nearest double.
__device__ double acc_value(const unsigned long long *words) {
    unsigned long long digit[kAccWords];
    unsigned long long carry = 0;
    for (int k = 0; k < kAccWords; ++k) {
        const unsigned long long t = words[k] + carry;
        digit[k] = t & 0xffffffffull;
        carry = t >> 32;
    }
    if (carry) return __longlong_as_double(0x7ff0000000000000ll);  // beyond the range: +Inf
    int top = kAccWords - 1;
    while (top >= 0 && digit[top] == 0) --top;
    if (top < 0) return 0.0;
    // the top three digits as one 96-bit window, left-justified, its top 64
    // bits with every lower bit folded into a sticky bit, then one rounding
    unsigned __int128 win = static_cast<unsigned __int128>(digit[top]) << 64;
    if (top >= 1) win |= static_cast<unsigned __int128>(digit[top - 1]) << 32;
    if (top >= 2) win |= digit[top - 2];
    bool sticky = false;
    for (int k = 0; k < top - 2; ++k) sticky |= digit[k] != 0;
    const int lz = __clzll(static_cast<long long>(digit[top])) - 32;
    win <<= 32 + lz;  // the top bit at bit 127
    unsigned long long hi = static_cast<unsigned long long>(win >> 64);
    sticky |= static_cast<unsigned long long>(win) != 0;
    if (sticky) hi |= 1ull;
    // window bit 95 - lz weighs 2^(32 * (top - 2) + 95 - lz - 149); it is hi's bit 63
    const int scale = 32 * (top - 2) + 95 - lz + kAccLsb - 63;
    return ldexp(__ull2double_rn(hi), scale);
}

// Deterministic sum over a warp (fixed shuffle tree); the result is in lane 0.
__device__ __forceinline__ double warp_sum(double v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    return v;
}

// The fused reduce-scatter writes the fp32 main grads and every CTA
// accumulates the sum of their squares over the tiles it visits (fp32
// squares summed pairwise per 8-element vector, then one fp64 add per
// vector, then the CTA's threads in a fixed order; a vector whose fp32 sum
// reaches 2^120 -- a grad of 2^60 or more, whose fp32 square may overflow
// where the pages' sum of squares does not -- is summed in fp64 instead)
// and adds that partial to
// the workspace's exact accumulator.  The grid is a few tiles per CTA, or a
// persistent grid (see norm_grid on the host); the finalize kernel after it
// turns the sum into the norm and the coefficient.
template <typename G, int DC>
__global__ void __launch_bounds__(kThreads) dopt_rs_norm_kernel(const __grid_constant__ NormArgs a) {
    // the step pass may be scheduled as soon as every CTA of this grid runs:
    // it reads nothing of this pass before its griddepcontrol.wait
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    double local = 0.0;
    unsigned int bad = 0;  // non-finite reduced grads seen by this thread
    for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
        const int64_t tile = a.rv.tile0 + t;
        const int64_t e0 = tile * kDoptTileElems + int64_t(threadIdx.x) * kVec;
        int j;
        const VecKind kind = locate(a.rv, tile, e0, j);
        if (kind == kFull && vector_in_buffer(a.rv, e0)) {
            float acc[8];
            reduce_vec<G, DC>(a, a.scale, e0, acc);
            if (a.round_grad) to_grad_type8<G>(acc);
            st_stream_f4(a.main_grad + e0, make_float4(acc[0], acc[1], acc[2], acc[3]));
            st_stream_f4(a.main_grad + e0 + 4, make_float4(acc[4], acc[5], acc[6], acc[7]));
            float sq[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                sq[k] = __fmul_rn(acc[k], acc[k]);
                bad += isfinite(acc[k]) ? 0u : 1u;
            }
            const float s01 = __fadd_rn(sq[0], sq[1]), s23 = __fadd_rn(sq[2], sq[3]);
            const float s45 = __fadd_rn(sq[4], sq[5]), s67 = __fadd_rn(sq[6], sq[7]);
            const float s = __fadd_rn(__fadd_rn(s01, s23), __fadd_rn(s45, s67));
            if (s < 0x1p120f) {
                local += double(s);
            } else {
                // a square or their sum overflowed fp32, or came near it
                // (a grad of 2^60 or more), or a grad is NaN: the vector's
                // squares again in fp64, where no finite fp32 grad overflows
                double d = 0.0;
#pragma unroll
                for (int k = 0; k < 8; ++k) d += double(acc[k]) * double(acc[k]);
                local += d;
            }
        } else if (kind == kMixed) {
            // one lane per straddling vector: sharing them out over the warp
            // (as the other kernels do) made this persistent loop, and the
            // clipped step, 1.7 % slower
            const int D = DC > 0 ? DC : a.D;
            bool done = false;
            for (int k = 0; k < kVec && !done; ++k) {
                const int64_t e = e0 + k;
                if (!owned_at(a.rv, e, j, done) || !element_in_buffer(a.rv, e)) continue;
                float g = reduce_scalar<G>(a.grads, D, a.R, a.scale, e);
                if (a.round_grad) g = to_grad_type<G>(g);
                a.main_grad[e] = g;
                // fp32 square, or fp64 from 2^60 on (where fp32 overflows)
                local += fabsf(g) < 0x1p60f ? double(__fmul_rn(g, g)) : double(g) * double(g);
                bad += isfinite(g) ? 0u : 1u;
            }
        }
    }
    __shared__ double warp_part[kThreads / 32];
    __shared__ unsigned int warp_bad[kThreads / 32];
    // this pass is a programmatic dependent of the kernel that zeroes the
    // workspace: its grads and tables it may read at once, the workspace
    // only after that kernel has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    local = warp_sum(local);
    bad = __reduce_add_sync(0xffffffffu, bad);
    if (lane == 0) {
        warp_part[threadIdx.x >> 5] = local;
        warp_bad[threadIdx.x >> 5] = bad;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double cta = 0.0;
        unsigned long long cta_bad = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            cta += warp_part[w];
            cta_bad += warp_bad[w];
        }
        acc_add(a.ws->acc[blockIdx.x % kAccCopies], &a.ws->special, cta);
        if (cta_bad) atomicAdd(&a.ws->nonfinite, cta_bad);  // integer: order-free
    }
}

// The clipped step's third launch, one CTA: a programmatic dependent of the
// norm pass (every partial added once that pass has completed), it rounds
// the exact sum of squares once and writes the norm and the clipping
// coefficient min(1, max_norm / (norm + 1e-6)) (NaN, a skip, when
// non-finite grads were counted and the caller asked to skip).  The step
// pass after it starts as soon as this kernel does and waits for it before
// it reads the main grads and the coefficient.
__global__ void __launch_bounds__(kThreads) dopt_clip_finalize_kernel(const __grid_constant__ NormArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ unsigned long long words[kAccWords];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x < kAccWords) {  // the copies of one word (integers: any order)
        unsigned long long t = 0;
        for (int c = 0; c < kAccCopies; ++c) t += __ldcg(&a.ws->acc[c][threadIdx.x]);
        words[threadIdx.x] = t;
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    const unsigned int special = __ldcg(&a.ws->special);
    const double v = (special & 2u)   ? __longlong_as_double(0x7ff8000000000000ll)
                     : (special & 1u) ? __longlong_as_double(0x7ff0000000000000ll)
                                      : acc_value(words);
    const double norm = sqrt(v);
    double coef = double(a.max_norm) / (norm + 1e-6);
    if (coef > 1.0) coef = 1.0;
    const unsigned long long nonfinite = __ldcg(&a.ws->nonfinite);
    float c = float(coef);
    if (a.skip_nonfinite && nonfinite != 0) {
        c = __int_as_float(0x7fc00000);  // skip
        // a skipped step is not counted (the counter kernel before the norm
        // pass advanced the counter; nothing else reads it until this step's
        // kernels are done)
        if (a.counter && a.counter->hot.status == 0) a.counter->next_step -= 1;
    }
    a.ws->norm_sq = v;
    a.ws->norm = float(norm);
    a.ws->coef = c;
    if (a.norm_out) {
        dopt_clip_report *rep = reinterpret_cast<dopt_clip_report *>(a.norm_out);
        rep->norm = float(norm);
        rep->coef = c;
        if (a.skip_nonfinite) rep->nonfinite = nonfinite;
    }
}

// ---------------------------------------------------------------------------
// The gather kernel: each rank's owned elements from its replica to all.
// ---------------------------------------------------------------------------

// The gather of the warp's vectors that straddle a run edge, element by
// element over the warp's lanes.
__device__ __noinline__ void gather_mixed(const GatherArgs &a, unsigned mixed) {
    for_straddling_elements(a.rv, a.rv.tile0 + blockIdx.x, mixed, [&](int64_t e, int32_t meta) {
        const int q = meta >> kRunRankShift;
        for (int base = 0; base < a.D; base += a.R) {
            const uint16_t bits = static_cast<const uint16_t *>(a.params[base + q])[e];
            for (int r = base; r < base + a.R; ++r)
                if (r != base + q) static_cast<uint16_t *>(a.params[r])[e] = bits;
        }
    });
}

// Launched like the step kernels: a programmatic dependent of the kernel
// before it (the step that wrote the owners' replicas), touching params only
// after griddepcontrol.wait.
__global__ void __launch_bounds__(kThreads) dopt_gather_kernel(const __grid_constant__ GatherArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t tile = a.rv.tile0 + blockIdx.x;
    const int64_t e0 = tile * kDoptTileElems + int64_t(threadIdx.x) * kVec;
    int j;
    const VecKind kind = locate(a.rv, tile, e0, j);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (kind == kFull && vector_in_buffer(a.rv, e0)) {
        const int q = a.rv.run_meta[j] >> kRunRankShift;
        for (int base = 0; base < a.D; base += a.R) {
            const uint4 val = ld_stream(static_cast<const __nv_bfloat16 *>(a.params[base + q]) + e0);
            for (int r = base; r < base + a.R; ++r)
                if (r != base + q) st_stream(static_cast<__nv_bfloat16 *>(a.params[r]) + e0, val);
        }
    }
    const unsigned mixed = __ballot_sync(0xffffffffu, kind == kMixed);
    if (mixed != 0) gather_mixed(a, mixed);
}

}  // namespace
