#pragma once
// The stream probe of dopt_stream_probe: the HBM bandwidth of a mix of read
// and write streams, against which the step kernels are measured.  Included
// by step.cu after kernels.cuh (it uses the same block size).
#include <cstdint>

#include <cuda_runtime.h>

namespace {

constexpr int kMaxProbeStreams = 16;

struct ProbeArgs {
    const uint4 *in[kMaxProbeStreams];
    uint4 *out[kMaxProbeStreams];
    int64_t n;  // 16-byte vectors per stream
    int32_t reads, writes;
};

// One 16-byte vector of each read stream in, their XOR with a seed made of
// the vector index to each write stream out, one vector per thread, with the
// step kernels' streaming loads and stores: the ceiling of a read/write mix
// against which those kernels are measured.  With no write stream the
// result is stored (into the first read stream) only if it equals a fixed
// pattern, which keeps the loads from being optimised away.  RMAX (1, 2, 4,
// 8 or 16, at least `reads`) bounds the loads a thread holds at once: every
// load is issued before any is used, as in the step kernels, and a mix of
// few streams keeps few registers and many warps.
template <int RMAX>
__global__ void __launch_bounds__(kThreads) dopt_stream_probe_kernel(const __grid_constant__ ProbeArgs a) {
    const int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x;
    if (i >= a.n) return;
    uint4 acc = make_uint4(uint32_t(i), uint32_t(i >> 32), 0x9e3779b9u, 0x7f4a7c15u);
    uint4 v[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r)
        if (r < a.reads) v[r] = __ldcs(a.in[r] + i);
#pragma unroll
    for (int r = 0; r < RMAX; ++r)
        if (r < a.reads) acc.x ^= v[r].x, acc.y ^= v[r].y, acc.z ^= v[r].z, acc.w ^= v[r].w;
#pragma unroll
    for (int w = 0; w < kMaxProbeStreams; ++w)
        if (w < a.writes) __stcs(a.out[w] + i, acc);
    if (a.writes == 0 && acc.x == 0xffffffffu && acc.y == 0xfffffffeu && acc.z == 0xfffffffdu &&
        acc.w == 0xfffffffcu)
        const_cast<uint4 *>(a.in[0])[i] = acc;  // keeps the loads live
}

}  // namespace
