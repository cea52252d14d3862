"""The boundary from plain C on the device: a C11 program that includes
include/dopt.h, allocates with the CUDA runtime, builds the layout, runs
two fused steps and a standalone gather through libdopt.so, and checks the
results against the CPU oracle's C functions, which it links as well (the
program is test infrastructure; the oracle and the library share nothing).
It also checks an error path: a misaligned replica gives DOPT_E_ALIGN and a
message."""
import os
import subprocess

import pytest

import oracle
from zero_distributed_optimizer_gb300 import build as libbuild

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "dopt.h"

/* the oracle's entry (test infrastructure; see oracle/dopt_oracle.c) */
typedef struct { float lr, beta1, beta2, eps, weight_decay, grad_scale; } orc_adam;
int orc_step(const int64_t *sizes, int32_t n, const uint8_t *wd_mask, int32_t D,
             int32_t instances, int64_t bucket_elems, int32_t pad_unit, const orc_adam *cfg,
             int64_t step, int32_t grad_type, const void *const *grads, float *master,
             float *exp_avg, float *exp_avg_sq, uint16_t *const *params, int32_t gather,
             float *main_grad_out, int64_t w0, int64_t w1, float clip_coef, int32_t round_grad,
             int32_t param_is_f16);

#define NR 4
#define CHECK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    printf("cuda error %s at %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)

static uint64_t rng = 88172645463325252ull;
static float next_unit(void)  /* xorshift64, uniform in [-1, 1) */
{
    rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17;
    return (float)((double)(rng >> 11) / 9007199254740992.0 * 2.0 - 1.0);
}
static uint16_t to_bf16_trunc(float f) { uint32_t u; memcpy(&u, &f, 4); return (uint16_t)(u >> 16); }

int main(void)
{
    const int64_t sizes[7] = {130, 260, 90, 310, 210, 5003, 17};
    const uint8_t wd[7] = {1, 1, 0, 1, 1, 1, 0};
    dopt_layout_cfg lc = {.D = NR, .bucket_elems = 0, .pad_unit = 8};
    dopt_layout *L = NULL;
    if (dopt_build_range_map(sizes, 7, wd, &lc, &L) != DOPT_OK || dopt_layout_to_device(L) != DOPT_OK) {
        printf("layout: %s\n", dopt_last_error());
        return 1;
    }
    int64_t N = 0;
    int32_t nb = 0, np = 0;
    dopt_layout_query(L, &N, &nb, &np);
    size_t n = (size_t)N;
    /* each param's place in the flat buffer: consecutive offsets */
    dopt_range po[7];
    if (dopt_layout_param_offsets(L, po) != DOPT_OK) {
        printf("param offsets: %s\n", dopt_last_error());
        return 1;
    }
    int64_t at = 0;
    for (int p = 0; p < 7; ++p) {
        if (po[p].start != at || po[p].end != at + sizes[p]) {
            printf("param %d at [%lld,%lld), expected start %lld\n", p, (long long)po[p].start,
                   (long long)po[p].end, (long long)at);
            return 1;
        }
        at = po[p].end;
    }
    printf("param offsets ok, %lld elements padded to %lld\n", (long long)at, (long long)N);
    uint16_t *hg[2][NR], *hp[NR], *op[NR];
    float *hs[3], *os[3];
    for (int s = 0; s < 3; ++s) {
        hs[s] = malloc(n * 4);
        os[s] = malloc(n * 4);
        for (size_t i = 0; i < n; ++i)
            hs[s][i] = s == 0 ? 0.02f * next_unit() : (s == 1 ? 1e-4f * next_unit() : 1e-6f * (next_unit() + 1.0f));
        memcpy(os[s], hs[s], n * 4);
    }
    for (int r = 0; r < NR; ++r) {
        hp[r] = malloc(n * 2);
        op[r] = malloc(n * 2);
        for (size_t i = 0; i < n; ++i) hp[r][i] = to_bf16_trunc(0.02f * next_unit());
        memcpy(op[r], hp[r], n * 2);
        for (int t = 0; t < 2; ++t) {
            hg[t][r] = malloc(n * 2);
            for (size_t i = 0; i < n; ++i) hg[t][r][i] = to_bf16_trunc(1e-3f * next_unit());
        }
    }
    void *dg[NR], *dp[NR];
    float *ds[3];
    for (int r = 0; r < NR; ++r) {
        CHECK(cudaMalloc(&dg[r], n * 2));
        CHECK(cudaMalloc(&dp[r], n * 2));
        CHECK(cudaMemcpy(dp[r], hp[r], n * 2, cudaMemcpyHostToDevice));
    }
    for (int s = 0; s < 3; ++s) {
        CHECK(cudaMalloc((void **)&ds[s], n * 4));
        CHECK(cudaMemcpy(ds[s], hs[s], n * 4, cudaMemcpyHostToDevice));
    }
    dopt_adam_cfg cfg = {1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 0.25f};
    orc_adam ocfg = {1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 0.25f};
    for (int t = 0; t < 2; ++t) {
        for (int r = 0; r < NR; ++r)
            CHECK(cudaMemcpy(dg[r], hg[t][r], n * 2, cudaMemcpyHostToDevice));
        /* step 1 with the fused gather; step 2 without it, then dopt_gather */
        uint32_t flags = t == 0 ? DOPT_STEP_GATHER : 0u;
        if (dopt_step(L, &cfg, t + 1, (const void *const *)dg, DOPT_BF16, ds[0], ds[1], ds[2], dp,
                      flags, NULL, 0) != DOPT_OK) {
            printf("step: %s\n", dopt_last_error());
            return 1;
        }
        if (t == 1 && dopt_gather(L, dp, 0) != DOPT_OK) {
            printf("gather: %s\n", dopt_last_error());
            return 1;
        }
        if (orc_step(sizes, 7, wd, NR, 1, 0, 8, &ocfg, t + 1, 0, (const void *const *)hg[t], os[0],
                     os[1], os[2], op, 1, NULL, 0, N, 1.0f, 0, 0) != 0) {
            printf("oracle failed\n");
            return 1;
        }
    }
    CHECK(cudaDeviceSynchronize());
    long diff = 0;
    for (int s = 0; s < 3; ++s) {
        CHECK(cudaMemcpy(hs[s], ds[s], n * 4, cudaMemcpyDeviceToHost));
        diff += memcmp(hs[s], os[s], n * 4) != 0;
    }
    for (int r = 0; r < NR; ++r) {
        CHECK(cudaMemcpy(hp[r], dp[r], n * 2, cudaMemcpyDeviceToHost));
        diff += memcmp(hp[r], op[r], n * 2) != 0;
    }
    printf("elements %lld buffers differing %ld\n", (long long)N, diff);
    /* an error path: a replica pointer off its 16-byte alignment */
    void *bad[NR] = {dg[0], (char *)dg[1] + 2, dg[2], dg[3]};
    int rc = dopt_step(L, &cfg, 3, (const void *const *)bad, DOPT_BF16, ds[0], ds[1], ds[2], dp,
                       DOPT_STEP_GATHER, NULL, 0);
    printf("misaligned -> %d (%s)\n", rc, dopt_last_error());
    dopt_layout_free(L);
    return diff == 0 && rc == DOPT_E_ALIGN ? 0 : 1;
}
"""


def test_c_program_steps_on_the_device(tmp_path):
    lib = libbuild.build()
    orc = oracle.build()
    src = tmp_path / "prog.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    cuda = libbuild.cuda_home()
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                           os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                           os.path.join(cuda, "targets", "x86_64-linux", "lib"))
               if os.path.isdir(d)]
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), str(src), "-o", str(exe),
           "-L", os.path.dirname(lib), "-ldopt", orc]
    for d in libdirs:
        cmd += ["-L", d]
    cmd += ["-lcudart", "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.dirname(orc)]
    cmd += ["-Wl,-rpath," + d for d in libdirs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "param offsets ok, 6020 elements padded to 6048" in out.stdout
    assert "buffers differing 0" in out.stdout
    assert "misaligned -> -3" in out.stdout
