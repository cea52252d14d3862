"""The boundary is plain C: a C11 program that includes include/dopt.h,
links libdopt.so and calls the host-only entry points as the boundary
states them (dopt_build_range_map, dopt_layout_query, dopt_layout_buckets,
dopt_layout_pieces, dopt_layout_param_offsets, dopt_layout_free; layout and range
map of the ownership demo on the distributed-optimizer page, §3) compiles without warnings and runs
without a GPU."""
import os
import subprocess

import pytest

from zero_distributed_optimizer_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "dopt.h"

_Static_assert(sizeof(dopt_step_counter) == 64, "dopt_step_counter is 64 bytes");

int main(void)
{
    const int64_t sizes[5] = {130, 260, 90, 310, 210};
    dopt_layout_cfg cfg = {.D = 4, .bucket_elems = 0, .pad_unit = 1};
    dopt_layout *L = NULL;
    if (dopt_build_range_map(sizes, 5, NULL, &cfg, &L) != DOPT_OK) {
        printf("build failed: %s\n", dopt_last_error());
        return 1;
    }
    int64_t numel = 0;
    int32_t nb = 0, np = 0;
    dopt_layout_query(L, &numel, &nb, &np);
    printf("numel %lld buckets %d pieces %d\n", (long long)numel, nb, np);
    dopt_piece pieces[16];
    dopt_layout_pieces(L, pieces);
    for (int i = 0; i < np; ++i)
        if (pieces[i].rank == 1)
            printf("rank 1 param %d world [%lld,%lld) local [%lld,%lld) param [%lld,%lld)\n",
                   pieces[i].param_id, (long long)pieces[i].gbuf_world.start,
                   (long long)pieces[i].gbuf_world.end, (long long)pieces[i].gbuf_local.start,
                   (long long)pieces[i].gbuf_local.end, (long long)pieces[i].param.start,
                   (long long)pieces[i].param.end);
    dopt_range buckets[1], params[5];
    dopt_layout_buckets(L, buckets);
    printf("bucket [%lld,%lld)\n", (long long)buckets[0].start, (long long)buckets[0].end);
    if (dopt_layout_param_offsets(L, params) != DOPT_OK) return 1;
    for (int p = 0; p < 5; ++p)
        printf("param %d [%lld,%lld)\n", p, (long long)params[p].start, (long long)params[p].end);
    dopt_layout_cfg bad = {.D = 0, .bucket_elems = 0, .pad_unit = 1};
    dopt_layout *L2 = NULL;
    printf("bad D -> %d\n", dopt_build_range_map(sizes, 5, NULL, &bad, &L2));
    dopt_layout_free(L);
    printf("%s\n", dopt_version());
    return 0;
}
"""


def test_c11_program_uses_the_boundary(tmp_path):
    lib = libbuild.build()
    src = tmp_path / "prog.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    cuda_inc = os.path.join(libbuild.cuda_home(), "include")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", cuda_inc, str(src), "-o", str(exe), "-L", os.path.dirname(lib), "-ldopt",
           "-Wl,-rpath," + os.path.dirname(lib)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    lines = out.stdout.splitlines()
    assert lines[0] == "numel 1000 buckets 1 pieces 8"
    assert lines[1:4] == ["rank 1 param 1 world [250,390) local [0,140) param [120,260)",
                          "rank 1 param 2 world [390,480) local [140,230) param [0,90)",
                          "rank 1 param 3 world [480,500) local [230,250) param [0,20)"]
    assert lines[4] == "bucket [0,1000)"
    assert lines[5:10] == ["param 0 [0,130)", "param 1 [130,390)", "param 2 [390,480)",
                           "param 3 [480,790)", "param 4 [790,1000)"]
    assert lines[10] == "bad D -> -1"
    assert "sm_103a" in lines[11]
