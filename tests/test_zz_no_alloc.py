"""dopt_step_clipped_noalloc against dopt_step_clipped.

The no-allocation entry point serves callers that cannot allocate device
memory on the step's path (a framework's caching allocator owns the memory,
or the loop cannot take the synchronisation that cudaMalloc/cudaFree can
cause).  It keeps the norm pass's scratch in a static array inside the
library instead of a caller workspace.  This file checks, through the C ABI,
that two calls in a row give the same results as the workspace entry point
within the parity tolerance, including the second call, which finds the
first call's contents still in the shared scratch, and that this second
call takes no device memory (the device's free memory, as cudaMemGetInfo
reports it, and the count of torch's allocations stay as they were).  It is
collected last and also passes alone in a fresh process."""
import pytest
import torch

from parity import assert_bf16_close, assert_f32_close, t2np_bf16, t2np_f32
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("grad_dtype,D", [("bf16", 8), ("fp32", 3)])
def test_noalloc_matches_workspace_entry_point(grad_dtype, D):
    sizes, wd = [300000, 5, 70001, 4096, 123], [1, 0, 1, 1, 0]
    L = B.dopt_build_range_map(sizes, D, 100000, 64, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 2, grad_dtype, seed=D)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    mga = torch.full((N,), -1.0, device=DEV)
    mgb = mga.clone()
    na = torch.zeros(2, device=DEV)
    nb = torch.zeros(2, device=DEV)
    ws = B.clip_workspace(DEV)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    dev_grads = [[x.to(DEV) for x in grads[i]] for i in range(2)]
    torch.cuda.synchronize()
    for i, max_norm in enumerate((0.05, 1e9)):  # clipping engaged, then not
        g = dev_grads[i]
        B.dopt_step_clipped(L, adam, i + 1, max_norm, g, *a, pa, mga, ws, norm_out=na)
        if i == 1:  # after the first call's set-up: nothing may allocate
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            allocs_before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        B.dopt_step_clipped_noalloc(L, adam, i + 1, max_norm, g, *b, pb, mgb, norm_out=nb)
        torch.cuda.synchronize()
        if i == 1:
            # no device memory taken by the call: not from CUDA (free
            # memory of the device unchanged), not from torch's allocator
            assert torch.cuda.mem_get_info()[0] == free_before
            assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs_before
        assert_f32_close(t2np_f32(nb), t2np_f32(na), f"norm/coef call {i}")
        for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), b, a):
            assert_f32_close(t2np_f32(x), t2np_f32(y), f"{name} call {i}")
        assert_f32_close(t2np_f32(mgb), t2np_f32(mga), f"main_grad call {i}")
        for r in range(D):
            assert_bf16_close(t2np_bf16(pb[r]), t2np_bf16(pa[r]), f"param{r} call {i}")
    assert nb[1].item() == 1.0 and na[1].item() == 1.0
