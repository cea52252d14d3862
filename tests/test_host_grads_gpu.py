"""DOPT_STEP_HOST_GRADS: the kernels read pinned host grad replicas in place.
The results must equal the same step from device copies of the grads, bit
for bit; memory that is not pinned host memory is refused before launch."""
import ctypes

import numpy as np
import pytest
import torch

from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(sizes, wd, D, bucket, pad, dtype, seed, instances=1):
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=instances).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 2, dtype, seed)
    return L, N, master, m, v, params, grads


def _eq(xs, ys):
    for x, y in zip(xs, ys):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D,instances", [(8, 1), (3, 1), (8, 2)])
def test_step_reads_pinned_host_grads(dtype, D, instances):
    L, N, master, m, v, params, grads = _setup([300000, 5, 70001], [1, 0, 1], D, 100000, 64,
                                               dtype, seed=D, instances=instances)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    mga = torch.zeros(N, device=DEV)
    mgb = torch.zeros(N, device=DEV)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    for i in range(2):
        B.dopt_step(L, adam, i + 1, [g.to(DEV) for g in grads[i]], *a, pa, main_grad_out=mga)
        host = [g.contiguous().pin_memory() for g in grads[i]]
        B.dopt_step(L, adam, i + 1, host, *b, pb, main_grad_out=mgb, host_grads=True)
        torch.cuda.synchronize()
    _eq(a + pa + [mga], b + pb + [mgb])


def test_clipped_and_allreduce_with_host_grads():
    D = 4
    L, N, master, m, v, params, grads = _setup([200000, 77, 9000], [1, 0, 1], D, 0, 8, "bf16", 3)
    adam = B.AdamConfig(grad_scale=0.25)
    # clipped
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    B.dopt_step_clipped(L, adam, 1, 0.05, [g.to(DEV) for g in grads[0]], *a, pa,
                        torch.empty(N, device=DEV), B.clip_workspace(DEV))
    host = [g.contiguous().pin_memory() for g in grads[0]]
    import zero_distributed_optimizer_gb300.binding as bb

    gp = (ctypes.c_void_p * D)(*[h.data_ptr() for h in host])
    pp = (ctypes.c_void_p * D)(*[p.data_ptr() for p in pb])
    mg = torch.empty(N, device=DEV)
    ws = B.clip_workspace(DEV)
    cfg = adam.to_c()
    rc = bb.lib().dopt_step_clipped(L.handle, ctypes.byref(cfg), 1, 0.05, gp, B.DOPT_BF16,
                                    b[0].data_ptr(), b[1].data_ptr(), b[2].data_ptr(), pp,
                                    B.DOPT_STEP_GATHER | B.DOPT_STEP_HOST_GRADS, mg.data_ptr(),
                                    ws.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert rc == B.DOPT_OK, bb.lib().dopt_last_error()
    torch.cuda.synchronize()
    _eq(a + pa, b + pb)
    # force_all_reduce writes the reduced grads back into the host buffers
    dev = [g.to(DEV) for g in grads[1]]
    host = [g.contiguous().pin_memory() for g in grads[1]]
    c = [master.to(DEV), m.to(DEV), v.to(DEV)]
    d = [x.clone() for x in c]
    pc = [p.to(DEV) for p in params]
    pd = [p.clone() for p in pc]
    B.dopt_step_allreduce(L, adam, 2, dev, *c, pc)
    gp = (ctypes.c_void_p * D)(*[h.data_ptr() for h in host])
    pp = (ctypes.c_void_p * D)(*[p.data_ptr() for p in pd])
    rc = bb.lib().dopt_step_allreduce(L.handle, ctypes.byref(cfg), 2, gp, B.DOPT_BF16,
                                      d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), pp,
                                      B.DOPT_STEP_GATHER | B.DOPT_STEP_HOST_GRADS, None,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == B.DOPT_OK, bb.lib().dopt_last_error()
    torch.cuda.synchronize()
    _eq(c + pc, d + pd)
    for x, h in zip(dev, host):
        assert torch.equal(x.cpu().view(torch.int16), h.view(torch.int16))


def test_step_from_host_zero_copy_equals_staged():
    D = 8
    L, N, master, m, v, params, grads = _setup([500000, 3, 12345], [1, 0, 1], D, 0, 64, "bf16", 8)
    host = [g.contiguous().pin_memory() for g in grads[0]]
    stage = [torch.empty_like(g, device=DEV) for g in grads[0]]
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    outa = torch.empty(N, dtype=torch.bfloat16).pin_memory()
    outb = torch.empty(N, dtype=torch.bfloat16).pin_memory()
    adam = B.AdamConfig(grad_scale=0.125)
    B.step_from_host(L, adam, 1, host, stage, *a, pa, outa)
    B.step_from_host(L, adam, 1, host, None, *b, pb, outb, zero_copy=True)
    torch.cuda.synchronize()
    _eq(a + pa, b + pb)
    assert torch.equal(outa.view(torch.int16), outb.view(torch.int16))


def test_host_grads_refuses_unpinned_memory():
    D = 2
    L, N, master, m, v, params, grads = _setup([4096, 8], None, D, 0, 8, "bf16", 1)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    p = [x.to(DEV) for x in params]
    with pytest.raises(B.DoptError):  # the binding wants pinned tensors
        B.dopt_step(L, B.AdamConfig(), 1, [g.contiguous() for g in grads[0]], *d, p,
                    host_grads=True)
    # through the C ABI: pageable numpy memory and device memory are refused
    pageable = [np.zeros(N + 64, np.uint16) for _ in range(D)]
    ptrs = [(a.ctypes.data + 63) & ~63 for a in pageable]
    cfg = B.AdamConfig().to_c()
    pp = (ctypes.c_void_p * D)(*[x.data_ptr() for x in p])
    for gptrs in (ptrs, [g.to(DEV).data_ptr() for g in grads[0]]):
        gp = (ctypes.c_void_p * D)(*gptrs)
        rc = B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, B.DOPT_BF16,
                               d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), pp,
                               B.DOPT_STEP_GATHER | B.DOPT_STEP_HOST_GRADS, None, None)
        assert rc == B.DOPT_E_ARG, rc
    torch.cuda.synchronize()  # the context is still usable


def test_host_stepper_results():
    """The pipelined stepper gives the same state and, after synchronize,
    the same host copy of the params as step_from_host, step by step."""
    D = 4
    L, N, master, m, v, params, grads = _setup([400000, 3, 12345], [1, 0, 1], D, 0, 64, "bf16", 9)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    outa = torch.empty(N, dtype=torch.bfloat16).pin_memory()
    outb = torch.empty(N, dtype=torch.bfloat16).pin_memory()
    adam = B.AdamConfig(grad_scale=0.25)
    stepper = B.HostStepper(L, adam, *b, pb, outb)
    for i in range(2):
        host = [g.contiguous().pin_memory() for g in grads[i]]
        B.step_from_host(L, adam, i + 1, host, None, *a, pa, outa, zero_copy=True)
        stepper.step(i + 1, host)
        stepper.synchronize()
        torch.cuda.synchronize()
        assert torch.equal(outa.view(torch.int16), outb.view(torch.int16))
    _eq(a + pa, b + pb)


@pytest.mark.parametrize("host_replicas", [(0,), (0, 1, 2, 3)])
def test_step_writes_pinned_host_params(host_replicas):
    """DOPT_STEP_HOST_PARAMS: param replicas in pinned host memory (replica
    0 alone, or all of them) are written in place by the step, with host
    grads too; every buffer equals the all-device step bit for bit."""
    D = 4
    L, N, master, m, v, params, grads = _setup([300000, 5, 70001], [1, 0, 1], D, 100000, 64,
                                               "bf16", seed=11)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone().pin_memory() if r in host_replicas else p.to(DEV)
          for r, p in enumerate(params)]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    for i in range(2):
        B.dopt_step(L, adam, i + 1, [g.to(DEV) for g in grads[i]], *a, pa)
        host = [g.contiguous().pin_memory() for g in grads[i]]
        B.dopt_step(L, adam, i + 1, host, *b, pb, host_grads=True, host_params=True)
        torch.cuda.synchronize()
    _eq(a + pa, b + [p.to(DEV) for p in pb])


def test_step_from_host_params_out_in_place():
    """The end-to-end form: host grads read in place and param replica 0
    written straight into the pinned output; it equals the staged form's
    copy of replica 0."""
    D = 8
    L, N, master, m, v, params, grads = _setup([300000, 5, 70001], [1, 0, 1], D, 100000, 64,
                                               "bf16", seed=12)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    # the in-place output is replica 0 itself, so it starts as replica 0 did
    # (the step never writes padding); the staged form copies the whole
    # replica, padding included
    out_a = torch.empty(N, dtype=torch.bfloat16).pin_memory()
    out_b = params[0].clone().pin_memory()
    adam = B.AdamConfig(grad_scale=1.0 / D)
    stage = [torch.empty(N, dtype=torch.bfloat16, device=DEV) for _ in range(D)]
    for i in range(2):
        host = [g.contiguous().pin_memory() for g in grads[i]]
        B.step_from_host(L, adam, i + 1, host, stage, *a, pa, out_a)
        B.step_from_host(L, adam, i + 1, host, None, *b, pb, out_b, zero_copy=True,
                         params_out_in_place=True)
        torch.cuda.synchronize()
    _eq(a + pa[1:] + [out_a], b + pb[1:] + [out_b])


def test_host_params_refuses_pageable_memory():
    D = 2
    L, N, master, m, v, params, grads = _setup([1000, 24], None, D, 0, 8, "bf16", seed=13)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    g = [x.to(DEV) for x in grads[0]]
    pageable = torch.zeros(N, dtype=torch.bfloat16)  # not pinned
    pp = (ctypes.c_void_p * D)(pageable.data_ptr(), params[1].to(DEV).data_ptr())
    gp = (ctypes.c_void_p * D)(*[x.data_ptr() for x in g])
    cfg = B.AdamConfig().to_c()
    import zero_distributed_optimizer_gb300.binding as bb

    rc = bb.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, B.DOPT_BF16, d[0].data_ptr(),
                            d[1].data_ptr(), d[2].data_ptr(), pp,
                            B.DOPT_STEP_GATHER | B.DOPT_STEP_HOST_PARAMS, None,
                            torch.cuda.current_stream().cuda_stream)
    assert rc == B.DOPT_E_ARG and "param replica 0" in bb.lib().dopt_last_error().decode()
    torch.cuda.synchronize()  # the context is still usable
