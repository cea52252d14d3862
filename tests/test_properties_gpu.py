"""Properties that hold at any size, checked over the whole buffer of
full-size workloads on the device (the windowed oracle comparisons cover the
values themselves):

* all-reduce = reduce-scatter + all-gather (tutorial "AllReduce"): the
  all-reduced bf16 grads equal the bf16 rounding of the main grads the step
  reports, at every owned element, in every replica;
* after the fused gather all D param replicas are identical;
* padding is never written, in any buffer;
* integer-valued grads make the result independent of D (exact sums)."""
import pytest
import torch

from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _owned_mask(L):
    mask = torch.zeros(L.padded_numel, dtype=torch.bool, device=DEV)
    for a, b in L.param_offsets():
        mask[a:b] = True
    return mask


@pytest.mark.parametrize("make", [W.gpt2_small, lambda: W.sweep_256m(16, 1)],
                         ids=["gpt2_small", "sweep_256m_D16_b1M"])
def test_whole_buffer_properties(make):
    w = make()
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    N = L.padded_numel
    owned = _owned_mask(L)
    pad = ~owned
    master, m, v = W.make_state(w, N, DEV)
    params = [p + 0 for p in W.make_params(master, w.D)]
    for r, p in enumerate(params):  # distinct padding per replica
        p[pad] = float(r + 1)
    before = [x.clone() for x in (master, m, v)]
    pbefore = [p.clone() for p in params]
    grads = W.make_grads(w, N, 1, DEV)
    mg = torch.full((N,), 7.0, device=DEV)
    adam = B.AdamConfig(**w.adam_kwargs())
    B.dopt_step(L, adam, 1, grads, master, m, v, params, main_grad_out=mg)
    B.dopt_allreduce(L, grads, w.grad_scale)
    torch.cuda.synchronize()
    want = mg.to(torch.bfloat16)
    for g in grads:
        assert torch.equal(g[owned].view(torch.int16), want[owned].view(torch.int16))
    for p in params[1:]:
        assert torch.equal(p[owned].view(torch.int16), params[0][owned].view(torch.int16))
    for x, x0 in zip((master, m, v), before):
        assert torch.equal(x[pad].view(torch.int32), x0[pad].view(torch.int32))
        assert not torch.equal(x[owned], x0[owned])
    for p, p0 in zip(params, pbefore):
        assert torch.equal(p[pad].view(torch.int16), p0[pad].view(torch.int16))
    assert torch.all(mg[pad] == 7.0)


def test_full_size_d_independence():
    """GPT-2-small layout, integer-valued grads g_r = (G + (2r - D + 1)*2)/1024
    with scaling 1/D: every partial sum is exact, so D = 1, 2, 4, 8 give
    bitwise the same master, m, v and params for every param after 2 steps."""
    base = W.gpt2_small()
    n = base.numel
    gen = torch.Generator(device=DEV)
    gen.manual_seed(W.seed_of("d_independence"))
    G = [torch.randint(-64, 65, (n,), generator=gen, device=DEV).float() for _ in range(2)]
    results = {}
    for D in (1, 2, 4, 8):
        w = base.with_(D=D, grad_scale=1.0 / D)
        L = B.dopt_build_range_map(list(w.sizes), D, w.bucket_elems, w.pad_unit,
                                   list(w.wd_mask)).to_device()
        N = L.padded_numel
        owned = _owned_mask(L)
        master, m, v = (torch.zeros(N, device=DEV) for _ in range(3))
        init = W.make_state(base.with_(name="d_independence"), n, DEV)
        for x, x0 in zip((master, m, v), init):
            x[owned] = x0
        params = W.make_params(master, D)
        adam = B.AdamConfig(**w.adam_kwargs())
        for t in range(2):
            grads = []
            for r in range(D):
                g = torch.zeros(N, device=DEV)
                g[owned] = (G[t] + (2 * r - (D - 1)) * 2) / 1024.0
                grads.append(g.to(torch.bfloat16))
            B.dopt_step(L, adam, t + 1, grads, master, m, v, params)
            del grads
        torch.cuda.synchronize()
        results[D] = [x[owned].view(torch.int32).clone() for x in (master, m, v)] + \
                     [params[0][owned].view(torch.int16).clone(),
                      params[-1][owned].view(torch.int16).clone()]
        del master, m, v, params
    for D in (2, 4, 8):
        for a, b in zip(results[D], results[1]):
            assert torch.equal(a, b), D
