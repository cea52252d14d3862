"""The library called from several host threads at once (ctypes releases
the GIL, so the calls overlap in the C library): each thread steps its own
layout on its own stream, with the plain, clipped and counted entry points
and a deliberate argument error in between; every result equals the same
calls made one after another, and each thread sees its own error text."""
import ctypes
import threading

import pytest
import torch

from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

LAYOUTS = [
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 0, 1),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 3, 20000, 1),
    ([65536, 1000, 65536], [1, 0, 1], 16, 0, 64),
    ([123457, 99], [1, 0], 4, 0, 1),
]


def _setup(i):
    sizes, wd, D, bucket, pad = LAYOUTS[i]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 3, "bf16", 3000 + i)
    state = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dparams = [p.to(DEV) for p in params]
    dgrads = [[x.to(DEV) for x in gs] for gs in grads]
    return L, D, N, state, dparams, dgrads


def _work(i, L, D, N, state, params, grads, stream, errors):
    adam = B.AdamConfig(grad_scale=1.0 / D)
    with torch.cuda.stream(stream):  # everything of this thread on its own stream
        counter = B.step_counter(2, DEV)
        mg = torch.empty(N, device=DEV)
        ws = B.clip_workspace(DEV)
        B.dopt_step(L, adam, 1, grads[0], *state, params, stream=stream)
        # a misaligned replica, straight through the C ABI: refused before any
        # launch, with the message in this thread's last-error slot
        gp = (ctypes.c_void_p * D)(*([grads[1][0].data_ptr() + 2] +
                                     [g.data_ptr() for g in grads[1][1:]]))
        pp = (ctypes.c_void_p * D)(*[q.data_ptr() for q in params])
        cfg = adam.to_c()
        rc = B.lib().dopt_step(L.handle, ctypes.byref(cfg), 2, gp, B.DOPT_BF16,
                               *[x.data_ptr() for x in state], pp, B.DOPT_STEP_GATHER, None,
                               stream.cuda_stream)
        errors[i] = (rc, B.lib().dopt_last_error().decode())
        B.dopt_step_counted(L, adam, counter, grads[1], *state, params, stream=stream)
        B.dopt_step_clipped(L, adam, 3, 0.05, grads[2], *state, params, mg, ws, stream=stream)
    stream.synchronize()


def test_concurrent_host_threads_match_sequential_calls():
    runs = [_setup(i) for i in range(len(LAYOUTS))]
    seq = [(L, D, N, [x.clone() for x in st], [p.clone() for p in pr], g)
           for L, D, N, st, pr, g in runs]
    torch.cuda.synchronize()  # inputs ready before other streams use them
    errors_seq = {}
    for i, (L, D, N, st, pr, g) in enumerate(seq):
        _work(i, L, D, N, st, pr, g, torch.cuda.Stream(), errors_seq)
    errors = {}
    threads = [threading.Thread(target=_work, args=(i, L, D, N, st, pr, g, torch.cuda.Stream(),
                                                    errors))
               for i, (L, D, N, st, pr, g) in enumerate(runs)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    for (L, D, N, st, pr, g), (_, _, _, st2, pr2, _) in zip(runs, seq):
        for x, y in zip(st + pr, st2 + pr2):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert errors == errors_seq and len(errors) == len(LAYOUTS)
    for rc, text in errors.values():
        assert rc == B.DOPT_E_ALIGN and "dopt_step" in text and "aligned" in text, text
