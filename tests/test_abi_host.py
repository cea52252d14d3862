"""Host-side checks of libdopt.so that need no GPU: the library loads and
exports every function include/*.h declares; the range map it builds is
bit-exact with the oracle's; invalid arguments are refused before any CUDA
call is made."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
import pins
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import build as libbuild
from zero_distributed_optimizer_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.lib()


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(dopt_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    # the calls of the boundary as the scope table names them
    for required in ("dopt_build_range_map", "dopt_layout_query", "dopt_layout_buckets",
                     "dopt_layout_pieces", "dopt_layout_param_offsets", "dopt_layout_free",
                     "dopt_step", "dopt_gather", "dopt_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(B.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing
    assert "sm_103a" in B.version()


def _lib_layout(sizes, D, bucket, pad, wd=None):
    return B.dopt_build_range_map(sizes, D, bucket_elems=bucket, pad_unit=pad, wd_mask=wd)


def _compare_with_oracle(sizes, D, bucket, pad):
    L = _lib_layout(sizes, D, bucket, pad)
    O = oracle.range_map(sizes, D, bucket, pad)
    assert L.padded_numel == O.numel
    assert L.buckets() == list(zip(O.bucket_start.tolist(), O.bucket_end.tolist()))
    assert L.param_offsets() == list(zip(O.param_start.tolist(), O.param_end.tolist()))
    assert L.param_ranges() == L.param_offsets()
    assert L.pieces() == O.pieces
    return L


def test_range_map_matches_oracle_tiny(lib):
    for sizes, D, bucket, pad in pins.random_tiny_layouts(400, seed=99):
        _compare_with_oracle(sizes, D, bucket, pad)


def test_range_map_page1_example(lib):
    L = _compare_with_oracle([130, 260, 90, 310, 210], 4, 0, 1)
    assert [pc for pc in L.pieces() if pc["rank"] == 1][0]["gbuf_world"] == (250, 390)


@pytest.mark.parametrize("w", W.all_configs(), ids=lambda w: w.name)
def test_range_map_matches_oracle_configs(lib, w):
    _compare_with_oracle(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)


def test_range_map_matches_oracle_sweep(lib):
    for D in W.SWEEP_D:
        for b in W.SWEEP_BUCKET_MI:
            w = W.sweep_256m(D, b)
            _compare_with_oracle(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)


def test_range_map_larger_random(lib):
    rng = np.random.default_rng(5)
    for _ in range(30):
        n = int(rng.integers(1, 300))
        sizes = [int(x) for x in rng.integers(0, 5000, n)]
        D = int(rng.integers(1, 65))
        bucket = int(rng.choice([0, int(rng.integers(1, 50000))]))
        pad = int(rng.integers(1, 130))
        _compare_with_oracle(sizes, D, bucket, pad)


def test_layout_errors(lib):
    for sizes, D, bucket, pad in (([4], 0, 0, 1), ([4], 65, 0, 1), ([4, -1], 2, 0, 1),
                                  ([4], 2, 0, 0), ([4], 2, -1, 1)):
        with pytest.raises(B.DoptError) as e:
            _lib_layout(sizes, D, bucket, pad)
        assert e.value.code == B.DOPT_E_ARG
        assert B.lib().dopt_last_error().decode().startswith("dopt_build_range_map")
    out = ctypes.c_void_p()
    assert B.lib().dopt_build_range_map(None, 3, None, None, ctypes.byref(out)) == B.DOPT_E_ARG
    assert B.lib().dopt_build_range_map(None, 0, None, None, None) == B.DOPT_E_ARG


def test_empty_layouts(lib):
    L = _lib_layout([], 4, 0, 1)
    assert L.padded_numel == 0 and L.n_buckets == 0 and L.n_pieces == 0
    L = _lib_layout([0, 0], 3, 0, 2)
    assert L.padded_numel == 0 and L.n_buckets == 1 and L.n_pieces == 0


def _raw_step(L, ptr_grads, ptr_state, ptr_params, step=1, flags=1, dtype=B.DOPT_BF16, cfg=None,
              main_grad=None):
    D = L.D
    cfg = cfg or B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * D)(*ptr_grads)
    pp = (ctypes.c_void_p * D)(*ptr_params)
    return B.lib().dopt_step(L.handle, ctypes.byref(cfg), step, gp, dtype, ptr_state[0],
                             ptr_state[1], ptr_state[2], pp, flags, main_grad, None)


def test_step_argument_checks_before_cuda(lib):
    """Refusals that come before the library touches CUDA (no GPU needed):
    the fake pointers below are never dereferenced."""
    L = _lib_layout([100, 30], 2, 0, 8)
    good = [0x10000, 0x20000]
    state = [0x30000, 0x40000, 0x50000]
    assert _raw_step(L, good, state, good, step=0) == B.DOPT_E_ARG
    assert _raw_step(L, good, state, good, flags=8) == B.DOPT_E_ARG
    assert _raw_step(L, good, state, good, dtype=7) == B.DOPT_E_ARG
    assert _raw_step(L, [0x10000, 0], state, good) == B.DOPT_E_ARG
    assert _raw_step(L, [0x10000, 0x20002], state, good) == B.DOPT_E_ALIGN
    assert _raw_step(L, good, [0x30000, 0x40008, 0x50000], good) == B.DOPT_E_ALIGN
    assert _raw_step(L, good, state, good, main_grad=0x60004) == B.DOPT_E_ALIGN
    bad_cfg = B.AdamConfig(beta1=1.0).to_c()
    assert _raw_step(L, good, state, good, cfg=bad_cfg) == B.DOPT_E_ARG
    bad_cfg = B.AdamConfig(lr=float("nan")).to_c()
    assert _raw_step(L, good, state, good, cfg=bad_cfg) == B.DOPT_E_ARG
    assert B.lib().dopt_step(None, None, 1, None, 0, None, None, None, None, 1, None, None) == B.DOPT_E_ARG
    # an empty layout is a no-op that never needs the device
    E = _lib_layout([], 2, 0, 1)
    assert _raw_step(E, good, state, good) == B.DOPT_OK
    # with valid arguments the next check needs the device tables
    rc = _raw_step(L, good, state, good)
    assert rc in (B.DOPT_E_STATE, B.DOPT_E_CUDA)
    assert B.lib().dopt_last_error().decode()


def test_gather_argument_checks_before_cuda(lib):
    L = _lib_layout([100, 30], 2, 0, 8)
    pp = (ctypes.c_void_p * 2)(0x10000, 0x20001)
    assert B.lib().dopt_gather(L.handle, pp, None) == B.DOPT_E_ALIGN
    pp = (ctypes.c_void_p * 2)(0x10000, 0)
    assert B.lib().dopt_gather(L.handle, pp, None) == B.DOPT_E_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch

    L = _lib_layout([16], 1, 0, 1)
    t = torch.zeros(16)
    with pytest.raises(B.DoptError):
        B.dopt_step(L, B.AdamConfig(), 1, [t.bfloat16()], t, t.clone(), t.clone(), [t.bfloat16()])


def test_clipped_step_argument_checks_before_cuda(lib):
    L = _lib_layout([100, 30], 2, 0, 8)
    cfg = B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)

    def call(max_norm=1.0, main=0x70000, ws=0x80000, norm_out=None):
        return B.lib().dopt_step_clipped(L.handle, ctypes.byref(cfg), 1, max_norm, gp, 0,
                                         0x30000, 0x40000, 0x50000, gp, 1, main, ws, norm_out,
                                         None)

    assert call(main=None) == B.DOPT_E_ARG
    assert call(ws=None) == B.DOPT_E_ARG
    assert call(max_norm=0.0) == B.DOPT_E_ARG
    assert call(max_norm=float("inf")) == B.DOPT_E_ARG
    assert call(ws=0x80004) == B.DOPT_E_ALIGN
    assert call(main=0x70004) == B.DOPT_E_ALIGN
    assert call(norm_out=0x90004) == B.DOPT_E_ALIGN
    assert call() in (B.DOPT_E_STATE, B.DOPT_E_CUDA)


def test_bucket_and_allreduce_argument_checks_before_cuda(lib):
    L = _lib_layout([100, 50, 60], 2, 40, 8)
    assert L.n_buckets == 3
    cfg = B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)

    def buckets(first, count):
        return B.lib().dopt_step_buckets(L.handle, ctypes.byref(cfg), 1, first, count, gp, 0,
                                         0x30000, 0x40000, 0x50000, gp, 1, None, None)

    assert buckets(-1, 1) == B.DOPT_E_ARG
    assert buckets(0, 4) == B.DOPT_E_ARG
    assert buckets(3, 1) == B.DOPT_E_ARG
    assert buckets(1, -1) == B.DOPT_E_ARG
    assert buckets(3, 0) == B.DOPT_OK  # an empty range needs no device
    assert buckets(1, 2) in (B.DOPT_E_STATE, B.DOPT_E_CUDA)
    assert B.lib().dopt_allreduce(L.handle, gp, 5, 1.0, None) == B.DOPT_E_ARG
    assert B.lib().dopt_allreduce(L.handle, gp, 0, float("nan"), None) == B.DOPT_E_ARG
    bad = (ctypes.c_void_p * 2)(0x10000, 0x20008)
    assert B.lib().dopt_allreduce(L.handle, bad, 0, 1.0, None) == B.DOPT_E_ALIGN
    assert B.lib().dopt_allreduce(L.handle, gp, 0, 1.0, None) in (B.DOPT_E_STATE, B.DOPT_E_CUDA)
    assert B.lib().dopt_step_allreduce(L.handle, ctypes.byref(cfg), 0, gp, 0, 0x30000, 0x40000,
                                       0x50000, gp, 1, None, None) == B.DOPT_E_ARG


@pytest.mark.parametrize("D,instances", [(8, 2), (8, 4), (8, 8), (6, 3), (16, 4), (12, 2)])
def test_range_map_with_instances_matches_oracle(lib, D, instances):
    """With several optimizer instances the buckets are sharded R = D/I
    ways: the layout equals the oracle's for R ranks."""
    rng = np.random.default_rng(D * 10 + instances)
    R = D // instances
    for _ in range(20):
        n = int(rng.integers(1, 40))
        sizes = [int(x) for x in rng.integers(0, 3000, n)]
        bucket = int(rng.choice([0, int(rng.integers(1, 9000))]))
        pad = int(rng.integers(1, 70))
        L = B.dopt_build_range_map(sizes, D, bucket, pad, instances=instances)
        O = oracle.range_map(sizes, R, bucket, pad)
        assert L.R == R and L.padded_numel == O.numel
        assert L.buckets() == list(zip(O.bucket_start.tolist(), O.bucket_end.tolist()))
        assert L.pieces() == O.pieces


def test_instances_errors(lib):
    for D, instances in ((8, 3), (4, -1), (6, 4)):
        with pytest.raises(B.DoptError) as e:
            B.dopt_build_range_map([10, 20], D, 0, 1, instances=instances)
        assert e.value.code == B.DOPT_E_ARG
    cfg = B.dopt_layout_cfg(4, 0, 1, 1, 7)  # reserved must be 0
    out = ctypes.c_void_p()
    sizes = (ctypes.c_int64 * 1)(10)
    assert B.lib().dopt_build_range_map(sizes, 1, None, ctypes.byref(cfg), ctypes.byref(out)) == B.DOPT_E_ARG
    L = B.dopt_build_range_map([10, 20], 8, 0, 1, instances=0)  # 0 means one instance
    assert L.padded_numel == B.dopt_build_range_map([10, 20], 8, 0, 1).padded_numel


def test_counted_step_argument_checks_before_cuda(lib):
    L = _lib_layout([100, 30], 2, 0, 8)
    cfg = B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)

    def call(counter=0x90000, grads=gp, flags=1):
        return B.lib().dopt_step_counted(L.handle, ctypes.byref(cfg), counter, grads, 0, 0x30000,
                                         0x40000, 0x50000, gp, flags, None, None)

    assert call(counter=None) == B.DOPT_E_ARG
    assert call(counter=0x90008) == B.DOPT_E_ALIGN
    assert call(grads=(ctypes.c_void_p * 2)(0x10000, 0)) == B.DOPT_E_ARG
    assert call(flags=8) == B.DOPT_E_ARG
    assert call() in (B.DOPT_E_STATE, B.DOPT_E_CUDA)  # nothing was launched
    assert ctypes.sizeof(ctypes.c_int64) * 8 == B.DOPT_STEP_COUNTER_BYTES


def test_stage_flag_checks_before_cuda(lib):
    """DOPT_STEP_STAGE: taken by the plain, bucket-range and counted steps
    for one-instance layouts with D in {1, 2, 4, 8, 16} and device grads,
    refused otherwise before anything reaches CUDA."""
    cfg = B.AdamConfig().to_c()
    st = (0x30000, 0x40000, 0x50000)
    stage = B.DOPT_STEP_GATHER | B.DOPT_STEP_STAGE
    for D, inst, ok in ((2, 1, True), (8, 1, True), (16, 1, True), (3, 1, False), (8, 2, False),
                        (32, 1, False)):
        L = B.dopt_build_range_map([100, 30], D, 0, 8, instances=inst)
        gp = (ctypes.c_void_p * D)(*[0x10000 * (r + 1) for r in range(D)])
        rcs = [B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp, stage, None,
                                 None),
               B.lib().dopt_step_buckets(L.handle, ctypes.byref(cfg), 1, 0, 1, gp, 0, *st, gp,
                                         stage, None, None),
               B.lib().dopt_step_counted(L.handle, ctypes.byref(cfg), 0x90000, gp, 0, *st, gp,
                                         stage, None, None)]
        for rc in rcs:
            if ok:  # past the flag checks: the next check needs the device
                assert rc in (B.DOPT_E_STATE, B.DOPT_E_CUDA), (D, inst, rc)
            else:
                assert rc == B.DOPT_E_ARG, (D, inst, rc)
    L = _lib_layout([100, 30], 2, 0, 8)
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    assert B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp,
                             stage | B.DOPT_STEP_HOST_GRADS, None, None) == B.DOPT_E_ARG
    assert B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp,
                             stage | B.DOPT_STEP_HOST_PARAMS, None, None) == B.DOPT_E_ARG
    # the other entry points do not take it
    assert B.lib().dopt_step_allreduce(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp, stage,
                                       None, None) == B.DOPT_E_ARG
    assert B.lib().dopt_step_clipped(L.handle, ctypes.byref(cfg), 1, 1.0, gp, 0, *st, gp, stage,
                                     0x70000, 0x80000, None, None) == B.DOPT_E_ARG


def test_host_params_flag_accepted_before_cuda(lib):
    """DOPT_STEP_HOST_PARAMS passes the flag checks of every step entry point
    (the pointers are resolved only once the device is needed)."""
    L = _lib_layout([100, 30], 2, 0, 8)
    cfg = B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    st = (0x30000, 0x40000, 0x50000)
    f = B.DOPT_STEP_GATHER | B.DOPT_STEP_HOST_PARAMS
    rcs = [B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp, f, None, None),
           B.lib().dopt_step_buckets(L.handle, ctypes.byref(cfg), 1, 0, 1, gp, 0, *st, gp, f,
                                     None, None),
           B.lib().dopt_step_allreduce(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp, f, None,
                                       None),
           B.lib().dopt_step_counted(L.handle, ctypes.byref(cfg), 0x90000, gp, 0, *st, gp, f,
                                     None, None),
           B.lib().dopt_step_clipped(L.handle, ctypes.byref(cfg), 1, 1.0, gp, 0, *st, gp, f,
                                     0x70000, 0x80000, None, None)]
    for rc in rcs:
        assert rc in (B.DOPT_E_STATE, B.DOPT_E_CUDA), rc


def test_skip_nonfinite_only_on_the_clipped_step(lib):
    L = _lib_layout([100, 30], 2, 0, 8)
    cfg = B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    skip = B.DOPT_STEP_GATHER | B.DOPT_STEP_SKIP_NONFINITE
    st = (0x30000, 0x40000, 0x50000)
    assert B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp, skip, None,
                             None) == B.DOPT_E_ARG
    assert B.lib().dopt_step_buckets(L.handle, ctypes.byref(cfg), 1, 0, 1, gp, 0, *st, gp, skip,
                                     None, None) == B.DOPT_E_ARG
    assert B.lib().dopt_step_allreduce(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp, skip,
                                       None, None) == B.DOPT_E_ARG
    assert B.lib().dopt_step_counted(L.handle, ctypes.byref(cfg), 0x90000, gp, 0, *st, gp, skip,
                                     None, None) == B.DOPT_E_ARG
    assert B.lib().dopt_step_clipped_noalloc(L.handle, ctypes.byref(cfg), 1, 1.0, gp, 0, *st, gp,
                                             skip, 0x70000, None, None) == B.DOPT_E_ARG
    assert B.lib().dopt_step_clipped(L.handle, ctypes.byref(cfg), 1, 1.0, gp, 0, *st, gp, skip,
                                     0x70000, 0x80000, None, None) in (B.DOPT_E_STATE,
                                                                       B.DOPT_E_CUDA)


def test_fp16_dtype_and_param_flag_accepted_before_cuda(lib):
    L = _lib_layout([100, 30], 2, 0, 8)
    cfg = B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    st = (0x30000, 0x40000, 0x50000)
    flags = B.DOPT_STEP_GATHER | B.DOPT_STEP_PARAMS_FP16
    assert B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, B.DOPT_FP16, *st, gp, flags,
                             None, None) in (B.DOPT_E_STATE, B.DOPT_E_CUDA)
    assert B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, 3, *st, gp, flags, None,
                             None) == B.DOPT_E_ARG
    assert B.lib().dopt_allreduce(L.handle, gp, B.DOPT_FP16, 1.0, None) in (B.DOPT_E_STATE,
                                                                           B.DOPT_E_CUDA)
    assert B.lib().dopt_step(L.handle, ctypes.byref(cfg), 1, gp, 0, *st, gp, 128, None,
                             None) == B.DOPT_E_ARG


def test_clipped_counted_argument_checks_before_cuda(lib):
    L = _lib_layout([100, 30], 2, 0, 8)
    cfg = B.AdamConfig().to_c()
    gp = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    st = (0x30000, 0x40000, 0x50000)

    def call(counter=0x90000, ws=0x80000, main=0x70000, flags=1):
        return B.lib().dopt_step_clipped_counted(L.handle, ctypes.byref(cfg), counter, 1.0, gp,
                                                 0, *st, gp, flags, main, ws, None, None)

    assert call(counter=None) == B.DOPT_E_ARG
    assert call(counter=0x90004) == B.DOPT_E_ALIGN
    assert call(ws=None) == B.DOPT_E_ARG
    assert call(main=None) == B.DOPT_E_ARG
    assert call(flags=128) == B.DOPT_E_ARG
    assert call(flags=1 | B.DOPT_STEP_SKIP_NONFINITE) in (B.DOPT_E_STATE, B.DOPT_E_CUDA)


def test_product_build_has_no_device_checks(lib):
    """dopt_device_checks answers DOPT_E_STATE in the product library (the
    checks exist only in the libdopt_checked.so test build) and needs no
    device to say so."""
    if B.LIB_PATH.endswith("libdopt_checked.so"):
        pytest.skip("this process runs the checked build")
    with pytest.raises(B.DoptError) as e:
        B.device_checks()
    assert e.value.code == B.DOPT_E_STATE
    assert "DOPT_DEVICE_CHECKS" in str(e.value)
    # nor the hook that makes the staged wait run out
    for extra in (0, 16):
        with pytest.raises(B.DoptError) as e:
            B.stage_wait_test(extra)
        assert e.value.code == B.DOPT_E_STATE
        assert "DOPT_DEVICE_CHECKS" in str(e.value)


def test_checked_build_compiles_and_exports_the_same_symbols():
    """The test build with device-side checks compiles for sm_103a, exports
    every symbol the header declares, and its dopt_device_checks reaches the
    CUDA runtime (an error without a device, not DOPT_E_STATE)."""
    import subprocess
    import sys

    path = libbuild.build(checked=True)
    assert path.endswith("libdopt_checked.so")
    checked = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(checked, n)]
    assert not missing, missing
    import torch

    if torch.cuda.is_available():
        return
    code = ("import zero_distributed_optimizer_gb300.binding as B\n"
            "assert B.LIB_PATH.endswith('libdopt_checked.so')\n"
            "try:\n    B.device_checks()\nexcept B.DoptError as e:\n    print('CODE', e.code)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       env=dict(os.environ, DOPT_CHECKED="1"), timeout=300)
    assert f"CODE {B.DOPT_E_CUDA}" in r.stdout, r.stdout + r.stderr


def test_stream_probe_argument_checks_before_cuda(lib):
    """The measurement probe refuses stream counts outside 0..16, no streams
    at all, NULL or misaligned buffers before anything reaches CUDA; zero
    vectors is a no-op."""
    vp = ctypes.c_void_p
    good = (vp * 2)(0x10000, 0x20000)
    probe = B.lib().dopt_stream_probe
    assert probe(17, 1, good, good, 16, None) == B.DOPT_E_ARG
    assert probe(0, 0, good, good, 16, None) == B.DOPT_E_ARG
    assert probe(-1, 1, good, good, 16, None) == B.DOPT_E_ARG
    assert probe(1, 1, None, good, 16, None) == B.DOPT_E_ARG
    assert probe(2, 0, (vp * 2)(0x10000, 0), None, 16, None) == B.DOPT_E_ARG
    assert probe(1, 1, (vp * 1)(0x10008), good, 16, None) == B.DOPT_E_ALIGN
    assert probe(1, 1, good, (vp * 1)(0x20004), 16, None) == B.DOPT_E_ALIGN
    assert probe(1, 1, good, good, -1, None) == B.DOPT_E_ARG
    assert probe(2, 2, good, good, 0, None) == B.DOPT_OK


def test_package_exports_the_binding():
    """Every public entry point and constant of the binding is importable
    from the package itself."""
    import zero_distributed_optimizer_gb300 as pkg

    internal = {"lib", "dataclass", "dopt_adam_cfg", "dopt_layout_cfg", "dopt_piece", "dopt_range"}
    public = [n for n in dir(B) if not n.startswith("_") and n not in internal
              and (n.startswith("DOPT_") or callable(getattr(B, n)))]
    missing = [n for n in public if not hasattr(pkg, n)]
    assert not missing, missing
