"""CPU oracle for the ZeRO-1 distributed-optimizer step (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product (the CUDA library and its Python binding) never does, and shares
no code with it.

The arithmetic lives in ``dopt_oracle.c`` (plain C, single thread, compiled
with ``-O2 -ffp-contract=off`` so that every fp32 multiply and add is rounded
on its own).  This module compiles it with gcc on first use and wraps it with
ctypes.  Each wrapper cites the passage of the Megatron-LM distributed
optimizer page ("04 · 分布式优化器") that it follows; the C file lists the
readings taken where the pages leave a step open.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dopt_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

ORC_OK, ORC_E_ARG, ORC_E_LAYOUT, ORC_E_NOMEM = 0, -1, -2, -6


class OracleError(RuntimeError):
    pass


class Range(ctypes.Structure):
    """Half-open interval [start, end) (distributed-optimizer page, §4.1 "Range")."""

    _fields_ = [("start", ctypes.c_int64), ("end", ctypes.c_int64)]


class Piece(ctypes.Structure):
    """One (param, rank) piece with its four ranges (distributed-optimizer page, §4.1 table)."""

    _fields_ = [
        ("gbuf_world", Range),
        ("gbuf_world_in_bucket", Range),
        ("gbuf_local", Range),
        ("param", Range),
        ("param_id", ctypes.c_int32),
        ("bucket_id", ctypes.c_int32),
        ("rank", ctypes.c_int32),
        ("unused", ctypes.c_int32),
    ]


class Adam(ctypes.Structure):
    _fields_ = [
        ("lr", ctypes.c_float),
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("weight_decay", ctypes.c_float),
        ("grad_scale", ctypes.c_float),
    ]


def _compile(src: str, out: str, extra_flags=()) -> None:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)


def lib_path_for(src: str = _SRC) -> str:
    """Build path keyed by the source hash, so an edited source is rebuilt."""
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read() + " ".join(CFLAGS).encode()).hexdigest()[:16]
    return os.path.join(_BUILD_DIR, f"liboracle_{digest}.so")


def build(force: bool = False) -> str:
    """Compile the oracle (gcc) if needed and return the shared-library path."""
    path = lib_path_for()
    if force or not os.path.exists(path):
        _compile(_SRC, path)
    return path


def _declare(lib) -> None:
    i64p = ctypes.POINTER(ctypes.c_int64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.orc_layout.restype = ctypes.c_int
    lib.orc_layout.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                               ctypes.c_int32, i64p, i64p, i32p, i64p, i64p, i32p, i64p]
    lib.orc_range_map.restype = ctypes.c_int
    lib.orc_range_map.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_int32, i64p, i64p, i32p, i64p, i64p, i32p, i64p,
                                  ctypes.POINTER(Piece), i32p]
    lib.orc_step.restype = ctypes.c_int
    lib.orc_step.argtypes = [
        i64p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
        ctypes.c_int32,
        ctypes.POINTER(Adam), ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p),
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p),
        ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
        ctypes.c_int32, ctypes.c_int32,
    ]
    lib.orc_grad_norm_sq.restype = ctypes.c_int
    lib.orc_grad_norm_sq.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int64,
                                     ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_void_p), ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_double)]
    lib.orc_count_nonfinite.restype = ctypes.c_int
    lib.orc_count_nonfinite.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                        ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p),
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.POINTER(ctypes.c_int64)]
    lib.orc_allreduce.restype = ctypes.c_int
    lib.orc_allreduce.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int64,
                                  ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                                  ctypes.POINTER(ctypes.c_void_p), ctypes.c_int64, ctypes.c_int64]
    lib.orc_clip_coef.restype = ctypes.c_float
    lib.orc_clip_coef.argtypes = [ctypes.c_double, ctypes.c_float]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.orc_f32_to_f16.restype = ctypes.c_uint16
    lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
    lib.orc_f16_to_f32.restype = ctypes.c_float
    lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f32.restype = ctypes.c_float
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_step_scalars.restype = None
    lib.orc_step_scalars.argtypes = [ctypes.POINTER(Adam), ctypes.c_int64,
                                     ctypes.POINTER(ctypes.c_float)]


def load(path: str | None = None):
    """Load the oracle library (building it first if needed)."""
    global _lib
    with _lock:
        if path is not None:
            lib = ctypes.CDLL(path)
            _declare(lib)
            return lib
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
        return _lib


GRAD_BF16, GRAD_F32, GRAD_F16 = 0, 1, 2


def _grad_type(grads) -> int:
    """Grad element type of the replicas: uint16 arrays hold bf16 bits,
    float16 arrays are IEEE binary16, float32 arrays fp32."""
    dt = grads[0].dtype
    code = {np.dtype(np.uint16): GRAD_BF16, np.dtype(np.float32): GRAD_F32,
            np.dtype(np.float16): GRAD_F16}.get(np.dtype(dt))
    if code is None:
        raise OracleError(f"grad dtype {dt}: use uint16 (bf16 bits), float16 or float32")
    for g in grads:
        if g.dtype != dt or not g.flags.c_contiguous:
            raise OracleError("grads must be contiguous and all of one dtype")
    return code


def _i64(a):
    a = np.ascontiguousarray(a, dtype=np.int64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


@dataclass
class OracleLayout:
    """Flat-buffer layout: param ranges, padded buckets, pieces."""

    param_start: np.ndarray
    param_end: np.ndarray
    param_bucket: np.ndarray
    bucket_start: np.ndarray
    bucket_end: np.ndarray
    numel: int
    pieces: list  # list of dicts, sorted by (bucket, rank, gbuf_world.start)

    @property
    def n_buckets(self) -> int:
        return len(self.bucket_start)


def range_map(sizes, D: int, bucket_elems: int, pad_unit: int, lib=None) -> OracleLayout:
    """Layout + four-way range map (distributed-optimizer page, §2, §3 and §4.1)."""
    lib = lib or load()
    sizes_a, sizes_p = _i64(sizes)
    n = len(sizes_a)
    cap = max(n, 1)
    ps = np.zeros(cap, np.int64)
    pe = np.zeros(cap, np.int64)
    pb = np.zeros(cap, np.int32)
    bs = np.zeros(cap, np.int64)
    be = np.zeros(cap, np.int64)
    nb = ctypes.c_int32(0)
    numel = ctypes.c_int64(0)
    pieces = (Piece * (n + D * cap + 1))()
    npc = ctypes.c_int32(0)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    rc = lib.orc_range_map(sizes_p, n, D, bucket_elems, pad_unit,
                           ps.ctypes.data_as(i64p), pe.ctypes.data_as(i64p),
                           pb.ctypes.data_as(i32p), bs.ctypes.data_as(i64p),
                           be.ctypes.data_as(i64p), ctypes.byref(nb), ctypes.byref(numel),
                           pieces, ctypes.byref(npc))
    if rc != ORC_OK:
        raise OracleError(f"orc_range_map failed: {rc}")
    out = []
    for i in range(npc.value):
        pc = pieces[i]
        out.append({
            "gbuf_world": (pc.gbuf_world.start, pc.gbuf_world.end),
            "gbuf_world_in_bucket": (pc.gbuf_world_in_bucket.start, pc.gbuf_world_in_bucket.end),
            "gbuf_local": (pc.gbuf_local.start, pc.gbuf_local.end),
            "param": (pc.param.start, pc.param.end),
            "param_id": pc.param_id,
            "bucket_id": pc.bucket_id,
            "rank": pc.rank,
        })
    return OracleLayout(ps[:n].copy(), pe[:n].copy(), pb[:n].copy(), bs[:nb.value].copy(),
                        be[:nb.value].copy(), int(numel.value), out)


def range_map_rc(sizes, D: int, bucket_elems: int, pad_unit: int, lib=None) -> int:
    """Status code of the layout call alone (for error-path tests)."""
    lib = lib or load()
    sizes_a, sizes_p = _i64(sizes)
    n = len(sizes_a)
    cap = max(n, 1)
    bufs = [np.zeros(cap, np.int64) for _ in range(2)] + [np.zeros(cap, np.int32)]
    bb = [np.zeros(cap, np.int64) for _ in range(2)]
    nb = ctypes.c_int32(0)
    numel = ctypes.c_int64(0)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    return lib.orc_layout(sizes_p, n, D, bucket_elems, pad_unit,
                          bufs[0].ctypes.data_as(i64p), bufs[1].ctypes.data_as(i64p),
                          bufs[2].ctypes.data_as(i32p), bb[0].ctypes.data_as(i64p),
                          bb[1].ctypes.data_as(i64p), ctypes.byref(nb), ctypes.byref(numel))


def make_adam(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, grad_scale=1.0) -> Adam:
    return Adam(lr, beta1, beta2, eps, weight_decay, grad_scale)


def step(sizes, wd_mask, D: int, bucket_elems: int, pad_unit: int, adam: Adam, t: int,
         grads, master, exp_avg, exp_avg_sq, params, gather: bool = True,
         main_grad_out=None, window=None, clip_coef: float = 1.0, instances: int = 1,
         round_grad: bool = False, lib=None) -> None:
    """One ZeRO-1 step for all D simulated ranks, in place on numpy arrays.

    grads: D arrays (uint16 bf16 bits or float32); master/exp_avg/exp_avg_sq:
    float32; params: D uint16 arrays (bf16 bits); main_grad_out: optional
    float32.  All are buffer-indexed and cover ``window = (w0, w1)`` (default:
    the whole padded buffer).  Follows the distributed-optimizer page, §4.2 (reduce-scatter), §4.3
    (main grads, Adam, write-back) and §4.4 (all-gather).  ``clip_coef``
    (from :func:`clip_coef`) multiplies every reduced grad before Adam.
    ``instances`` > 1 splits the D ranks into that many optimizer instances
    (distributed-optimizer page, §5): reduce-scatter inside each, then a sum across instances.
    ``round_grad`` rounds every reduced grad to the grad type first.
    """
    lib = lib or load()
    sizes_a, sizes_p = _i64(sizes)
    n = len(sizes_a)
    if len(grads) != D or len(params) != D:
        raise OracleError("need D grad and D param arrays")
    grad_type = _grad_type(grads)
    for a in (master, exp_avg, exp_avg_sq):
        if a.dtype != np.float32 or not a.flags.c_contiguous:
            raise OracleError("state arrays must be contiguous float32")
    param_is_f16 = params[0].dtype == np.float16
    for p in params:
        if p.dtype != params[0].dtype or p.dtype not in (np.uint16, np.float16) \
                or not p.flags.c_contiguous:
            raise OracleError("params must be contiguous, all uint16 (bf16 bits) or all float16")
    if window is None:
        w0, w1 = 0, len(master)
    else:
        w0, w1 = int(window[0]), int(window[1])
    span = w1 - w0
    for a in list(grads) + [master, exp_avg, exp_avg_sq] + list(params):
        if len(a) != span:
            raise OracleError("array length must equal the window length")
    if main_grad_out is not None and (main_grad_out.dtype != np.float32 or len(main_grad_out) != span):
        raise OracleError("main_grad_out must be float32 of the window length")
    wd = None
    if wd_mask is not None:
        wd = np.ascontiguousarray(wd_mask, dtype=np.uint8)
    gp = (ctypes.c_void_p * D)(*[g.ctypes.data for g in grads])
    pp = (ctypes.c_void_p * D)(*[p.ctypes.data for p in params])
    rc = lib.orc_step(sizes_p, n, None if wd is None else wd.ctypes.data, D, int(instances),
                      bucket_elems,
                      pad_unit, ctypes.byref(adam), t, grad_type, gp,
                      master.ctypes.data, exp_avg.ctypes.data, exp_avg_sq.ctypes.data, pp,
                      int(bool(gather)),
                      None if main_grad_out is None else main_grad_out.ctypes.data, w0, w1,
                      float(clip_coef), int(bool(round_grad)), int(param_is_f16))
    if rc != ORC_OK:
        raise OracleError(f"orc_step failed: {rc}")


def grad_norm_sq(sizes, D: int, bucket_elems: int, pad_unit: int, grad_scale: float, grads,
                 window=None, instances: int = 1, round_grad: bool = False, lib=None) -> float:
    """Sum of squares of the reduced grads over the owned elements of the
    window (tutorial §8.3 global norm), accumulated in double."""
    lib = lib or load()
    sizes_a, sizes_p = _i64(sizes)
    grad_type = _grad_type(grads)
    span = len(grads[0])
    w0, w1 = (0, span) if window is None else (int(window[0]), int(window[1]))
    if w1 - w0 != span or len(grads) != D:
        raise OracleError("grads must be D arrays of the window length")
    gp = (ctypes.c_void_p * D)(*[g.ctypes.data for g in grads])
    out = ctypes.c_double(0.0)
    rc = lib.orc_grad_norm_sq(sizes_p, len(sizes_a), D, int(instances), bucket_elems, pad_unit,
                              float(grad_scale), grad_type, gp, w0, w1,
                              int(bool(round_grad)), ctypes.byref(out))
    if rc != ORC_OK:
        raise OracleError(f"orc_grad_norm_sq failed: {rc}")
    return float(out.value)


def count_nonfinite(sizes, D: int, bucket_elems: int, pad_unit: int, grad_scale: float, grads,
                    window=None, instances: int = 1, round_grad: bool = False, lib=None) -> int:
    """Owned elements of the window whose reduced grad is Inf or NaN (the
    non-finite check, reading R13 of the C file; the tutorial's §8.2 notes
    that FP16 overflows easily)."""
    lib = lib or load()
    sizes_a, sizes_p = _i64(sizes)
    grad_type = _grad_type(grads)
    span = len(grads[0])
    w0, w1 = (0, span) if window is None else (int(window[0]), int(window[1]))
    if w1 - w0 != span or len(grads) != D:
        raise OracleError("grads must be D arrays of the window length")
    gp = (ctypes.c_void_p * D)(*[g.ctypes.data for g in grads])
    out = ctypes.c_int64(0)
    rc = lib.orc_count_nonfinite(sizes_p, len(sizes_a), D, int(instances), bucket_elems,
                                 pad_unit, float(grad_scale), grad_type, gp, w0, w1,
                                 int(bool(round_grad)), ctypes.byref(out))
    if rc != ORC_OK:
        raise OracleError(f"orc_count_nonfinite failed: {rc}")
    return int(out.value)


def allreduce(sizes, D: int, bucket_elems: int, pad_unit: int, grad_scale: float, grads,
              window=None, instances: int = 1, lib=None) -> None:
    """All-reduce of the grads in place (distributed-optimizer page, §5 force_all_reduce; the
    tutorial's AllReduce = reduce-scatter + all-gather): every replica gets
    the reduced grad at every owned element, rounded to the grad type."""
    lib = lib or load()
    sizes_a, sizes_p = _i64(sizes)
    grad_type = _grad_type(grads)
    span = len(grads[0])
    w0, w1 = (0, span) if window is None else (int(window[0]), int(window[1]))
    if w1 - w0 != span or len(grads) != D:
        raise OracleError("grads must be D arrays of the window length")
    gp = (ctypes.c_void_p * D)(*[g.ctypes.data for g in grads])
    rc = lib.orc_allreduce(sizes_p, len(sizes_a), D, int(instances), bucket_elems, pad_unit,
                           float(grad_scale),
                           grad_type, gp, w0, w1)
    if rc != ORC_OK:
        raise OracleError(f"orc_allreduce failed: {rc}")


def clip_coef(norm_sq: float, max_norm: float, lib=None) -> float:
    """min(1, max_norm / (sqrt(norm_sq) + 1e-6)), rounded to float once."""
    lib = lib or load()
    return float(lib.orc_clip_coef(float(norm_sq), float(max_norm)))


def f32_to_f16(x, lib=None) -> np.ndarray:
    """Round fp32 values to IEEE binary16 bits (nearest, ties to even)."""
    lib = lib or load()
    x = np.asarray(x, np.float32).ravel()
    return np.array([lib.orc_f32_to_f16(float(v)) for v in x], np.uint16)


def f16_to_f32(bits, lib=None) -> np.ndarray:
    """Widen IEEE binary16 bits to fp32 (exact)."""
    lib = lib or load()
    bits = np.asarray(bits, np.uint16).ravel()
    return np.array([lib.orc_f16_to_f32(int(b)) for b in bits], np.float32)


def f32_to_bf16(x, lib=None) -> np.ndarray:
    """Round fp32 values to bf16 bits (nearest, ties to even), element by element."""
    lib = lib or load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def bf16_to_f32(h, lib=None) -> np.ndarray:
    lib = lib or load()
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([lib.orc_bf16_to_f32(int(v)) for v in h], dtype=np.float32)


def step_scalars(adam: Adam, t: int, lib=None) -> dict:
    """The per-step fp32 scalars of the AdamW update (bias corrections etc.)."""
    lib = lib or load()
    out = (ctypes.c_float * 9)()
    lib.orc_step_scalars(ctypes.byref(adam), t, out)
    keys = ["b1", "b2", "one_minus_b1", "one_minus_b2", "decay", "step_size", "bc2_sqrt",
            "eps", "scale"]
    return dict(zip(keys, list(out)))
