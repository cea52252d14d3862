"""Python binding of the dopt C ABI (include/dopt.h): argument marshalling only.

Every function here checks what the C ABI cannot (tensor device, dtype,
length, contiguity) and passes raw pointers and sizes to libdopt.so; all of
the step's work runs in the library's CUDA kernels.  There is no fallback:
if libdopt.so is missing or fails to load, every call raises.

Names follow the C entry points: ``dopt_build_range_map``, ``dopt_step``,
``dopt_gather``.
"""
from __future__ import annotations

import contextlib
import ctypes
import functools
import os
import threading
from dataclasses import dataclass

PKG = os.path.dirname(os.path.abspath(__file__))
# DOPT_CHECKED=1 loads the test build with the kernels' device-side index
# checks (libdopt_checked.so, see dopt_device_checks in dopt.h) instead.
LIB_PATH = os.path.join(PKG, "libdopt_checked.so" if os.environ.get("DOPT_CHECKED") == "1"
                        else "libdopt.so")

DOPT_OK = 0
DOPT_E_ARG = -1
DOPT_E_LAYOUT = -2
DOPT_E_ALIGN = -3
DOPT_E_CUDA = -4
DOPT_E_STATE = -5
DOPT_E_NOMEM = -6
DOPT_CHECK_INDEX = 1
DOPT_CHECK_ALIGN = 2
DOPT_MAX_D = 64
DOPT_BF16 = 0
DOPT_FP32 = 1
DOPT_FP16 = 2
DOPT_STEP_GATHER = 1
DOPT_STEP_HOST_GRADS = 2
DOPT_STEP_ROUND_GRAD = 4
DOPT_STEP_SKIP_NONFINITE = 8
DOPT_STEP_PARAMS_FP16 = 16
DOPT_STEP_STAGE = 32
DOPT_STEP_HOST_PARAMS = 64
DOPT_CLIP_WORKSPACE_BYTES = 16384
DOPT_STEP_COUNTER_BYTES = 64  # sizeof(dopt_step_counter)
DOPT_COUNTER_BAD_STEP = 1

_ERROR_NAMES = {DOPT_E_ARG: "DOPT_E_ARG", DOPT_E_LAYOUT: "DOPT_E_LAYOUT",
                DOPT_E_ALIGN: "DOPT_E_ALIGN", DOPT_E_CUDA: "DOPT_E_CUDA",
                DOPT_E_STATE: "DOPT_E_STATE", DOPT_E_NOMEM: "DOPT_E_NOMEM"}


class DoptError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{_ERROR_NAMES.get(code, code)}: {message}")
        self.code = code


class dopt_range(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int64), ("end", ctypes.c_int64)]


class dopt_piece(ctypes.Structure):
    _fields_ = [("gbuf_world", dopt_range), ("gbuf_world_in_bucket", dopt_range),
                ("gbuf_local", dopt_range), ("param", dopt_range), ("param_id", ctypes.c_int32),
                ("bucket_id", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class dopt_layout_cfg(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int32), ("bucket_elems", ctypes.c_int64),
                ("pad_unit", ctypes.c_int32), ("instances", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class dopt_adam_cfg(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("grad_scale", ctypes.c_float)]


_lock = threading.Lock()
_lib = None


def _declare(lib):
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    lib.dopt_build_range_map.restype = ctypes.c_int
    lib.dopt_build_range_map.argtypes = [P(ctypes.c_int64), ctypes.c_int32, P(ctypes.c_uint8),
                                         P(dopt_layout_cfg), P(vp)]
    lib.dopt_layout_query.restype = ctypes.c_int
    lib.dopt_layout_query.argtypes = [vp, P(ctypes.c_int64), P(ctypes.c_int32), P(ctypes.c_int32)]
    lib.dopt_layout_buckets.restype = ctypes.c_int
    lib.dopt_layout_buckets.argtypes = [vp, P(dopt_range)]
    lib.dopt_layout_pieces.restype = ctypes.c_int
    lib.dopt_layout_pieces.argtypes = [vp, P(dopt_piece)]
    lib.dopt_layout_param_offsets.restype = ctypes.c_int
    lib.dopt_layout_param_offsets.argtypes = [vp, P(dopt_range)]
    lib.dopt_layout_param_ranges.restype = ctypes.c_int
    lib.dopt_layout_param_ranges.argtypes = [vp, P(dopt_range)]
    lib.dopt_layout_to_device.restype = ctypes.c_int
    lib.dopt_layout_to_device.argtypes = [vp]
    lib.dopt_layout_free.restype = None
    lib.dopt_layout_free.argtypes = [vp]
    lib.dopt_step.restype = ctypes.c_int
    lib.dopt_step.argtypes = [vp, P(dopt_adam_cfg), ctypes.c_int64, P(vp), ctypes.c_int, vp, vp,
                              vp, P(vp), ctypes.c_uint32, vp, vp]
    lib.dopt_step_counted.restype = ctypes.c_int
    lib.dopt_step_counted.argtypes = [vp, P(dopt_adam_cfg), vp, P(vp), ctypes.c_int, vp, vp, vp,
                                      P(vp), ctypes.c_uint32, vp, vp]
    lib.dopt_step_clipped.restype = ctypes.c_int
    lib.dopt_step_clipped.argtypes = [vp, P(dopt_adam_cfg), ctypes.c_int64, ctypes.c_float, P(vp),
                                      ctypes.c_int, vp, vp, vp, P(vp), ctypes.c_uint32, vp, vp,
                                      vp, vp]
    lib.dopt_step_clipped_counted.restype = ctypes.c_int
    lib.dopt_step_clipped_counted.argtypes = [vp, P(dopt_adam_cfg), vp, ctypes.c_float, P(vp),
                                              ctypes.c_int, vp, vp, vp, P(vp), ctypes.c_uint32,
                                              vp, vp, vp, vp]
    lib.dopt_step_clipped_noalloc.restype = ctypes.c_int
    lib.dopt_step_clipped_noalloc.argtypes = [vp, P(dopt_adam_cfg), ctypes.c_int64, ctypes.c_float,
                                              P(vp), ctypes.c_int, vp, vp, vp, P(vp),
                                              ctypes.c_uint32, vp, vp, vp]
    lib.dopt_step_buckets.restype = ctypes.c_int
    lib.dopt_step_buckets.argtypes = [vp, P(dopt_adam_cfg), ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_int32, P(vp), ctypes.c_int, vp, vp, vp, P(vp),
                                      ctypes.c_uint32, vp, vp]
    lib.dopt_step_allreduce.restype = ctypes.c_int
    lib.dopt_step_allreduce.argtypes = [vp, P(dopt_adam_cfg), ctypes.c_int64, P(vp), ctypes.c_int,
                                        vp, vp, vp, P(vp), ctypes.c_uint32, vp, vp]
    lib.dopt_allreduce.restype = ctypes.c_int
    lib.dopt_allreduce.argtypes = [vp, P(vp), ctypes.c_int, ctypes.c_float, vp]
    lib.dopt_gather.restype = ctypes.c_int
    lib.dopt_gather.argtypes = [vp, P(vp), vp]
    lib.dopt_stream_probe.restype = ctypes.c_int
    lib.dopt_stream_probe.argtypes = [ctypes.c_int32, ctypes.c_int32, P(vp), P(vp), ctypes.c_int64,
                                      vp]
    lib.dopt_stage_timeouts.restype = ctypes.c_int
    lib.dopt_stage_timeouts.argtypes = [ctypes.c_int, P(ctypes.c_uint32)]
    lib.dopt_stage_wait_test.restype = ctypes.c_int
    lib.dopt_stage_wait_test.argtypes = [ctypes.c_uint32]
    lib.dopt_device_checks.restype = ctypes.c_int
    lib.dopt_device_checks.argtypes = [ctypes.c_int, P(ctypes.c_uint32), P(ctypes.c_int64)]
    lib.dopt_last_error.restype = ctypes.c_char_p
    lib.dopt_last_error.argtypes = []
    lib.dopt_version.restype = ctypes.c_char_p
    lib.dopt_version.argtypes = []


def lib():
    """The loaded libdopt.so.  Raises if it has not been built."""
    global _lib
    loaded = _lib
    if loaded is not None:
        return loaded
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m zero_distributed_optimizer_gb300.build` (no fallback exists)")
            handle = ctypes.CDLL(LIB_PATH)
            _declare(handle)
            _lib = handle
        return _lib


def device_checks(reset: bool = False):
    """(flags, first_bad) of the device-side checks in the checked test
    build (DOPT_CHECK_* bits, 0 if every check passed; the first failing
    element index, -1 if none); reset clears them.  Raises DoptError with
    DOPT_E_STATE in the product build, which has no checks."""
    flags, first = ctypes.c_uint32(0), ctypes.c_int64(0)
    _check(lib().dopt_device_checks(1 if reset else 0, ctypes.byref(flags), ctypes.byref(first)))
    return flags.value, first.value


def dopt_stream_probe(read_buffers, write_buffers, stream=None) -> None:
    """One launch of the stream probe (dopt_stream_probe in dopt.h): vector i
    of every read buffer in, their XOR with a seed of i to vector i of every
    write buffer.  Buffers: CUDA tensors of one device, contiguous, the same
    byte size (a multiple of 16).  Time it with CUDA events."""
    import torch

    bufs = list(read_buffers) + list(write_buffers)
    if not bufs:
        raise DoptError(DOPT_E_ARG, "no buffers")
    nbytes = bufs[0].numel() * bufs[0].element_size()
    for b in bufs:
        if (b.device.type != "cuda" or b.device != bufs[0].device or not b.is_contiguous()
                or b.numel() * b.element_size() != nbytes or nbytes % 16):
            raise DoptError(DOPT_E_ARG, "probe buffers must be contiguous CUDA tensors of one "
                            "device and one byte size, a multiple of 16")
    rp = (ctypes.c_void_p * max(len(read_buffers), 1))(*[b.data_ptr() for b in read_buffers])
    wp = (ctypes.c_void_p * max(len(write_buffers), 1))(*[b.data_ptr() for b in write_buffers])
    with _on(bufs[0].device):
        _check(lib().dopt_stream_probe(len(read_buffers), len(write_buffers), rp, wp, nbytes // 16,
                                       _stream_handle(stream)))


def stage_timeouts(reset: bool = False) -> int:
    """Staged CTAs (DOPT_STEP_STAGE) on the current device whose bulk copies
    ran past their time limit and skipped their tile (0 unless a bulk copy
    failed to complete); reset clears the count."""
    c = ctypes.c_uint32(0)
    _check(lib().dopt_stage_timeouts(1 if reset else 0, ctypes.byref(c)))
    return c.value


def stage_wait_test(extra_bytes: int) -> None:
    """Test build only (dopt_stage_wait_test in dopt.h): staged CTAs
    launched afterwards expect `extra_bytes` that no copy delivers, so their
    bounded wait runs out; 0 restores normal staging.  Raises DoptError
    with DOPT_E_STATE in the product build."""
    _check(lib().dopt_stage_wait_test(ctypes.c_uint32(int(extra_bytes))))


def _check(rc: int):
    if rc != DOPT_OK:
        raise DoptError(rc, lib().dopt_last_error().decode(errors="replace"))


@dataclass(frozen=True)
class AdamConfig:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    grad_scale: float = 1.0

    def to_c(self) -> dopt_adam_cfg:
        """The C struct (one per distinct config, kept: the library only reads it)."""
        return _adam_c(self)


@functools.lru_cache(maxsize=256)
def _adam_c(adam: AdamConfig) -> dopt_adam_cfg:
    return dopt_adam_cfg(adam.lr, adam.beta1, adam.beta2, adam.eps, adam.weight_decay,
                         adam.grad_scale)


def _on(device):
    """torch.cuda.device(device), or nothing when it is already current."""
    import torch

    if device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


class Layout:
    """Owner of a dopt_layout handle (freed with the object)."""

    def __init__(self, handle: int, D: int, n_params: int, instances: int = 1):
        self._h = ctypes.c_void_p(handle)
        self.D = D
        self.instances = instances
        self.R = D // instances  # ranks per instance: the shard count of a bucket
        self.n_params = n_params
        numel = ctypes.c_int64()
        nb = ctypes.c_int32()
        npc = ctypes.c_int32()
        _check(lib().dopt_layout_query(self._h, ctypes.byref(numel), ctypes.byref(nb),
                                       ctypes.byref(npc)))
        self.padded_numel = int(numel.value)
        self.n_buckets = int(nb.value)
        self.n_pieces = int(npc.value)
        self._device = None

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise DoptError(DOPT_E_ARG, "layout already freed")
        return self._h

    def buckets(self) -> list:
        arr = (dopt_range * max(self.n_buckets, 1))()
        _check(lib().dopt_layout_buckets(self.handle, arr))
        return [(arr[i].start, arr[i].end) for i in range(self.n_buckets)]

    def param_offsets(self) -> list:
        """Each param's [start, end) in the flat buffer (dopt_layout_param_offsets)."""
        arr = (dopt_range * max(self.n_params, 1))()
        _check(lib().dopt_layout_param_offsets(self.handle, arr))
        return [(arr[i].start, arr[i].end) for i in range(self.n_params)]

    def param_ranges(self) -> list:
        """The same list through the call's earlier name, dopt_layout_param_ranges."""
        arr = (dopt_range * max(self.n_params, 1))()
        _check(lib().dopt_layout_param_ranges(self.handle, arr))
        return [(arr[i].start, arr[i].end) for i in range(self.n_params)]

    def pieces(self) -> list:
        arr = (dopt_piece * max(self.n_pieces, 1))()
        _check(lib().dopt_layout_pieces(self.handle, arr))
        out = []
        for i in range(self.n_pieces):
            pc = arr[i]
            out.append({
                "gbuf_world": (pc.gbuf_world.start, pc.gbuf_world.end),
                "gbuf_world_in_bucket": (pc.gbuf_world_in_bucket.start, pc.gbuf_world_in_bucket.end),
                "gbuf_local": (pc.gbuf_local.start, pc.gbuf_local.end),
                "param": (pc.param.start, pc.param.end),
                "param_id": pc.param_id, "bucket_id": pc.bucket_id, "rank": pc.rank,
            })
        return out

    def to_device(self, device=None) -> "Layout":
        """Copy the kernel tables to `device` (default: the current device)."""
        import torch

        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        with torch.cuda.device(dev):
            _check(lib().dopt_layout_to_device(self.handle))
        self._device = dev
        return self

    def free(self):
        if self._h:
            lib().dopt_layout_free(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def dopt_build_range_map(param_sizes, D: int, bucket_elems: int = 0, pad_unit: int = 1,
                         wd_mask=None, instances: int = 1) -> Layout:
    """Flat-buffer layout and four-way range map (host only, no CUDA call).
    ``instances`` > 1 groups the D ranks into that many optimizer instances
    of D // instances ranks each (distributed-optimizer page, §5)."""
    n = len(param_sizes)
    sizes = (ctypes.c_int64 * max(n, 1))(*[int(s) for s in param_sizes])
    wd = None
    if wd_mask is not None:
        if len(wd_mask) != n:
            raise DoptError(DOPT_E_ARG, "wd_mask length differs from param_sizes")
        wd = (ctypes.c_uint8 * max(n, 1))(*[1 if x else 0 for x in wd_mask])
    cfg = dopt_layout_cfg(int(D), int(bucket_elems), int(pad_unit), int(instances), 0)
    out = ctypes.c_void_p()
    _check(lib().dopt_build_range_map(sizes, n, wd, ctypes.byref(cfg), ctypes.byref(out)))
    return Layout(out.value, int(D), n, max(int(instances), 1))


def _stream_handle(stream):
    """The cudaStream_t of `stream`, or of torch's current stream on the
    current device (the callers run with the tensors' device current)."""
    import torch

    if stream is None:
        # torch's raw query of the current stream, where it exists: a few
        # tenths of a microsecond against ~3 us for building a Stream object
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_tensor(t, name, dtype, numel, device):
    index = device.index if device.type == "cuda" else -1
    if (index is not None and t.dtype is dtype and t.get_device() == index and t.is_contiguous()
            and t.numel() >= numel):
        return  # the common case, without building device objects
    if t.device != device:
        raise DoptError(DOPT_E_ARG, f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise DoptError(DOPT_E_ARG, f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous() or t.numel() < numel:
        raise DoptError(DOPT_E_ARG, f"{name} must be contiguous with >= {numel} elements")


def _flags(gather: bool, host_grads: bool = False, round_grad: bool = False,
           stage: bool = False) -> int:
    return ((DOPT_STEP_GATHER if gather else 0) | (DOPT_STEP_HOST_GRADS if host_grads else 0)
            | (DOPT_STEP_ROUND_GRAD if round_grad else 0) | (DOPT_STEP_STAGE if stage else 0))


def _grad_code(gdt) -> int:
    """dopt_dtype of a torch grad dtype."""
    import torch

    codes = {torch.bfloat16: DOPT_BF16, torch.float32: DOPT_FP32, torch.float16: DOPT_FP16}
    if gdt not in codes:
        raise DoptError(DOPT_E_ARG, f"grad dtype {gdt} is not bf16, fp16 or fp32")
    return codes[gdt]


def _param_flag(param_replicas, N, device, host_params: bool = False) -> int:
    """Check the param replicas (all bf16 or all fp16; with host_params each
    on the step's device or a pinned CPU tensor) and return the flags for
    them."""
    import torch

    pdt = param_replicas[0].dtype
    if pdt not in (torch.bfloat16, torch.float16):
        raise DoptError(DOPT_E_ARG, f"param dtype {pdt} is not bf16 or fp16")
    for i, p in enumerate(param_replicas):
        if host_params and p.device.type == "cpu":
            if not p.is_pinned():
                raise DoptError(DOPT_E_ARG, f"param_replicas[{i}] must be on {device} or pinned")
            _check_tensor(p, f"param_replicas[{i}]", pdt, N, p.device)
        else:
            _check_tensor(p, f"param_replicas[{i}]", pdt, N, device)
    return ((DOPT_STEP_PARAMS_FP16 if pdt == torch.float16 else 0)
            | (DOPT_STEP_HOST_PARAMS if host_params else 0))


def _check_grads(grad_replicas, gdt, N, device, host_grads):
    """Device grads on the step's device, or (host_grads) pinned CPU tensors
    that the library reads in place."""
    for i, g in enumerate(grad_replicas):
        if host_grads:
            if g.device.type != "cpu" or not g.is_pinned():
                raise DoptError(DOPT_E_ARG, f"grad_replicas[{i}] must be a pinned CPU tensor")
            _check_tensor(g, f"grad_replicas[{i}]", gdt, N, g.device)
        else:
            _check_tensor(g, f"grad_replicas[{i}]", gdt, N, device)


def _step_pointers(layout: Layout, grad_replicas, master, exp_avg, exp_avg_sq, param_replicas,
                   main_grad_out, host_grads=False, host_params=False):
    import torch

    D = layout.D
    if len(grad_replicas) != D or len(param_replicas) != D:
        raise DoptError(DOPT_E_ARG, f"need {D} grad and {D} param replicas")
    N = layout.padded_numel
    device = master.device
    if device.type != "cuda":
        raise DoptError(DOPT_E_ARG, "the step needs CUDA tensors (no CPU path exists)")
    gdt = grad_replicas[0].dtype
    dt = _grad_code(gdt)
    _check_grads(grad_replicas, gdt, N, device, host_grads)
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq)):
        _check_tensor(t, name, torch.float32, N, device)
    pflag = _param_flag(param_replicas, N, device, host_params)
    if main_grad_out is not None:
        _check_tensor(main_grad_out, "main_grad_out", torch.float32, N, device)
    gp = (ctypes.c_void_p * D)(*[g.data_ptr() for g in grad_replicas])
    pp = (ctypes.c_void_p * D)(*[p.data_ptr() for p in param_replicas])
    mg = None if main_grad_out is None else main_grad_out.data_ptr()
    return device, gp, pp, dt, mg, pflag


def dopt_step_buckets(layout: Layout, adam: AdamConfig, step: int, first_bucket: int,
                      n_buckets: int, grad_replicas, master, exp_avg, exp_avg_sq,
                      param_replicas, gather: bool = True, main_grad_out=None,
                      stream=None, host_grads: bool = False, round_grad: bool = False,
                      stage: bool = False) -> None:
    """The step over buckets [first_bucket, first_bucket + n_buckets) only."""
    import torch

    device, gp, pp, dt, mg, pflag = _step_pointers(layout, grad_replicas, master, exp_avg, exp_avg_sq,
                                            param_replicas, main_grad_out, host_grads)
    flags = _flags(gather, host_grads, round_grad, stage) | pflag
    cfg = adam.to_c()
    with _on(device):
        _check(lib().dopt_step_buckets(
            layout.handle, ctypes.byref(cfg), int(step), int(first_bucket), int(n_buckets), gp,
            dt, master.data_ptr(), exp_avg.data_ptr(), exp_avg_sq.data_ptr(), pp, flags, mg,
            _stream_handle(stream)))


def dopt_step_allreduce(layout: Layout, adam: AdamConfig, step: int, grad_replicas, master,
                        exp_avg, exp_avg_sq, param_replicas, gather: bool = True,
                        main_grad_out=None, stream=None, round_grad: bool = False) -> None:
    """The step that also all-reduces the grads in place (force_all_reduce)."""
    import torch

    device, gp, pp, dt, mg, pflag = _step_pointers(layout, grad_replicas, master, exp_avg, exp_avg_sq,
                                            param_replicas, main_grad_out)
    cfg = adam.to_c()
    with _on(device):
        _check(lib().dopt_step_allreduce(
            layout.handle, ctypes.byref(cfg), int(step), gp, dt, master.data_ptr(),
            exp_avg.data_ptr(), exp_avg_sq.data_ptr(), pp,
            _flags(gather, round_grad=round_grad) | pflag,
            mg, _stream_handle(stream)))


def dopt_allreduce(layout: Layout, grad_replicas, grad_scale: float, stream=None) -> None:
    """All-reduce of the D grad replicas in place (scaled, fp32 rank order,
    rounded back to the grad type)."""
    import torch

    D = layout.D
    if len(grad_replicas) != D:
        raise DoptError(DOPT_E_ARG, f"need {D} grad replicas")
    device = grad_replicas[0].device
    if device.type != "cuda":
        raise DoptError(DOPT_E_ARG, "dopt_allreduce needs CUDA tensors")
    gdt = grad_replicas[0].dtype
    dt = _grad_code(gdt)
    for i, g in enumerate(grad_replicas):
        _check_tensor(g, f"grad_replicas[{i}]", gdt, layout.padded_numel, device)
    gp = (ctypes.c_void_p * D)(*[g.data_ptr() for g in grad_replicas])
    with _on(device):
        _check(lib().dopt_allreduce(layout.handle, gp, dt, float(grad_scale),
                                    _stream_handle(stream)))


def dopt_step(layout: Layout, adam: AdamConfig, step: int, grad_replicas, master, exp_avg,
              exp_avg_sq, param_replicas, gather: bool = True, main_grad_out=None,
              stream=None, host_grads: bool = False, round_grad: bool = False,
              stage: bool = False, host_params: bool = False) -> None:
    """One fused ZeRO-1 step (reduce-scatter, AdamW, write-back, all-gather).

    grad_replicas: D bf16 or fp32 CUDA tensors (or, with host_grads, pinned
    CPU tensors the kernel reads in place); master/exp_avg/exp_avg_sq: fp32;
    param_replicas: D bf16; main_grad_out: optional fp32.  Each holds at
    least layout.padded_numel elements.  Asynchronous on `stream` (default:
    torch's current stream).  stage: read through shared memory with bulk
    copies (DOPT_STEP_STAGE).  host_params: any param replica may be a
    pinned CPU tensor, which the kernel writes in place
    (DOPT_STEP_HOST_PARAMS).
    """
    import torch

    device, gp, pp, dt, mg, pflag = _step_pointers(layout, grad_replicas, master, exp_avg, exp_avg_sq,
                                            param_replicas, main_grad_out, host_grads,
                                            host_params)
    flags = _flags(gather, host_grads, round_grad, stage) | pflag
    cfg = adam.to_c()
    with _on(device):
        _check(lib().dopt_step(layout.handle, ctypes.byref(cfg), int(step), gp, dt,
                               master.data_ptr(), exp_avg.data_ptr(), exp_avg_sq.data_ptr(), pp,
                               flags, mg, _stream_handle(stream)))


def step_counter(next_step: int = 1, device=None):
    """A dopt_step_counter in device memory (an int64 tensor of 8 elements:
    element 0 is next_step, the low half of element 1 the status)."""
    import torch

    c = torch.zeros(DOPT_STEP_COUNTER_BYTES // 8, dtype=torch.int64,
                    device=device if device is not None else "cuda")
    c[0] = int(next_step)
    return c


def counter_state(counter):
    """(next_step, status) of a step counter (synchronises with the device)."""
    import torch

    h = counter.cpu()
    return int(h[0]), int(h[1:2].view(torch.int32)[0])


def counter_scalars(counter):
    """(step_size, bc2_sqrt): the two step-dependent Adam scalars the last
    counted step took, as float32 bit patterns read back (synchronises)."""
    import torch

    h = counter.cpu()[2:3].view(torch.float32)
    return float(h[0]), float(h[1])


def counter_diagnostics(counter):
    """(exact_steps, undecided_steps) of a step counter: the counted steps
    whose two scalars needed the device's exact evaluation, and those where
    even it could not decide (see dopt_step_counted; synchronises)."""
    import torch

    h = counter.cpu()[4:5].view(torch.int32)
    return int(h[0]), int(h[1])


def _check_counter(counter, device):
    import torch

    if (not isinstance(counter, torch.Tensor) or counter.dtype != torch.int64
            or counter.device != device or not counter.is_contiguous()
            or counter.numel() * 8 < DOPT_STEP_COUNTER_BYTES):
        raise DoptError(DOPT_E_ARG, "counter must be a contiguous int64 tensor of "
                        f"{DOPT_STEP_COUNTER_BYTES // 8} elements on {device} (step_counter())")


def dopt_step_counted(layout: Layout, adam: AdamConfig, counter, grad_replicas, master,
                      exp_avg, exp_avg_sq, param_replicas, gather: bool = True,
                      main_grad_out=None, stream=None, host_grads: bool = False,
                      round_grad: bool = False, stage: bool = False) -> None:
    """dopt_step with the step number read from, and advanced in, a device
    counter (:func:`step_counter`): the launches do not depend on the step,
    so they can be captured once in a CUDA graph and replayed every step."""
    import torch

    device, gp, pp, dt, mg, pflag = _step_pointers(layout, grad_replicas, master, exp_avg, exp_avg_sq,
                                            param_replicas, main_grad_out, host_grads)
    _check_counter(counter, master.device)
    flags = _flags(gather, host_grads, round_grad, stage) | pflag
    cfg = adam.to_c()
    with _on(device):
        _check(lib().dopt_step_counted(layout.handle, ctypes.byref(cfg), counter.data_ptr(), gp,
                                       dt, master.data_ptr(), exp_avg.data_ptr(),
                                       exp_avg_sq.data_ptr(), pp, flags, mg,
                                       _stream_handle(stream)))


class StepPlan:
    """The arguments of repeated steps over the same buffers, checked and
    marshalled once: each ``step`` / ``step_buckets`` is then one call into
    the library (the per-call checks of :func:`dopt_step` cost more host time
    than a small launch).  The plan keeps the tensors alive; the caller must
    not reallocate them while the plan is in use."""

    def __init__(self, layout: Layout, adam: AdamConfig, grad_replicas, master, exp_avg,
                 exp_avg_sq, param_replicas, gather: bool = True, main_grad_out=None,
                 host_grads: bool = False, round_grad: bool = False, stream=None,
                 stage: bool = False):
        import torch

        self.device, self._gp, self._pp, self._dt, self._mg, pflag = _step_pointers(
            layout, grad_replicas, master, exp_avg, exp_avg_sq, param_replicas, main_grad_out,
            host_grads)
        self.layout = layout
        self._keep = (list(grad_replicas), master, exp_avg, exp_avg_sq, list(param_replicas),
                      main_grad_out)
        self._state = (master.data_ptr(), exp_avg.data_ptr(), exp_avg_sq.data_ptr())
        self._flags = _flags(gather, host_grads, round_grad, stage) | pflag
        self._cfg = adam.to_c()
        with torch.cuda.device(self.device):
            self._stream = _stream_handle(stream)
        self._lib = lib()

    def step(self, step: int) -> None:
        """dopt_step on the planned buffers."""
        _check(self._lib.dopt_step(self.layout.handle, ctypes.byref(self._cfg), int(step), self._gp,
                                   self._dt, *self._state, self._pp, self._flags, self._mg,
                                   self._stream))

    def step_counted(self, counter) -> None:
        """dopt_step_counted on the planned buffers."""
        _check_counter(counter, self._keep[1].device)
        _check(self._lib.dopt_step_counted(self.layout.handle, ctypes.byref(self._cfg),
                                           counter.data_ptr(), self._gp, self._dt, *self._state,
                                           self._pp, self._flags, self._mg, self._stream))

    def step_buckets(self, step: int, first_bucket: int, n_buckets: int = 1, stream=None) -> None:
        """dopt_step_buckets on the planned buffers (optionally another stream)."""
        st = self._stream if stream is None else _stream_handle(stream)
        _check(self._lib.dopt_step_buckets(self.layout.handle, ctypes.byref(self._cfg), int(step),
                                           int(first_bucket), int(n_buckets), self._gp, self._dt,
                                           *self._state, self._pp, self._flags, self._mg, st))


class HostStepper:
    """Steps whose grads arrive in pinned host memory and whose result (param
    replica 0) goes back to pinned host memory, pipelined: every step reads
    the host grads in place (DOPT_STEP_HOST_GRADS), copies replica 0 to a
    device staging buffer, and returns it to `host_params_out` on a side
    stream while the next step runs.  `host_params_out` holds the result of
    the latest step once :meth:`synchronize` (or a device-wide sync) has
    returned; reading it earlier races with the copy."""

    def __init__(self, layout: Layout, adam: AdamConfig, master, exp_avg, exp_avg_sq,
                 param_replicas, host_params_out, stream=None):
        import torch

        if host_params_out.device.type != "cpu" or not host_params_out.is_pinned():
            raise DoptError(DOPT_E_ARG, "host_params_out must be a pinned CPU tensor")
        _check_tensor(host_params_out, "host_params_out", param_replicas[0].dtype,
                      layout.padded_numel, host_params_out.device)
        self.layout, self.adam = layout, adam
        self.state = (master, exp_avg, exp_avg_sq)
        self.params = list(param_replicas)
        self.out = host_params_out
        self.device = master.device
        self.stream = torch.cuda.current_stream(self.device) if stream is None else stream
        self.copy_stream = torch.cuda.Stream(self.device)
        self.stage = torch.empty_like(self.params[0])
        self.copied = None

    def step(self, step: int, host_grads) -> None:
        import torch

        with torch.cuda.stream(self.stream):
            dopt_step(self.layout, self.adam, step, host_grads, *self.state, self.params,
                      gather=True, stream=self.stream, host_grads=True)
            if self.copied is not None:  # the staging buffer is free again
                self.stream.wait_event(self.copied)
            self.stage.copy_(self.params[0], non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(self.stream)
        self.copy_stream.wait_event(ready)
        with torch.cuda.stream(self.copy_stream):
            self.out.copy_(self.stage, non_blocking=True)
            self.copied = torch.cuda.Event()
            self.copied.record(self.copy_stream)

    def synchronize(self) -> None:
        """Make the caller's stream wait for the last result copy."""
        if self.copied is not None:
            self.stream.wait_event(self.copied)


def clip_workspace(device=None):
    """A device workspace for dopt_step_clipped (DOPT_CLIP_WORKSPACE_BYTES)."""
    import torch

    return torch.zeros(DOPT_CLIP_WORKSPACE_BYTES, dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def clip_report(device=None):
    """A device buffer for the dopt_clip_report of dopt_step_clipped (16
    bytes: norm, coefficient, count of non-finite reduced grads)."""
    import torch

    return torch.zeros(4, dtype=torch.float32, device=device if device is not None else "cuda")


def read_clip_report(report):
    """(norm, coef, nonfinite) of a :func:`clip_report` buffer
    (synchronises with the device)."""
    import torch

    h = report.cpu()
    return float(h[0]), float(h[1]), int(h[2:4].view(torch.int64)[0])


def dopt_step_clipped(layout: Layout, adam: AdamConfig, step: int, max_norm: float,
                      grad_replicas, master, exp_avg, exp_avg_sq, param_replicas, main_grad,
                      workspace, gather: bool = True, norm_out=None, stream=None,
                      round_grad: bool = False, skip_nonfinite: bool = False) -> None:
    """The step with global grad-norm clipping (two passes over memory: the
    norm pass, then the step; see dopt_step_clipped in dopt.h).

    main_grad: fp32 CUDA tensor of >= padded_numel elements (receives the
    reduced grads before clipping); workspace: from :func:`clip_workspace`;
    norm_out: optional fp32 CUDA tensor of 2 elements (norm, coefficient),
    or a :func:`clip_report` (required size with skip_nonfinite).
    skip_nonfinite: store nothing when any reduced grad is Inf or NaN (the
    report then holds the count and a NaN coefficient).
    """
    import torch

    D = layout.D
    if len(grad_replicas) != D or len(param_replicas) != D:
        raise DoptError(DOPT_E_ARG, f"need {D} grad and {D} param replicas")
    N = layout.padded_numel
    device = master.device
    if device.type != "cuda":
        raise DoptError(DOPT_E_ARG, "dopt_step_clipped needs CUDA tensors (no CPU path exists)")
    gdt = grad_replicas[0].dtype
    dt = _grad_code(gdt)
    for i, g in enumerate(grad_replicas):
        _check_tensor(g, f"grad_replicas[{i}]", gdt, N, device)
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq),
                    ("main_grad", main_grad)):
        _check_tensor(t, name, torch.float32, N, device)
    pflag = _param_flag(param_replicas, N, device)
    _check_tensor(workspace, "workspace", torch.uint8, DOPT_CLIP_WORKSPACE_BYTES, device)
    if norm_out is not None:
        _check_tensor(norm_out, "norm_out", torch.float32, 4 if skip_nonfinite else 2, device)
    gp = (ctypes.c_void_p * D)(*[g.data_ptr() for g in grad_replicas])
    pp = (ctypes.c_void_p * D)(*[p.data_ptr() for p in param_replicas])
    cfg = adam.to_c()
    with _on(device):
        _check(lib().dopt_step_clipped(
            layout.handle, ctypes.byref(cfg), int(step), float(max_norm), gp,
            dt, master.data_ptr(),
            exp_avg.data_ptr(), exp_avg_sq.data_ptr(), pp,
            _flags(gather, round_grad=round_grad) | pflag
            | (DOPT_STEP_SKIP_NONFINITE if skip_nonfinite else 0),
            main_grad.data_ptr(), workspace.data_ptr(),
            None if norm_out is None else norm_out.data_ptr(), _stream_handle(stream)))


def dopt_step_clipped_counted(layout: Layout, adam: AdamConfig, counter, max_norm: float,
                              grad_replicas, master, exp_avg, exp_avg_sq, param_replicas,
                              main_grad, workspace, gather: bool = True, norm_out=None,
                              stream=None, round_grad: bool = False,
                              skip_nonfinite: bool = False) -> None:
    """dopt_step_clipped with the step number read from, and advanced in, a
    device counter (:func:`step_counter`), for graph capture."""
    import torch

    device, gp, pp, dt, mg, pflag = _step_pointers(layout, grad_replicas, master, exp_avg,
                                                   exp_avg_sq, param_replicas, main_grad)
    if main_grad is None:
        raise DoptError(DOPT_E_ARG, "main_grad is required")
    _check_counter(counter, device)
    _check_tensor(workspace, "workspace", torch.uint8, DOPT_CLIP_WORKSPACE_BYTES, device)
    if norm_out is not None:
        _check_tensor(norm_out, "norm_out", torch.float32, 4 if skip_nonfinite else 2, device)
    flags = (_flags(gather, round_grad=round_grad) | pflag
             | (DOPT_STEP_SKIP_NONFINITE if skip_nonfinite else 0))
    cfg = adam.to_c()
    with _on(device):
        _check(lib().dopt_step_clipped_counted(
            layout.handle, ctypes.byref(cfg), counter.data_ptr(), float(max_norm), gp, dt,
            master.data_ptr(), exp_avg.data_ptr(), exp_avg_sq.data_ptr(), pp, flags, mg,
            workspace.data_ptr(), None if norm_out is None else norm_out.data_ptr(),
            _stream_handle(stream)))


def dopt_step_clipped_noalloc(layout: Layout, adam: AdamConfig, step: int, max_norm: float,
                              grad_replicas, master, exp_avg, exp_avg_sq, param_replicas,
                              main_grad, gather: bool = True, norm_out=None, stream=None) -> None:
    """dopt_step_clipped without a workspace argument, for callers that must
    not allocate device memory on the step's path: the scratch lives in a
    static device array inside libdopt.so, shared by every call on a device
    (calls that overlap on the GPU race on it).  The first call on a device
    looks up that array's address; make it before any stream capture."""
    import torch

    D = layout.D
    if len(grad_replicas) != D or len(param_replicas) != D:
        raise DoptError(DOPT_E_ARG, f"need {D} grad and {D} param replicas")
    N = layout.padded_numel
    device = master.device
    if device.type != "cuda":
        raise DoptError(DOPT_E_ARG, "dopt_step_clipped_noalloc needs CUDA tensors")
    gdt = grad_replicas[0].dtype
    dt = _grad_code(gdt)
    for i, g in enumerate(grad_replicas):
        _check_tensor(g, f"grad_replicas[{i}]", gdt, N, device)
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq),
                    ("main_grad", main_grad)):
        _check_tensor(t, name, torch.float32, N, device)
    pflag = _param_flag(param_replicas, N, device)
    if norm_out is not None:
        _check_tensor(norm_out, "norm_out", torch.float32, 2, device)
    gp = (ctypes.c_void_p * D)(*[g.data_ptr() for g in grad_replicas])
    pp = (ctypes.c_void_p * D)(*[p.data_ptr() for p in param_replicas])
    cfg = adam.to_c()
    with _on(device):
        _check(lib().dopt_step_clipped_noalloc(
            layout.handle, ctypes.byref(cfg), int(step), float(max_norm), gp,
            dt, master.data_ptr(),
            exp_avg.data_ptr(), exp_avg_sq.data_ptr(), pp,
            (DOPT_STEP_GATHER if gather else 0) | pflag,
            main_grad.data_ptr(), None if norm_out is None else norm_out.data_ptr(),
            _stream_handle(stream)))


def dopt_gather(layout: Layout, param_replicas, stream=None) -> None:
    """The all-gather alone: every rank's owned elements into every replica."""
    import torch

    D = layout.D
    if len(param_replicas) != D:
        raise DoptError(DOPT_E_ARG, f"need {D} param replicas")
    device = param_replicas[0].device
    if device.type != "cuda":
        raise DoptError(DOPT_E_ARG, "dopt_gather needs CUDA tensors")
    _param_flag(param_replicas, layout.padded_numel, device)  # bf16 or fp16: 16-bit copies
    pp = (ctypes.c_void_p * D)(*[p.data_ptr() for p in param_replicas])
    with _on(device):
        _check(lib().dopt_gather(layout.handle, pp, _stream_handle(stream)))


def version() -> str:
    return lib().dopt_version().decode()


def step_from_host(layout: Layout, adam: AdamConfig, step: int, host_grads, dev_grads, master,
                   exp_avg, exp_avg_sq, param_replicas, host_params_out=None, stream=None,
                   zero_copy: bool = False, params_out_in_place: bool = False) -> None:
    """The step for a caller whose grads sit in pinned host memory.

    Staged (default): copy the D host grad replicas into the device buffers
    `dev_grads`, then run dopt_step.  zero_copy: the kernel reads the pinned
    host replicas in place over the host link (DOPT_STEP_HOST_GRADS);
    `dev_grads` is not used.  Either way replica 0 of the updated params is
    copied back into `host_params_out` (if given).  params_out_in_place
    (with zero_copy): `host_params_out` (pinned) is itself param replica 0,
    which the kernel writes over the host link (DOPT_STEP_HOST_PARAMS);
    `param_replicas[0]` on the device is then not written.  Everything is
    queued on `stream`; the caller synchronises before reading
    `host_params_out`."""
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    with torch.cuda.stream(s):
        if zero_copy and params_out_in_place:
            if host_params_out is None:
                raise DoptError(DOPT_E_ARG, "params_out_in_place needs host_params_out")
            dopt_step(layout, adam, step, host_grads, master, exp_avg, exp_avg_sq,
                      [host_params_out] + list(param_replicas[1:]), gather=True, stream=s,
                      host_grads=True, host_params=True)
            return
        if zero_copy:
            dopt_step(layout, adam, step, host_grads, master, exp_avg, exp_avg_sq, param_replicas,
                      gather=True, stream=s, host_grads=True)
        else:
            for h, d in zip(host_grads, dev_grads):
                d.copy_(h, non_blocking=True)
            dopt_step(layout, adam, step, dev_grads, master, exp_avg, exp_avg_sq,
                      param_replicas, gather=True, stream=s)
        if host_params_out is not None:
            host_params_out.copy_(param_replicas[0], non_blocking=True)
