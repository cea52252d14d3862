"""GB300-native ZeRO-1 distributed-optimizer step (Megatron-style, flat buffer).

The work runs in libdopt.so (hand-written sm_103a CUDA kernels behind the C
ABI declared in include/dopt.h); this package is its thin Python binding.
The library is loaded on first use and every call raises if it is missing.
"""
from .binding import (  # noqa: F401
    DOPT_BF16,
    DOPT_CLIP_WORKSPACE_BYTES,
    DOPT_COUNTER_BAD_STEP,
    DOPT_E_ALIGN,
    DOPT_E_ARG,
    DOPT_E_CUDA,
    DOPT_E_LAYOUT,
    DOPT_E_NOMEM,
    DOPT_E_STATE,
    DOPT_FP32,
    DOPT_MAX_D,
    DOPT_OK,
    DOPT_STEP_GATHER,
    DOPT_STEP_HOST_GRADS,
    DOPT_STEP_COUNTER_BYTES,
    DOPT_STEP_ROUND_GRAD,
    AdamConfig,
    DoptError,
    HostStepper,
    Layout,
    StepPlan,
    dopt_allreduce,
    dopt_build_range_map,
    dopt_gather,
    dopt_step,
    dopt_step_allreduce,
    dopt_step_buckets,
    dopt_step_clipped,
    dopt_step_clipped_noalloc,
    dopt_step_counted,
    clip_workspace,
    counter_state,
    step_counter,
    step_from_host,
    version,
)
