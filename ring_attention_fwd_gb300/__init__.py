"""GB300-native ring-order blockwise attention (sm_103a).

The compute lives in ``libringattn.so`` (C ABI, hand-written CUDA kernels);
``binding`` marshals arguments to it.  The library is loaded on first use and
a missing build raises immediately: there is no fallback path.
"""
from . import flops, inputs  # noqa: F401
from .binding import (  # noqa: F401
    RingAttnError, bwd, bwd_noalloc, bwd_step, bwd_workspace_bytes, check_device_status, decode, decode_workspace_bytes, ffn,
    ffn_workspace_bytes, fwd, fwd_step, fwd_step_fold, kernel_times, merge, read_checks, set_fwd_kernel, set_kernel_timing, set_timing_buffer,
    use_checked_build, version,
)
