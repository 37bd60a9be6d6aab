"""GB300-native ring-order blockwise attention (sm_103a).

The compute lives in ``libringattn.so`` (C ABI, hand-written CUDA kernels);
``binding`` marshals arguments to it.  The library is loaded on first use and
a missing or stale build raises immediately: there is no fallback path.
"""
from . import flops, inputs  # noqa: F401
