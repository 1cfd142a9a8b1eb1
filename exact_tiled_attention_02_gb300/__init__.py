"""Exact tiled attention for NVIDIA GB300 (sm_103a).

The compute lives in ``libfa.so`` (hand-written TMA + tcgen05 kernels behind
the C ABI declared in ``include/fa.h``); ``binding`` marshals torch tensors
into those calls.  Importing the package does not load the library; the first
use of a ``fa_*`` name does, and fails loudly if the library is missing.
"""

__all__ = ["fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_static_workspace", "fa_last_device_status", "fa_set_wait_limit_us",
           "fa_selftest_wait_timeout", "fa_status_string", "fa_version", "FaError"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
