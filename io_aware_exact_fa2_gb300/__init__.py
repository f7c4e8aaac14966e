"""GB300-native exact FlashAttention-2 forward (sm_103a, tcgen05 + TMA).

The compute path is the C-ABI library ``libfa2_gb300.so`` built from
``csrc/`` (declared in ``include/fa2.h``); this package is the thin Python
binding over it.  The binding symbols (``fa2_fwd`` and friends) are resolved
on first use: if the CUDA library has not been built, that raises ImportError
-- there is no CPU fallback.

``workloads`` (seeded synthetic inputs) imports no CUDA code and is usable on
a machine without a GPU.
"""
from . import workloads  # noqa: F401

_BINDING_NAMES = (
    "fa2_fwd", "fa2_fwd_fp8", "fa2_fwd_from_host", "fa2_get_device_error", "fa2_status_string",
    "fa2_workspace_size", "fa2_workspace", "fa2_fwd_noalloc", "NOALLOC_SCRATCH_BYTES",
    "fa2_bwd", "fa2_bwd_window", "fa2_bwd_ex", "fa2_bwd_workspace_size", "fa2_fwd_window", "fa2_fwd_ex",
    "fa2_version", "Fa2Error", "library_path", "load_library", "STATUS",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
