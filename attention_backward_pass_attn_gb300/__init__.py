"""GB300-native exact-attention forward and fused backward.

The CUDA kernels live in ``csrc/`` and are compiled for sm_103a into the
in-tree shared library ``libattn_gb300.so``, whose C ABI is declared in
``include/attn.h``.  ``binding`` wraps that ABI with ctypes; PyTorch only
provides device memory and streams.  Importing this package does not load the
library; the first call into ``binding`` does, and raises if it is missing.
"""

from .inputs import WORKLOADS, WORKLOAD_ORDER, Workload, make_inputs  # noqa: F401

_BINDING_NAMES = (
    "attn_fwd", "attn_fwd_fp8", "attn_bwd", "attn_bwd_fp8", "attn_bwd_preprocess", "attn_bwd_main",
    "attn_bwd_dq_convert", "attn_bwd_main_dkdv", "attn_bwd_dq", "attn_bwd_workspace_size", "alloc_workspace",
    "attn_last_device_error", "attn_device_error_word", "attn_watchdog_selftest",
    "status_string", "AttnError", "load_library", "ssd_fwd", "ssd_bwd", "ssd_workspace", "ATTN_DQ_AUTO", "ATTN_DQ_REDUCE",
    "ATTN_DQ_SEPARATE",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
