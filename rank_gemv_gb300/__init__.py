"""rank_gemv_gb300: Punica's SGMV (Segmented Gather Matrix-Vector multiplication)
multi-LoRA hot path, written for one GB300 (sm_103a).

The compute lives in ``libsgmv.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/sgmv.h``).  ``rank_gemv_gb300.sgmv`` is a thin ctypes
binding with the same function names; importing a name from it here loads the
library and raises if it has not been built.  ``rank_gemv_gb300.workloads``
draws seeded synthetic inputs and needs no GPU.
"""

__version__ = "0.1.0"

_BINDING_NAMES = {
    "sgmv_status_string", "sgmv_max_segments", "sgmv_build_segments",
    "sgmv_build_segments_device", "sgmv_workspace_bytes", "sgmv_shrink", "sgmv_expand",
    "sgmv_apply", "sgmv_apply_multi", "sgmv_apply_rows", "sgmv_apply_noalloc", "sgmv_load_adapter", "sgmv_copy_gather",
    "sgmv_get_device_error", "sgmv_last_launch_count", "sgmv_read_floor",
    "sgmv_debug_inject_wait_timeout", "sgmv_fused_workspace_bytes", "sgmv_fused_linear_lora",
    "SgmvError", "load_library",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import sgmv

        return getattr(sgmv, name)
    raise AttributeError(name)
