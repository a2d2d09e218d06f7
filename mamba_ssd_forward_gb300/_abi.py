"""ctypes view of the C ABI declared in include/ssd.h (libssd_gb300.so).

Marshalling only: every step of the forward pass runs in the library's CUDA
kernels.  If the library has not been built, loading fails loudly; there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libssd_gb300.so")

(SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_TIMEOUT,
 SSD_ERR_BOUNDS) = range(6)
SSD_F32, SSD_BF16 = 0, 1
# Size of the fixed scratch array of ssd_forward_noalloc (SSD_NOALLOC_SCRATCH_BYTES).
SSD_NOALLOC_SCRATCH_BYTES = 32 << 20
# Workspace header holding a call's device error word (SSD_WS_HEADER_BYTES).
SSD_WS_HEADER_BYTES = 256

# Every symbol include/ssd.h declares.
EXPORTS = (
    "ssd_status_string",
    "ssd_forward_workspace_size",
    "ssd_chunk_cumsum",
    "ssd_chunk_state",
    "ssd_state_passing",
    "ssd_chunk_scan",
    "ssd_forward",
    "ssd_forward_ex",
    "ssd_workspace_error",
    "ssd_device_error",
    "ssd_forward_profiled",
    "ssd_forward_host_workspace_size",
    "ssd_forward_host",
    "ssd_forward_noalloc",
    "ssd_decode_step",
    "ssd_forward_host_overlapped_workspace_size",
    "ssd_forward_host_overlapped",
    "ssd_forward_plan_candidates",
    "ssd_forward_default_plan",
    "ssd_forward_tune",
    "ssd_selftest_bounded_wait",
    "ssd_backward_workspace_size",
    "ssd_backward",
    "ssd_backward_profiled",
)


class SsdDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups", "chunk")]


class SsdPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("chunk_state_heads", "chunk_state_ctas", "scan_kernel", "scan_heads")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class SsdError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


_lib = None


def load(path: str | None = None):
    """Load libssd_gb300.so and declare its prototypes."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build the CUDA library first "
            "(python -m mamba_ssd_forward_gb300.build, or __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    vp, dims_p, i32, sz = ctypes.c_void_p, ctypes.POINTER(SsdDims), ctypes.c_int, ctypes.c_size_t
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_status_string.argtypes = [i32]
    lib.ssd_forward_workspace_size.restype = sz
    lib.ssd_forward_workspace_size.argtypes = [dims_p, i32]
    lib.ssd_chunk_cumsum.restype = i32
    lib.ssd_chunk_cumsum.argtypes = [dims_p, i32, vp, vp, vp, vp]
    lib.ssd_chunk_state.restype = i32
    lib.ssd_chunk_state.argtypes = [dims_p, i32, vp, vp, vp, vp, vp, vp]
    lib.ssd_state_passing.restype = i32
    lib.ssd_state_passing.argtypes = [dims_p, vp, vp, vp, vp, vp, vp]
    lib.ssd_chunk_scan.restype = i32
    lib.ssd_chunk_scan.argtypes = [dims_p, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    plan_p = ctypes.POINTER(SsdPlan)
    lib.ssd_forward.restype = i32
    lib.ssd_forward.argtypes = [dims_p, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_forward_ex.restype = i32
    lib.ssd_forward_ex.argtypes = [dims_p, i32] + [vp] * 10 + [sz, plan_p, vp]
    lib.ssd_workspace_error.restype = i32
    lib.ssd_workspace_error.argtypes = [vp, vp]
    lib.ssd_device_error.restype = i32
    lib.ssd_device_error.argtypes = [vp]
    lib.ssd_forward_profiled.restype = i32
    lib.ssd_forward_profiled.argtypes = ([dims_p, i32] + [vp] * 10 + [sz, plan_p, vp, vp, i32,
                                         ctypes.POINTER(ctypes.c_int)])
    lib.ssd_forward_host_workspace_size.restype = sz
    lib.ssd_forward_host_workspace_size.argtypes = [dims_p, i32, i32, i32, i32]
    lib.ssd_forward_host.restype = i32
    lib.ssd_forward_host.argtypes = [dims_p, i32] + [vp] * 10 + [sz, plan_p, vp]
    lib.ssd_forward_host_overlapped_workspace_size.restype = sz
    lib.ssd_forward_host_overlapped_workspace_size.argtypes = [dims_p, i32, i32, i32, i32, i32]
    lib.ssd_forward_host_overlapped.restype = i32
    lib.ssd_forward_host_overlapped.argtypes = ([dims_p, i32] + [vp] * 10 +
                                                [sz, i32, plan_p, vp, vp, vp])
    lib.ssd_decode_step.restype = i32
    lib.ssd_decode_step.argtypes = [dims_p, i32] + [vp] * 9
    lib.ssd_forward_noalloc.restype = i32
    lib.ssd_forward_noalloc.argtypes = [dims_p, i32] + [vp] * 9 + [vp]
    lib.ssd_forward_plan_candidates.restype = i32
    lib.ssd_forward_plan_candidates.argtypes = [dims_p, i32, plan_p, i32]
    lib.ssd_forward_default_plan.restype = i32
    lib.ssd_forward_default_plan.argtypes = [dims_p, i32, plan_p]
    lib.ssd_selftest_bounded_wait.restype = i32
    lib.ssd_selftest_bounded_wait.argtypes = [ctypes.c_uint64, vp, vp]
    lib.ssd_forward_tune.restype = i32
    lib.ssd_forward_tune.argtypes = [dims_p, i32] + [vp] * 10 + [sz, i32, vp, sz, vp, plan_p]
    lib.ssd_backward_workspace_size.restype = sz
    lib.ssd_backward_workspace_size.argtypes = [dims_p, i32]
    lib.ssd_backward.restype = i32
    lib.ssd_backward.argtypes = [dims_p, i32] + [vp] * 17 + [sz, vp]
    lib.ssd_backward_profiled.restype = i32
    lib.ssd_backward_profiled.argtypes = ([dims_p, i32] + [vp] * 17 +
                                          [sz, vp, vp, i32, ctypes.POINTER(ctypes.c_int)])
    if path is None:
        _lib = lib
    return lib


def check(fn: str, code: int) -> None:
    if code != SSD_OK:
        msg = load().ssd_status_string(code).decode()
        raise SsdError(fn, code, msg)
