"""ctypes binding of libssd.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels.  If the
shared library is missing this module raises at import time: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libssd.so")

SSD_F32, SSD_BF16 = 0, 1
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_WORKSPACE",
          4: "SSD_ERR_CUDA", 5: "SSD_ERR_TIMEOUT", 6: "SSD_ERR_DEVICE_CHECK"}

# every symbol include/ssd.h declares
EXPORTS = ("ssd_fwd_workspace_size", "ssd_workspace_init", "ssd_fwd", "ssd_check_status",
           "ssd_status_string", "ssd_fwd_plan", "ssd_segsum_dump", "ssd_fwd_static_scratch", "ssd_step",
           "ssd_bwd_workspace_size", "ssd_bwd_workspace_size_doc_states", "ssd_bwd", "ssd_fwd_timed",
           "ssd_gate_norm", "ssd_check_status_where", "ssd_fwd_fault_inject")


class SSDParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int32),
                ("headdim", ctypes.c_int32), ("dstate", ctypes.c_int32), ("ngroups", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("split_len", ctypes.c_int32), ("ndocs", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class SSDError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libssd.so not built ({LIB_PATH}); run `python -m mamba_ssd_chunked_scan_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    P = ctypes.POINTER(SSDParams)
    lib.ssd_fwd_workspace_size.argtypes = [P]
    lib.ssd_fwd_workspace_size.restype = sz
    lib.ssd_workspace_init.argtypes = [vp, sz, vp]
    lib.ssd_workspace_init.restype = ctypes.c_int
    lib.ssd_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_fwd.restype = ctypes.c_int
    lib.ssd_check_status.argtypes = [vp, vp]
    lib.ssd_check_status.restype = ctypes.c_int
    lib.ssd_check_status_where.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.ssd_check_status_where.restype = ctypes.c_int
    lib.ssd_fwd_fault_inject.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, ctypes.c_uint32, vp]
    lib.ssd_fwd_fault_inject.restype = ctypes.c_int
    lib.ssd_status_string.argtypes = [ctypes.c_int]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_fwd_plan.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                 ctypes.POINTER(ctypes.c_int)]
    lib.ssd_fwd_plan.restype = ctypes.c_int
    lib.ssd_fwd_timed.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp,
                                  ctypes.POINTER(ctypes.c_float), ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.ssd_fwd_timed.restype = ctypes.c_int
    lib.ssd_fwd_static_scratch.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ssd_fwd_static_scratch.restype = ctypes.c_int
    lib.ssd_bwd_workspace_size.argtypes = [P]
    lib.ssd_bwd_workspace_size.restype = sz
    lib.ssd_bwd_workspace_size_doc_states.argtypes = [P]
    lib.ssd_bwd_workspace_size_doc_states.restype = sz
    lib.ssd_bwd.argtypes = [P] + [vp] * 18 + [sz, vp]
    lib.ssd_bwd.restype = ctypes.c_int
    lib.ssd_gate_norm.argtypes = [i64, i32, i32, i32, vp, vp, vp, ctypes.c_float, vp, vp]
    lib.ssd_gate_norm.restype = ctypes.c_int
    lib.ssd_step.argtypes = [i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ssd_step.restype = ctypes.c_int
    lib.ssd_segsum_dump.argtypes = [vp, i64, i32, vp, vp, vp, vp, vp]
    lib.ssd_segsum_dump.restype = ctypes.c_int
    return lib


lib = _load()


def make_params(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, split_len, ndocs, dtype) -> SSDParams:
    return SSDParams(int(batch), int(seqlen), int(nheads), int(headdim), int(dstate), int(ngroups),
                     int(chunk), int(split_len), int(ndocs), int(dtype))


def workspace_size(p: SSDParams) -> int:
    return int(lib.ssd_fwd_workspace_size(ctypes.byref(p)))


def plan(p: SSDParams, has_init: bool = False, has_final: bool = False):
    """(kernel family, launches per call, splits) for these params."""
    n, s = ctypes.c_int(0), ctypes.c_int(0)
    fam = lib.ssd_fwd_plan(ctypes.byref(p), int(has_init), int(has_final), ctypes.byref(n), ctypes.byref(s))
    return fam, n.value, s.value


def check(code: int, what: str) -> None:
    if code != 0:
        raise SSDError(code, what)
