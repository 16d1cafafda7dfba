"""fp64 CPU oracle for the Mamba-2 SSD forward pass.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark use it; the library's product path never imports it.  It
shares no code with the CUDA path (see ssd_oracle.c for what each function
computes and which passage it follows).

The C source is compiled with gcc into ``liboracle.so`` beside this file on
first use (or by :func:`build`).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, fp64, OpenMP, no fp contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            d = ctypes.POINTER(ctypes.c_double)
            i32 = ctypes.POINTER(ctypes.c_int32)
            f = ctypes.POINTER(ctypes.c_float)
            i64, ci = ctypes.c_int64, ctypes.c_int
            common = [i64, i64, ci, ci, ci, ci, d, d, d, d, d, d, d, i32, ci]
            lib.oracle_ssd_recurrence.argtypes = common + [d, d, ci]
            lib.oracle_ssd_quadratic.argtypes = common + [d]
            lib.oracle_ssd_chunked.argtypes = common + [ci, i64, d, d]
            lib.oracle_ssd_backward.argtypes = [i64, i64, ci, ci, ci, ci, d, d, d, d, d, d, d, i32, ci, d, d,
                                                d, d, d, d, d, d, d, ci]
            lib.oracle_segsum.argtypes = [d, i64, ci, d]
            lib.oracle_diff_segsum_f32.argtypes = [f, i64, ci, f]
            lib.oracle_max_threads.restype = ci
            for fn in (lib.oracle_ssd_recurrence, lib.oracle_ssd_quadratic, lib.oracle_ssd_chunked,
                       lib.oracle_ssd_backward, lib.oracle_segsum, lib.oracle_diff_segsum_f32):
                fn.restype = None
            _lib = lib
    return _lib


def _dp(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _args(p):
    """Widen a problem's (fp32 / bf16-exact) arrays to fp64 exactly."""
    arrs = dict(x=_f64(p.x), dt=_f64(p.dt), A=_f64(p.A), B=_f64(p.B), C=_f64(p.C), D=_f64(p.D),
                init=_f64(p.initial_states))
    cu = None if p.cu_seqlens is None else np.ascontiguousarray(p.cu_seqlens, dtype=np.int32)
    return arrs, cu


def _check(p):
    if p.nheads % p.ngroups != 0:
        raise ValueError("nheads must be a multiple of ngroups")
    if p.cu_seqlens is not None and p.batch != 1:
        raise ValueError("packed documents need batch == 1")


def _common(p, arrs, cu):
    i32p = None if cu is None else cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    return [p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups,
            _dp(arrs["x"]), _dp(arrs["dt"]), _dp(arrs["A"]), _dp(arrs["B"]), _dp(arrs["C"]),
            _dp(arrs["D"]), _dp(arrs["init"]), i32p, p.ndocs]


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def ssd_recurrence(p, want_final: bool = True, nthreads: int = 0):
    """Sequential recurrence, fp64. Returns (y, final_states or None)."""
    _check(p)
    lib = _load()
    arrs, cu = _args(p)
    y = np.zeros((p.batch, p.seqlen, p.nheads, p.headdim), dtype=np.float64)
    fin = np.zeros((p.nstates, p.nheads, p.headdim, p.dstate), dtype=np.float64) if want_final else None
    lib.oracle_ssd_recurrence(*_common(p, arrs, cu), _dp(y), _dp(fin), int(nthreads))
    return y, fin


class _StepProblem:
    """A one-token problem: the arrays of a decode step seen as seqlen = 1."""

    def __init__(self, state, x, dt, A, B, C, D):
        self.batch, self.nheads, self.headdim = x.shape
        self.ngroups, self.dstate = B.shape[1], B.shape[2]
        self.seqlen, self.ndocs, self.nstates, self.cu_seqlens = 1, 0, self.batch, None
        self.x = x.reshape(self.batch, 1, self.nheads, self.headdim)
        self.dt = dt.reshape(self.batch, 1, self.nheads)
        self.B = B.reshape(self.batch, 1, self.ngroups, self.dstate)
        self.C = C.reshape(self.batch, 1, self.ngroups, self.dstate)
        self.A, self.D, self.initial_states = A, D, state


def ssd_step(state, x, dt, A, B, C, D=None):
    """One decode step, fp64: the recurrence taken once from ``state``
    ("State Space Duality and Mamba-2", "Performance and Serving Economics":
    a fixed-size state updated once per generated token).

    state (batch, H, P, N), x (batch, H, P), dt (batch, H), A (H),
    B, C (batch, G, N), D (H) or None.  Returns (y (batch, H, P), state')."""
    q = _StepProblem(np.asarray(state), np.asarray(x), np.asarray(dt), np.asarray(A), np.asarray(B),
                     np.asarray(C), None if D is None else np.asarray(D))
    y, fin = ssd_recurrence(q, want_final=True)
    return y.reshape(q.batch, q.nheads, q.headdim), fin


def ssd_backward(p, dy, dfinal=None, nthreads: int = 0):
    """Gradients of <dy, y> + <dfinal, final_states> with respect to every input
    of the forward pass, fp64 (batch rows, or packed documents each with its own
    initial and final state).

    Returns a dict of arrays: dx, ddt, dA, dB, dC, dD (None without D) and
    dinit (the initial states' gradient, also when the forward had none)."""
    _check(p)
    lib = _load()
    arrs, cu = _args(p)
    cup = None if cu is None else cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    dy64 = _f64(dy)
    df64 = _f64(dfinal)
    out = dict(dx=np.zeros((p.batch, p.seqlen, p.nheads, p.headdim)), ddt=np.zeros((p.batch, p.seqlen, p.nheads)),
               dA=np.zeros(p.nheads), dB=np.zeros((p.batch, p.seqlen, p.ngroups, p.dstate)),
               dC=np.zeros((p.batch, p.seqlen, p.ngroups, p.dstate)),
               dD=None if p.D is None else np.zeros(p.nheads),
               dinit=np.zeros((p.nstates, p.nheads, p.headdim, p.dstate)))
    lib.oracle_ssd_backward(p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups,
                            _dp(arrs["x"]), _dp(arrs["dt"]), _dp(arrs["A"]), _dp(arrs["B"]), _dp(arrs["C"]),
                            _dp(arrs["D"]), _dp(arrs["init"]), cup, p.ndocs, _dp(dy64), _dp(df64),
                            _dp(out["dx"]), _dp(out["ddt"]), _dp(out["dA"]), _dp(out["dB"]), _dp(out["dC"]),
                            _dp(out["dD"]), _dp(out["dinit"]), int(nthreads))
    return out


def gate_norm(y, z, weight, group_size, eps):
    """Gated RMS normalisation, fp64 numpy: g = y * silu(z), then over each group
    of `group_size` consecutive channels out = g / sqrt(mean(g^2) + eps) * weight
    (the gating and normalisation that follow the scan in the Mamba-2 forward
    pass, "NVIDIA Accelerates Mamba-2 Forward Kernel with CUDA Tile", operator
    fusion; the gate is applied before the norm).  y, z: (rows, width)."""
    y = np.asarray(y, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    rows, width = y.shape
    g = y * (z / (1.0 + np.exp(-z)))
    gg = g.reshape(rows, width // group_size, group_size)
    ms = np.mean(gg * gg, axis=2, keepdims=True)
    return (gg / np.sqrt(ms + eps)).reshape(rows, width) * w


def ssd_quadratic(p):
    """(C B^T) o L form plus the initial-state term, fp64, O(L^2)."""
    _check(p)
    lib = _load()
    arrs, cu = _args(p)
    y = np.zeros((p.batch, p.seqlen, p.nheads, p.headdim), dtype=np.float64)
    lib.oracle_ssd_quadratic(*_common(p, arrs, cu), _dp(y))
    return y


def ssd_chunked(p, chunk: int, split_len: int = 0):
    """Block decomposition with split composition, fp64. Returns (y, final)."""
    _check(p)
    lib = _load()
    arrs, cu = _args(p)
    y = np.zeros((p.batch, p.seqlen, p.nheads, p.headdim), dtype=np.float64)
    fin = np.zeros((p.nstates, p.nheads, p.headdim, p.dstate), dtype=np.float64)
    lib.oracle_ssd_chunked(*_common(p, arrs, cu), int(chunk), int(split_len), _dp(y), _dp(fin))
    return y, fin


def segsum(ell):
    """ell (nrows, len) -> seg (nrows, len, len), fp64, -inf above the diagonal."""
    lib = _load()
    e = np.ascontiguousarray(ell, dtype=np.float64)
    nrows, ln = e.shape
    out = np.empty((nrows, ln, ln), dtype=np.float64)
    lib.oracle_segsum(_dp(e), nrows, ln, _dp(out))
    return out


def diff_segsum_f32(ell):
    """The prefix-subtraction comparator in fp32 (known unstable)."""
    lib = _load()
    e = np.ascontiguousarray(ell, dtype=np.float32)
    nrows, ln = e.shape
    out = np.empty((nrows, ln, ln), dtype=np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.oracle_diff_segsum_f32(e.ctypes.data_as(fp), nrows, ln, out.ctypes.data_as(fp))
    return out
