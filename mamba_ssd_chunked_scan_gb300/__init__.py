"""Mamba-2 SSD chunked-scan forward pass for GB300 (sm_103a).

Thin PyTorch-facing wrapper over the C ABI of ``libssd.so`` (include/ssd.h):
it checks tensor shapes, takes device pointers and the current CUDA stream,
and calls the library.  PyTorch provides device memory and streams only;
every arithmetic step runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import importlib

import torch

SSD_F32, SSD_BF16 = 0, 1


class _LazyLib:
    """Loads libssd.so on first use; raises ImportError if it is not built."""

    def __getattr__(self, name):
        mod = importlib.import_module(__name__ + "._lib")
        return getattr(mod, name)


_lib = _LazyLib()


def __getattr__(name):
    if name == "SSDError":
        return _lib.SSDError
    raise AttributeError(name)

__all__ = ["ssd_fwd", "SSDForward", "ssd_bwd", "ssd_step", "gate_norm", "segsum_dump", "check_status", "SSDError", "plan"]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    if t.dtype == torch.float32:
        return SSD_F32
    raise TypeError(f"x/B/C must be bf16 or fp32, got {t.dtype}")


class SSDForward:
    """A reusable SSD forward call with fixed shapes: owns its workspace.

    shapes: x (batch, L, H, P), dt (batch, L, H), A (H), B/C (batch, L, G, N),
    D (H) or None, initial/final states (nstates, H, P, N) fp32, cu_seqlens
    (ndocs + 1) int32 or None.
    """

    def __init__(self, batch, seqlen, nheads, headdim, dstate, ngroups=1, chunk=128, split_len=0,
                 ndocs=0, dtype=torch.bfloat16, device="cuda"):
        self.params = _lib.make_params(batch, seqlen, nheads, headdim, dstate, ngroups, chunk,
                                       split_len, ndocs, SSD_BF16 if dtype == torch.bfloat16 else SSD_F32)
        self.dtype = dtype
        nbytes = _lib.workspace_size(self.params)
        if nbytes == 0:
            raise _lib.SSDError(1, "invalid SSD parameters")
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        self.nstates = ndocs if ndocs > 0 else batch

    @property
    def workspace_bytes(self) -> int:
        return self.workspace.numel()

    def plan(self, has_init=False, has_final=False):
        return _lib.plan(self.params, has_init, has_final)

    def __call__(self, x, dt, A, B, C, D=None, initial_states=None, cu_seqlens=None, y=None,
                 final_states=None, stream=None):
        args, y = self._args(x, dt, A, B, C, D, initial_states, cu_seqlens, y, final_states, stream)
        _lib.check(_lib.lib.ssd_fwd(*args), "ssd_fwd")
        return y

    def launch_times(self, x, dt, A, B, C, D=None, initial_states=None, cu_seqlens=None, y=None,
                     final_states=None, stream=None):
        """The same call through ssd_fwd_timed: returns the duration (ms) of each
        kernel launch, in launch order (synchronises the stream)."""
        args, _ = self._args(x, dt, A, B, C, D, initial_states, cu_seqlens, y, final_states, stream)
        ms = (ctypes.c_float * 4)()
        n = ctypes.c_int(0)
        _lib.check(_lib.lib.ssd_fwd_timed(*args, ms, 4, ctypes.byref(n)), "ssd_fwd_timed")
        return [float(ms[k]) for k in range(min(n.value, 4))]

    def _args(self, x, dt, A, B, C, D, initial_states, cu_seqlens, y, final_states, stream):
        p = self.params
        shp_x = (p.batch, p.seqlen, p.nheads, p.headdim)
        shp_bc = (p.batch, p.seqlen, p.ngroups, p.dstate)
        shp_s = (self.nstates, p.nheads, p.headdim, p.dstate)
        for name, t, shp, dt_ in (("x", x, shp_x, self.dtype), ("dt", dt, shp_x[:3], torch.float32),
                                  ("A", A, (p.nheads,), torch.float32), ("B", B, shp_bc, self.dtype),
                                  ("C", C, shp_bc, self.dtype), ("D", D, (p.nheads,), torch.float32),
                                  ("initial_states", initial_states, shp_s, torch.float32),
                                  ("final_states", final_states, shp_s, torch.float32),
                                  ("y", y, shp_x, self.dtype)):
            if t is None:
                continue
            if tuple(t.shape) != shp or t.dtype != dt_ or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"{name}: expected contiguous {dt_} {shp} on {self.device}, got "
                                 f"{t.dtype} {tuple(t.shape)} on {t.device}")
        if (cu_seqlens is None) != (p.ndocs == 0):
            raise ValueError("cu_seqlens must be given exactly when ndocs > 0")
        if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or cu_seqlens.numel() != p.ndocs + 1
                                       or cu_seqlens.device != self.device):
            raise ValueError("cu_seqlens: expected int32 (ndocs + 1) on the device")
        if y is None:
            y = torch.empty(shp_x, dtype=self.dtype, device=self.device)
        args = (ctypes.byref(p), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(initial_states),
                _ptr(cu_seqlens), _ptr(y), _ptr(final_states), _ptr(self.workspace), self.workspace.numel(),
                _stream_handle(stream))
        return args, y

    def check_status(self, stream=None) -> int:
        return check_status(self.workspace, stream)

    def check_status_where(self, stream=None):
        """(status, code of the device wait that recorded it); clears the status."""
        where = ctypes.c_uint32(0)
        st = _lib.lib.ssd_check_status_where(_ptr(self.workspace), _stream_handle(stream), ctypes.byref(where))
        return int(st), int(where.value)

    def fault_inject(self, x, dt, A, B, C, D=None, initial_states=None, cu_seqlens=None, y=None,
                     final_states=None, max_wait_rounds=1 << 14, stream=None):
        """Test aid: the call with an injected stall (ssd_fwd_fault_inject): the
        kernel's loads are never issued and its waits give up after
        max_wait_rounds polls.  Read the outcome with check_status_where()."""
        args, y = self._args(x, dt, A, B, C, D, initial_states, cu_seqlens, y, final_states, stream)
        _lib.check(_lib.lib.ssd_fwd_fault_inject(*args[:-1], int(max_wait_rounds), args[-1]), "ssd_fwd_fault_inject")
        return y


def ssd_fwd(x, dt, A, B, C, D=None, initial_states=None, cu_seqlens=None, *, chunk=128, split_len=0,
            return_final_states=False, stream=None):
    """One SSD forward call.  Returns y, or (y, final_states) when asked."""
    batch, seqlen, nheads, headdim = x.shape
    ngroups, dstate = B.shape[2], B.shape[3]
    ndocs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    f = SSDForward(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, split_len, ndocs,
                   x.dtype, x.device)
    fin = None
    if return_final_states:
        fin = torch.empty((f.nstates, nheads, headdim, dstate), dtype=torch.float32, device=x.device)
    y = f(x, dt, A, B, C, D, initial_states, cu_seqlens, final_states=fin, stream=stream)
    st = f.check_status(stream)
    if st != 0:
        raise _lib.SSDError(st, "ssd_fwd device status")
    return (y, fin) if return_final_states else y


def ssd_bwd(x, dt, A, B, C, dy, D=None, initial_states=None, dfinal_states=None, cu_seqlens=None, *,
            chunk=128, split_len=0, want_dinit=None, stream=None, check_status=False):
    """Gradients of <dy, y> + <dfinal_states, final_states> for one ssd_fwd
    call's inputs.  With packed documents (cu_seqlens, batch 1) the states
    are per document: initial_states, dfinal_states and dinit are (ndocs, H,
    P, N).  Returns a dict with dx, ddt, dA, dB, dC, dD (None without D) and
    dinit (by default for batch rows, or for documents with initial_states).
    split_len: tokens per sequence split of the tensor-core backward (0:
    automatic); it changes only the rounding.  With check_status, also
    synchronises the stream and raises if a device-side wait ran out (the
    workspace's status word)."""
    batch, seqlen, nheads, headdim = x.shape
    ngroups, dstate = B.shape[2], B.shape[3]
    dev = x.device
    ndocs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    if want_dinit is None:
        want_dinit = cu_seqlens is None or initial_states is not None
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or cu_seqlens.device != dev):
        raise ValueError("cu_seqlens: expected int32 (ndocs + 1) on the device")
    params = _lib.make_params(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, split_len, ndocs,
                              _dtype_code(x))
    shp_x, shp_bc = (batch, seqlen, nheads, headdim), (batch, seqlen, ngroups, dstate)
    shp_s = (batch if cu_seqlens is None else ndocs, nheads, headdim, dstate)
    for name, t, shp, dt_ in (("x", x, shp_x, x.dtype), ("dt", dt, shp_x[:3], torch.float32),
                              ("A", A, (nheads,), torch.float32), ("B", B, shp_bc, x.dtype),
                              ("C", C, shp_bc, x.dtype), ("dy", dy, shp_x, x.dtype),
                              ("D", D, (nheads,), torch.float32),
                              ("initial_states", initial_states, shp_s, torch.float32),
                              ("dfinal_states", dfinal_states, shp_s, torch.float32)):
        if t is None:
            continue
        if tuple(t.shape) != shp or t.dtype != dt_ or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"{name}: expected contiguous {dt_} {shp} on {dev}, got "
                             f"{t.dtype} {tuple(t.shape)} on {t.device}")
    doc_states = cu_seqlens is not None and (initial_states is not None or dfinal_states is not None or want_dinit)
    size_fn = _lib.lib.ssd_bwd_workspace_size_doc_states if doc_states else _lib.lib.ssd_bwd_workspace_size
    nbytes = int(size_fn(ctypes.byref(params)))
    if nbytes == 0:
        raise _lib.SSDError(2, "ssd_bwd: unsupported parameters")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    g = dict(dx=torch.empty_like(x), ddt=torch.empty_like(dt), dA=torch.empty_like(A),
             dB=torch.empty_like(B), dC=torch.empty_like(C), dD=None if D is None else torch.empty_like(D),
             dinit=torch.empty(shp_s, dtype=torch.float32, device=dev) if want_dinit else None)
    rc = _lib.lib.ssd_bwd(ctypes.byref(params), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                          _ptr(initial_states), _ptr(cu_seqlens), _ptr(dy), _ptr(dfinal_states), _ptr(g["dx"]),
                          _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
                          _ptr(g["dinit"]), _ptr(ws), nbytes, _stream_handle(stream))
    _lib.check(rc, "ssd_bwd")
    if check_status:
        _lib.check(_lib.lib.ssd_check_status(_ptr(ws), _stream_handle(stream)), "ssd_bwd device status")
    return g


def gate_norm(y, z, weight, group_size, eps=1e-5, *, out=None, stream=None):
    """out = rmsnorm_groups(y * silu(z)) * weight over the last dimension, in one
    pass (groups of `group_size` channels).  y, z: (..., width) bf16 or fp32,
    contiguous; weight: (width,) fp32.  `out` may be y (in place)."""
    width = y.shape[-1]
    rows = y.numel() // width if width else 0
    if tuple(z.shape) != tuple(y.shape) or z.dtype != y.dtype or not (y.is_contiguous() and z.is_contiguous()):
        raise ValueError("z: expected the shape, dtype and layout of y")
    if weight.dtype != torch.float32 or tuple(weight.shape) != (width,) or weight.device != y.device:
        raise ValueError("weight: expected fp32 (width,) on y's device")
    if out is None:
        out = torch.empty_like(y)
    rc = _lib.lib.ssd_gate_norm(rows, width, int(group_size), _dtype_code(y), _ptr(y), _ptr(z), _ptr(weight),
                                float(eps), _ptr(out), _stream_handle(stream))
    _lib.check(rc, "ssd_gate_norm")
    return out


def ssd_step(state, x, dt, A, B, C, D=None, *, state_out=None, y=None, stream=None):
    """One decode step: a new token per batch row from the resident state.

    state (batch, H, P, N) fp32 is updated in place unless ``state_out`` (same
    shape, disjoint) is given; x (batch, H, P), dt (batch, H), A (H),
    B/C (batch, G, N), D (H) or None.  Returns y (batch, H, P) in x's dtype.
    """
    batch, nheads, headdim = x.shape
    ngroups, dstate = B.shape[1], B.shape[2]
    dev = x.device
    if state_out is None:
        state_out = state
    for name, t, shp, dt_ in (("state", state, (batch, nheads, headdim, dstate), torch.float32),
                              ("state_out", state_out, (batch, nheads, headdim, dstate), torch.float32),
                              ("x", x, (batch, nheads, headdim), x.dtype),
                              ("dt", dt, (batch, nheads), torch.float32), ("A", A, (nheads,), torch.float32),
                              ("B", B, (batch, ngroups, dstate), x.dtype), ("C", C, (batch, ngroups, dstate), x.dtype),
                              ("D", D, (nheads,), torch.float32), ("y", y, (batch, nheads, headdim), x.dtype)):
        if t is None:
            continue
        if tuple(t.shape) != shp or t.dtype != dt_ or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"{name}: expected contiguous {dt_} {shp} on {dev}, got "
                             f"{t.dtype} {tuple(t.shape)} on {t.device}")
    if y is None:
        y = torch.empty((batch, nheads, headdim), dtype=x.dtype, device=dev)
    rc = _lib.lib.ssd_step(batch, nheads, headdim, dstate, ngroups, _dtype_code(x), _ptr(state), _ptr(state_out),
                           _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(y), _stream_handle(stream))
    _lib.check(rc, "ssd_step")
    return y


def check_status(workspace: torch.Tensor, stream=None) -> int:
    return int(_lib.lib.ssd_check_status(_ptr(workspace), _stream_handle(stream)))


def plan(params) -> tuple:
    return _lib.plan(params)


def segsum_dump(log2decay: torch.Tensor, want_seg=True, want_L=True, want_factors=False, stream=None):
    """Run the hierarchy-aware segsum device routines on rows of log2-decays
    (nrows, chunk) fp32.  Returns (seg, L) — the log-domain routine's seg and
    the linear-domain routine's mask, each (nrows, chunk, chunk) or None — and,
    with want_factors, also the linear-domain row prefixes and column suffixes
    (nrows, chunk) as (seg, L, pexp, sfx)."""
    if log2decay.dtype != torch.float32 or log2decay.dim() != 2 or not log2decay.is_contiguous():
        raise ValueError("log2decay: contiguous fp32 (nrows, chunk)")
    nrows, q = log2decay.shape
    dev = log2decay.device
    seg = torch.empty((nrows, q, q), dtype=torch.float32, device=dev) if want_seg else None
    L = torch.empty((nrows, q, q), dtype=torch.float32, device=dev) if want_L else None
    pexp = torch.empty((nrows, q), dtype=torch.float32, device=dev) if want_factors else None
    sfx = torch.empty((nrows, q), dtype=torch.float32, device=dev) if want_factors else None
    rc = _lib.lib.ssd_segsum_dump(_ptr(log2decay), nrows, q, _ptr(seg), _ptr(L), _ptr(pexp), _ptr(sfx),
                                  _stream_handle(stream))
    _lib.check(rc, "ssd_segsum_dump")
    if want_factors:
        return seg, L, pexp, sfx
    return seg, L
