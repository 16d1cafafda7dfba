"""Shared helpers of the GPU parity tests: move a synthetic problem to the
device, run it through the C ABI, and measure errors against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import mamba_ssd_chunked_scan_gb300 as ssd

TOL = {"f32": 1e-5, "bf16": 2e-2}


def to_device(p, device="cuda"):
    """Device tensors holding exactly the bytes the oracle reads."""
    def t(a, dtype=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)

    if p.dtype == "bf16":
        def io(name):
            bits = p.storage(name).view(np.int16)
            return torch.from_numpy(bits.copy()).to(device).view(torch.bfloat16)
    else:
        def io(name):
            return t(getattr(p, name))
    d = dict(x=io("x"), B=io("B"), C=io("C"), dt=t(p.dt), A=t(p.A), D=t(p.D), init=t(p.initial_states))
    d["cu"] = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens.copy()).to(device)
    return d


def run(p, want_final=True, split_len=None, chunk=None, use_init=True, device="cuda"):
    d = to_device(p, device)
    dtype = torch.bfloat16 if p.dtype == "bf16" else torch.float32
    f = ssd.SSDForward(p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups,
                       chunk or p.chunk, p.split_len if split_len is None else split_len, p.ndocs,
                       dtype, device)
    fin = None
    if want_final:
        fin = torch.full((p.nstates, p.nheads, p.headdim, p.dstate), float("nan"), dtype=torch.float32,
                         device=device)
    y = f(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"] if use_init else None, d["cu"],
          final_states=fin)
    st = f.check_status()
    assert st == 0, f"device status {st}"
    torch.cuda.synchronize()
    yn = y.float().cpu().numpy().astype(np.float64)
    fn = None if fin is None else fin.cpu().numpy().astype(np.float64)
    return yn, fn, f


def rel_err(got, want):
    """max |got - want| / max |want| over the whole tensor."""
    return float(np.abs(got - want).max() / max(np.abs(want).max(), 1e-30))
