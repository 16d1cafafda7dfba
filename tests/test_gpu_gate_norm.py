"""GPU parity of the gated RMS normalisation (ssd_gate_norm) against the fp64
oracle: full-width groups (the Mamba-2 2.7B block norms all 5120 channels of a
token) and per-head groups, both storage types, in place and out of place."""
import numpy as np
import pytest
import torch

import oracle
import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


def data(rows, width, dtype, seed):
    r = np.random.default_rng(seed)
    y = r.standard_normal((rows, width)).astype(np.float32)
    z = (r.standard_normal((rows, width)) * 2).astype(np.float32)
    w = r.uniform(0.5, 1.5, width).astype(np.float32)
    if dtype == "bf16":
        yb, zb = synth.bf16_bits(y), synth.bf16_bits(z)
        y, z = synth.bf16_to_f32(yb), synth.bf16_to_f32(zb)
        yt = torch.from_numpy(yb.view(np.int16).copy()).cuda().view(torch.bfloat16)
        zt = torch.from_numpy(zb.view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        yt, zt = torch.from_numpy(y).cuda(), torch.from_numpy(z).cuda()
    return y, z, w, yt, zt, torch.from_numpy(w).cuda()


@pytest.mark.parametrize("rows,width,group,dtype", [
    (37, 5120, 5120, "bf16"),    # one group per token: all heads of the 2.7B-like layer
    (100, 512, 64, "bf16"),      # one group per head
    (9, 8192, 8192, "f32"),      # the largest group
    (3, 24, 8, "f32"),           # groups smaller than a warp's worth of vectors
    (5, 200, 40, "bf16"),        # a group that is not a power of two
])
def test_gate_norm_parity(rows, width, group, dtype):
    y, z, w, yt, zt, wt = data(rows, width, dtype, seed=rows + width)
    got = ssd.gate_norm(yt, zt, wt, group, 1e-5).float().cpu().numpy()
    want = oracle.gate_norm(y, z, w, group, 1e-5)
    err = float(np.abs(got - want).max() / np.abs(want).max())
    assert np.isfinite(got).all() and err <= TOL[dtype], err


def test_gate_norm_in_place():
    _, _, _, yt, zt, wt = data(16, 5120, "bf16", seed=5)
    out = ssd.gate_norm(yt, zt, wt, 5120)
    ssd.gate_norm(yt, zt, wt, 5120, out=yt)
    assert torch.equal(out, yt)
