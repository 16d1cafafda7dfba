"""ssd_fwd_static_scratch: the entry point for callers that cannot allocate
device memory (for example a plugin whose host application owns every device
allocation).  Its workspace is a library-owned device array, so the caller
passes only inputs and outputs.

Checked through the C ABI against ssd_fwd with a caller-owned workspace, on
two calls in a row (the array keeps the previous call's contents), with a
problem that uses the split-sequence scratch, plus the size limit.
"""
import ctypes

import numpy as np
import pytest
import torch

import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import _lib, synth

from gpu_helpers import TOL, rel_err, run, to_device

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_call(p, split_len):
    d = to_device(p)
    dtype = torch.bfloat16 if p.dtype == "bf16" else torch.float32
    params = _lib.make_params(p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk,
                              split_len, p.ndocs, _lib.SSD_BF16 if p.dtype == "bf16" else _lib.SSD_F32)
    y = torch.full(d["x"].shape, float("nan"), dtype=dtype, device="cuda")
    fin = torch.full((p.nstates, p.nheads, p.headdim, p.dstate), float("nan"), dtype=torch.float32,
                     device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _lib.lib.ssd_fwd_static_scratch(ctypes.byref(params), _ptr(d["x"]), _ptr(d["dt"]), _ptr(d["A"]),
                                         _ptr(d["B"]), _ptr(d["C"]), _ptr(d["D"]), _ptr(d["init"]),
                                         _ptr(d["cu"]), _ptr(y), _ptr(fin), stream)
    assert rc == 0, _lib.STATUS.get(rc, rc)
    return y.float().cpu().numpy().astype(np.float64), fin.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("split_len", [256, 0])
def test_static_scratch_matches_caller_workspace(split_len):
    p = synth.make_problem(batch=2, seqlen=1000, nheads=3, headdim=64, dstate=128, ngroups=1, chunk=128,
                           dtype="bf16", seed=71, init_std=0.1)
    y_ref, f_ref, f = run(p, split_len=split_len)
    if split_len:
        assert f.plan()[2] > 1   # the split buffers of the scratch are in use
    for _ in range(2):
        y, fin = _static_call(p, split_len)
        assert rel_err(y, y_ref) <= TOL["bf16"]
        assert rel_err(fin, f_ref) <= TOL["bf16"]
        assert np.array_equal(y, y_ref) and np.array_equal(fin, f_ref)


def test_static_scratch_fp32_varlen():
    lens = [5, 70, 64, 100]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=2, headdim=16, dstate=16, ngroups=1, chunk=64,
                           dtype="f32", seed=73, xbc="unit", dt_dist="softplus_m2", A_dist="exp",
                           doc_lengths=lens, init_std=0.3)
    y_ref, f_ref, _ = run(p, split_len=64)
    for _ in range(2):
        y, fin = _static_call(p, 64)
        assert rel_err(y, y_ref) <= TOL["f32"]
        assert rel_err(fin, f_ref) <= TOL["f32"]


def test_static_scratch_rejects_oversize_problems():
    # 1 row x 32 heads x 64 splits of 64 x 128 fp32 states: 32 MiB of split buffers
    params = _lib.make_params(1, 64 * 128, 32, 64, 128, 1, 128, 128, 0, _lib.SSD_BF16)
    assert _lib.workspace_size(params) > 8 << 20
    rc = _lib.lib.ssd_fwd_static_scratch(ctypes.byref(params), *([ctypes.c_void_p(0x10000)] * 10), None)
    assert rc == 3   # SSD_ERR_WORKSPACE, before any launch
