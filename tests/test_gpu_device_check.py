"""The device-side check of packed-document offsets.  cu_seqlens lives in
device memory, so the host cannot validate it; the last launch of a forward
or backward call checks 0 = cu[0] < cu[1] < ... < cu[ndocs] = seqlen and, on
a violation, records SSD_ERR_DEVICE_CHECK (where code 40) in the workspace
status word.  Every kernel that reads the offsets keeps its indexes in bounds
whatever they hold (the results are then undefined), so these cases fault
nothing, and the next call with valid offsets on the same workspace is clean."""
import numpy as np
import pytest
import torch

import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu
SSD_ERR_DEVICE_CHECK = 6
WHERE_CU_SEQLENS = 40
L = 256

# an empty document, offsets that end before the row's end, a first offset that is not 0
BAD = [[0, 100, 100, 256], [0, 100, 200], [5, 100, 256]]


def problem(dtype, headdim, dstate):
    return synth.make_problem(batch=1, seqlen=L, nheads=4, headdim=headdim, dstate=dstate, ngroups=1, chunk=128,
                              dtype=dtype, seed=41, doc_lengths=[100, 80, 76])


def valid_offsets(ndocs):
    return torch.tensor(np.linspace(0, L, ndocs + 1).astype(np.int32), device="cuda")


@pytest.mark.parametrize("dtype,headdim,dstate,states", [
    ("bf16", 64, 128, False),   # tensor-core forward, packed documents
    ("bf16", 64, 128, True),    # its document-event instance (initial and final states)
    ("f32", 16, 32, True),      # CUDA-core forward
])
@pytest.mark.parametrize("cu_bad", BAD)
def test_forward_reports_invalid_offsets(dtype, headdim, dstate, states, cu_bad):
    p = problem(dtype, headdim, dstate)
    d = to_device(p)
    ndocs = len(cu_bad) - 1
    f = ssd.SSDForward(1, L, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0, ndocs,
                       torch.bfloat16 if dtype == "bf16" else torch.float32, "cuda")
    shp = (ndocs, p.nheads, p.headdim, p.dstate)
    init = torch.randn(shp, device="cuda") * 0.3 if states else None
    fin = torch.empty(shp, device="cuda") if states else None
    cu = torch.tensor(cu_bad, dtype=torch.int32, device="cuda")
    f(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], init, cu, final_states=fin)
    assert f.check_status_where() == (SSD_ERR_DEVICE_CHECK, WHERE_CU_SEQLENS)
    f(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], init, valid_offsets(ndocs), final_states=fin)
    assert f.check_status_where() == (0, 0)


@pytest.mark.parametrize("states", [False, True])   # tensor-core backward; CUDA-core (per-document states)
@pytest.mark.parametrize("cu_bad", BAD)
def test_backward_reports_invalid_offsets(states, cu_bad):
    p = problem("bf16", 64, 128)
    d = to_device(p)
    ndocs = len(cu_bad) - 1
    dy = (torch.randn(d["x"].shape, device="cuda")).to(torch.bfloat16)
    init = torch.randn((ndocs, p.nheads, p.headdim, p.dstate), device="cuda") * 0.3 if states else None
    cu = torch.tensor(cu_bad, dtype=torch.int32, device="cuda")
    with pytest.raises(ssd._lib.SSDError) as e:
        ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"], init, None, cu, check_status=True)
    assert e.value.code == SSD_ERR_DEVICE_CHECK
    g = ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dy, d["D"], init, None, valid_offsets(ndocs),
                    check_status=True)
    assert torch.isfinite(g["dx"].float()).all()
