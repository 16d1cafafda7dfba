"""ssd_fwd_timed: the same results as ssd_fwd, bit for bit, with one positive
duration per kernel launch of the plan.  (In split plans whose aggregates run
on the tensor-core aggregate kernel, ssd_fwd starts the later launches as
programmatic dependents of the one before; the timed call's events serialise
them, so these cases also check the dependent launches against plain stream
order.)"""
import numpy as np
import pytest
import torch

import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("batch,seqlen,split_len", [(2, 300, 0), (1, 1000, 256), (3, 512, 1 << 16), (1, 4096, 512)])
def test_timed_matches_plain(batch, seqlen, split_len):
    p = synth.make_problem(batch=batch, seqlen=seqlen, nheads=8, headdim=64, dstate=128, ngroups=2, chunk=128,
                           dtype="bf16", seed=401, init_std=0.1)
    d = to_device(p)
    f = ssd.SSDForward(p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, 128, split_len, 0,
                       torch.bfloat16)
    fin1 = torch.empty((p.batch, p.nheads, p.headdim, p.dstate), dtype=torch.float32, device="cuda")
    fin2 = torch.empty_like(fin1)
    y1 = f(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], None, final_states=fin1)
    y2 = torch.empty_like(y1)
    ms = f.launch_times(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], None, y=y2, final_states=fin2)
    assert f.check_status() == 0
    _, launches, _ = f.plan(True, True)
    assert len(ms) == launches and all(t > 0 for t in ms)
    assert torch.equal(y1, y2) and torch.equal(fin1, fin2)


def test_timed_matches_plain_documents():
    """Packed documents with initial and final states in a split plan: the
    tensor-core split aggregates, the document-start aggregates, the scan and
    the full pass (dependent launches in the plain call)."""
    lens = [700, 900, 1200, 1296]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=8, headdim=64, dstate=128, ngroups=2, chunk=128,
                           dtype="bf16", seed=403, init_std=0.1, doc_lengths=lens)
    d = to_device(p)
    f = ssd.SSDForward(1, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, 128, 512, len(lens), torch.bfloat16)
    fin1 = torch.empty((len(lens), p.nheads, p.headdim, p.dstate), dtype=torch.float32, device="cuda")
    fin2 = torch.empty_like(fin1)
    y1 = f(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], d["cu"], final_states=fin1)
    y2 = torch.empty_like(y1)
    ms = f.launch_times(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], d["cu"], y=y2,
                        final_states=fin2)
    assert f.check_status() == 0
    assert len(ms) == 4 and all(t > 0 for t in ms)   # aggregates, document starts, scan, full pass
    assert torch.equal(y1, y2) and torch.equal(fin1, fin2)
