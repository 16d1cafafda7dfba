"""GPU parity of the persistent grid of the tensor-core kernel.

Split plans whose units (batch row, head, split) are at most 4 chunks long and
outnumber the SMs run on a persistent grid: one CTA per SM walks the units
k, k + grid, ... and keeps its pipeline running across unit boundaries (the
incoming state, the decay rate A_h, D_h and the document cursor all change at
each boundary).  These cases check every output against the fp64 oracle:
initial and final states, a last split shorter than the others, several
groups, and packed documents cut by the splits.
"""
import numpy as np
import pytest
import torch

import oracle
from mamba_ssd_chunked_scan_gb300 import synth

from gpu_helpers import TOL, rel_err, run

pytestmark = pytest.mark.gpu


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def check(p, split_len):
    y_o, f_o = oracle.ssd_recurrence(p, want_final=True)
    for _ in range(2):
        y_g, f_g, f = run(p, want_final=True, split_len=split_len)
        assert np.isfinite(y_g).all() and np.isfinite(f_g).all()
        ey, ef = rel_err(y_g, y_o), rel_err(f_g, f_o)
        assert ey <= TOL["bf16"], f"y err {ey:.3e}"
        assert ef <= TOL["bf16"], f"final state err {ef:.3e}"
    return f


@pytest.mark.parametrize("seqlen,split_len", [(1024, 128), (3 * 256 + 41, 256), (2 * 512 + 130, 512)])
def test_persistent_short_splits_with_states(seqlen, split_len):
    nsplit = (seqlen + split_len - 1) // split_len
    H = 8
    batch = max(1, (2 * sm_count()) // (H * nsplit) + 1)   # more units than SMs
    p = synth.make_problem(batch=batch, seqlen=seqlen, nheads=H, headdim=64, dstate=128, ngroups=2,
                           chunk=128, dtype="bf16", seed=95, init_std=0.1)
    assert batch * H * nsplit > sm_count()
    f = check(p, split_len)
    assert f.plan()[2] == nsplit


def test_persistent_packed_documents():
    lens = [3, 300, 128, 1, 257, 90, 500]    # ends before, on and after chunk and split edges
    H = 2 * sm_count() // 10 + 1
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=H, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=97, doc_lengths=lens)
    f = check(p, 128)
    assert f.plan()[2] * H > sm_count()
