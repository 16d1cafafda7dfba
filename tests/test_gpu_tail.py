"""GPU parity of the leftover-unit plan of the tensor-core kernel.

With one split and a (row, head) unit count U that is not a multiple of the
SM count S, the last U % S units are cut into pieces (their split aggregates,
the composition, then the whole units and the pieces in one launch), so the
last wave is short.  These cases check every output against the fp64 oracle:
whole and cut units side by side, initial and final states, a ragged last
chunk, and packed documents whose boundaries fall inside the cut units.
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


ONE_SPLIT = 1 << 16   # split_len >= seqlen: one split (the automatic plan would split these sizes)


def check(p, launches_expected=3):
    y_o, f_o = oracle.ssd_recurrence(p, want_final=True)
    for _ in range(2):
        y_g, f_g, f = run(p, want_final=True, split_len=ONE_SPLIT)
        assert np.isfinite(y_g).all() and np.isfinite(f_g).all()
        ey, ef = rel_err(y_g, y_o), rel_err(f_g, f_o)
        assert ey <= TOL["bf16"], f"y err {ey:.3e}"
        assert ef <= TOL["bf16"], f"final state err {ef:.3e}"
    fam, launches, ns = f.plan(p.initial_states is not None, True)
    assert fam == 1 and ns == 1 and launches == launches_expected   # the plan is in use


@pytest.mark.parametrize("seqlen", [1024, 1000 + 37])
def test_tail_units_with_states(seqlen):
    H = 8
    batch = sm_count() // H + 1                   # U = S + (a few leftover units)
    p = synth.make_problem(batch=batch, seqlen=seqlen, nheads=H, headdim=64, dstate=128, ngroups=2,
                           chunk=128, dtype="bf16", seed=101, init_std=0.1)
    assert (batch * H) % sm_count() != 0
    check(p)


def test_tail_units_packed_documents():
    lens = [3, 300, 128, 1, 257, 90, 500]
    H = sm_count() + 5
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=H, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=103, doc_lengths=lens)
    check(p)


def test_tail_units_packed_documents_with_init_states():
    # documents with their own initial states, starting inside and at the edges of
    # the cut units' pieces (their aggregates then take the initial states too)
    lens = [3, 300, 128, 1, 257, 90, 500]
    H = sm_count() + 5
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=H, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=104, doc_lengths=lens, init_std=1.0)
    check(p, launches_expected=4)
