"""The hierarchy-aware segsum device routine (through ssd_segsum_dump):
zero strict log-domain monotonicity violations on stress rows where the
prefix-subtraction comparator fails, accuracy inside the recursive-summation
bound, and the exact mask structure."""
import numpy as np
import pytest
import torch

import oracle
import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

from test_oracle_segsum import violations

pytestmark = pytest.mark.gpu
LOG2E = np.float32(1.4426950408889634)


def dump(rows_l2):
    seg, L = ssd.segsum_dump(torch.from_numpy(rows_l2).cuda())
    torch.cuda.synchronize()
    return seg.cpu().numpy(), L.cpu().numpy()


@pytest.mark.parametrize("Q", [64, 128])
@pytest.mark.parametrize("family", ["stress", "varlen"])
def test_no_violations_where_diff_fails(Q, family):
    if family == "stress":
        rows = synth.stress_logdecay_rows(10000, Q, seed=100 + Q)
    else:
        rows = synth.varlen_logdecay_rows(10000, Q, seed=200 + Q)
    l2 = (rows * LOG2E).astype(np.float32)
    seg, L = dump(l2)
    assert violations(seg) == 0
    # structure of the mask the kernels multiply in
    up = np.triu(np.ones((Q, Q), bool), 1)
    assert np.all(L[:, up] == 0.0)
    assert np.all(L[:, np.arange(Q), np.arange(Q)] == 1.0)
    assert np.all(L <= 1.0) and np.all(L >= 0.0)
    # accuracy: a same-sign sum along a tree of height < Q, so within gamma_{Q-1}
    exact = oracle.segsum(l2.astype(np.float64))
    i, j = np.tril_indices(Q)
    e, g = exact[:, i, j], seg[:, i, j].astype(np.float64)
    fin = np.isfinite(e)
    assert np.array_equal(np.isneginf(g), np.isneginf(e))
    gamma = ((Q - 1) * 2.0 ** -24) / (1 - (Q - 1) * 2.0 ** -24)
    assert np.all(np.abs(g[fin] - e[fin]) <= gamma * np.abs(e[fin]))
    # the prefix-subtraction comparator on the same rows fails
    diff = oracle.diff_segsum_f32(l2).astype(np.float64)
    derr = np.abs(diff[:, i, j] - e)
    with np.errstate(invalid="ignore"):
        bad = violations(diff.astype(np.float32)) + np.count_nonzero(~(derr[fin] <= gamma * np.abs(e[fin])))
    assert bad > 0
    # L-domain row monotonicity is reported (exp2's own monotonicity is not ours)
    Lrow = int(np.count_nonzero((L[:, :, :-1] > L[:, :, 1:]) & np.tril(np.ones((Q, Q), bool))[None, :, 1:]))
    print(f"Q={Q} {family}: log-domain violations 0, diff-segsum failures {bad}, "
          f"L-domain row inversions {Lrow}")
