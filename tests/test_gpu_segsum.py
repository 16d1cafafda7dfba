"""The hierarchy-aware segsum device routines (through ssd_segsum_dump), both
forms that the forward kernels run:

- the log-domain routine (the SIMT kernel exponentiates its seg): zero strict
  monotonicity violations, accuracy inside the recursive-summation bound;
- the linear-domain routine (the tensor-core kernel multiplies in its row and
  column factors): zero strict row and column inversions of the mask, exact
  zeros above the diagonal and ones on it, 0 <= L <= 1, and every entry within
  the product-rounding bound of the exact product of its factors;

on stress rows where the prefix-subtraction (diff) comparator fails.
"GPU Hierarchy Meets Structured Matrices" (abstract): hierarchy-aware segsum
versus diff segsum."""
import numpy as np
import pytest
import torch

import oracle
import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

from test_oracle_segsum import violations

pytestmark = pytest.mark.gpu
LOG2E = np.float32(1.4426950408889634)
U = 2.0 ** -24


def gamma(n):
    return n * U / (1 - n * U)


def rows_for(family, Q):
    if family == "stress":
        rows = synth.stress_logdecay_rows(10000, Q, seed=100 + Q)
    else:
        rows = synth.varlen_logdecay_rows(10000, Q, seed=200 + Q)
    return (rows * LOG2E).astype(np.float32)


def diff_failures(l2, exact):
    """Strict violations plus summation-bound failures of the diff comparator."""
    Q = l2.shape[1]
    i, j = np.tril_indices(Q)
    e = exact[:, i, j]
    fin = np.isfinite(e)
    diff = oracle.diff_segsum_f32(l2).astype(np.float64)
    derr = np.abs(diff[:, i, j] - e)
    with np.errstate(invalid="ignore"):
        return violations(diff.astype(np.float32)) + np.count_nonzero(~(derr[fin] <= gamma(Q - 1) * np.abs(e[fin])))


@pytest.mark.parametrize("Q", [64, 128])
@pytest.mark.parametrize("family", ["stress", "varlen"])
def test_log_domain_no_violations_where_diff_fails(Q, family):
    l2 = rows_for(family, Q)
    seg, _ = ssd.segsum_dump(torch.from_numpy(l2).cuda(), want_L=False)
    torch.cuda.synchronize()
    seg = seg.cpu().numpy()
    assert violations(seg) == 0
    # accuracy: a same-sign sum along a path of fewer than Q terms, so within gamma_{Q-1}
    exact = oracle.segsum(l2.astype(np.float64))
    i, j = np.tril_indices(Q)
    e, g = exact[:, i, j], seg[:, i, j].astype(np.float64)
    fin = np.isfinite(e)
    assert np.array_equal(np.isneginf(g), np.isneginf(e))
    assert np.all(np.abs(g[fin] - e[fin]) <= gamma(Q - 1) * np.abs(e[fin]))
    assert np.all(np.isneginf(seg[:, ~np.tril(np.ones((Q, Q), bool))]))
    bad = diff_failures(l2, exact)
    assert bad > 0
    print(f"Q={Q} {family}: log-domain violations 0, diff-segsum failures {bad}")


def exact_products(a):
    """prod_{k=j+1..i} a_k for j <= i (fp64, exact up to ~1e-12 relative), 0 above."""
    nrows, Q = a.shape
    lg = np.where(a > 0, np.log(np.where(a > 0, a, 1.0)), -1.0e4)   # a zero factor kills the product
    cs = np.cumsum(lg, axis=1)
    with np.errstate(over="ignore", under="ignore"):
        P = np.exp(cs[:, :, None] - cs[:, None, :])
    return np.where(np.tril(np.ones((Q, Q), bool))[None], P, 0.0)


@pytest.mark.parametrize("Q", [64, 128])
@pytest.mark.parametrize("family", ["stress", "varlen"])
def test_linear_domain_mask_as_the_tensor_core_kernel_forms_it(Q, family):
    l2 = rows_for(family, Q)
    _, L, pexp, sfx = ssd.segsum_dump(torch.from_numpy(l2).cuda(), want_seg=False, want_factors=True)
    torch.cuda.synchronize()
    L, pexp, sfx = L.cpu().numpy(), pexp.cpu().numpy(), sfx.cpu().numpy()
    low = np.tril(np.ones((Q, Q), bool))
    # structure: exact zeros above the diagonal, exact ones on it, within [0, 1]
    assert np.all(L[:, ~low] == 0.0)
    assert np.all(L[:, np.arange(Q), np.arange(Q)] == 1.0)
    assert np.all(L >= 0.0) and np.all(L <= 1.0)
    # strict monotonicity, no tolerance: along rows (L(i, j) <= L(i, j+1)) and
    # down columns (L(i+1, j) <= L(i, j)), on and below the diagonal
    row_inv = int(np.count_nonzero((L[:, :, :-1] > L[:, :, 1:]) & low[None, :, 1:]))
    col_inv = int(np.count_nonzero((L[:, 1:, :] > L[:, :-1, :]) & low[None, :-1, :]))
    assert row_inv == 0 and col_inv == 0
    assert np.all(np.diff(pexp, axis=1) <= 0) and np.all(pexp <= 1.0) and np.all(pexp >= 0.0)
    assert np.all(np.diff(sfx, axis=1) >= 0) and np.all(sfx[:, -1] == 1.0)
    # the factors: the entry beside the diagonal is exactly one factor a_k, and
    # a_k is ex2(l_k) within the instruction's error (or flushed below 2^-126)
    a = np.empty((l2.shape[0], Q), np.float64)
    a[:, 1:] = L[:, np.arange(1, Q), np.arange(Q - 1)]
    a[:, 0] = pexp[:, 0]
    ref = np.exp2(l2.astype(np.float64))
    normal = ref >= 2.0 ** -125
    assert np.all(np.abs(a[normal] - ref[normal]) <= 2.0 ** -21 * ref[normal])
    assert np.all(a[~normal] <= 2.0 ** -125)
    assert np.all(a[np.isneginf(l2)] == 0.0)
    # every entry is the product of its factors within the rounding of at most
    # Q + 1 multiplications (plus the subnormal range's absolute error)
    slack = 2.0 ** -120
    for r0 in range(0, a.shape[0], 1000):   # in blocks of rows, to bound host memory
        ex = exact_products(a[r0:r0 + 1000])
        assert np.all(np.abs(L[r0:r0 + 1000] - ex) <= gamma(Q + 1) * ex + slack)
    pref = np.concatenate([np.ones((a.shape[0], 1)), np.cumprod(a, axis=1)], axis=1)[:, 1:]
    assert np.all(np.abs(pexp - pref) <= gamma(Q + 1) * pref + slack)
    suf = np.ones_like(a)
    for jj in range(Q - 2, -1, -1):
        suf[:, jj] = suf[:, jj + 1] * a[:, jj + 1]
    assert np.all(np.abs(sfx - suf) <= gamma(Q + 1) * suf + slack)
    # the prefix-subtraction comparator fails on the same rows
    bad = diff_failures(l2, oracle.segsum(l2.astype(np.float64)))
    assert bad > 0
    print(f"Q={Q} {family}: linear-domain row inversions {row_inv}, column inversions {col_inv}, "
          f"diff-segsum failures {bad}")
