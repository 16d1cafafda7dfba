"""Pins for the oracle's segsum and for the diff-segsum comparator.

seg(i, j) = sum_{k=j+1..i} l_k (j <= i) is the log of the 1-semiseparable
decay mask L_ij = prod_{k=j+1..i} a_k ("State Space Duality and Mamba-2",
the Hadamard factorisation M = (C B^T) o L).  "GPU Hierarchy Meets Structured
Matrices" (abstract) contrasts the stable direct form with the fast
prefix-subtraction (diff) form, which suffers monotonicity violations and
catastrophic cancellation.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from mamba_ssd_chunked_scan_gb300 import synth


def violations(seg):
    """Strict log-domain monotonicity violations of seg (nrows, Q, Q)."""
    Q = seg.shape[-1]
    low = np.tril(np.ones((Q, Q), dtype=bool))
    with np.errstate(invalid="ignore"):
        # row: seg(i, j) <= seg(i, j+1) for j+1 <= i
        row = (seg[:, :, :-1] > seg[:, :, 1:]) & low[None, :, 1:]
        # column: seg(i+1, j) <= seg(i, j) for j <= i
        col = (seg[:, 1:, :] > seg[:, :-1, :]) & low[None, :-1, :]
        pos = (seg > 0) & low[None]
        nan = np.isnan(seg) & low[None]
    return int(row.sum() + col.sum() + pos.sum() + nan.sum())


def test_structure_random():
    g = np.random.default_rng(0)
    ell = -g.exponential(1.0, size=(20, 64))
    seg = oracle.segsum(ell)
    Q = 64
    for r in range(20):
        assert np.all(np.diag(seg[r]) == 0.0)
        assert np.all(np.isneginf(seg[r][np.triu_indices(Q, 1)]))
    assert violations(seg) == 0
    L = np.exp(seg)
    assert np.all(L <= 1.0) and np.all(L[:, np.triu(np.ones((Q, Q), bool), 1)] == 0.0)


def test_exact_on_integers():
    """Integer-valued l: every partial sum is exact in fp64; compare to exact rationals."""
    g = np.random.default_rng(1)
    ell = -g.integers(0, 1000, size=(5, 48)).astype(np.float64)
    seg = oracle.segsum(ell)
    for r in range(5):
        for i in range(48):
            for j in range(i + 1):
                want = sum(Fraction(int(v)) for v in ell[r, j + 1:i + 1])
                assert seg[r, i, j] == float(want)


def test_constant_decay_geometric():
    """Constant l gives L_ij = exp((i - j) l): a geometric decay mask."""
    l = -0.37
    Q = 128
    seg = oracle.segsum(np.full((1, Q), l))
    i, j = np.tril_indices(Q)
    exact = (i - j) * l
    gamma = (Q * 2.0 ** -53) / (1 - Q * 2.0 ** -53)
    assert np.all(np.abs(seg[0, i, j] - exact) <= gamma * np.abs(exact) + 1e-300)
    np.testing.assert_allclose(np.exp(seg[0, i, j]), np.exp(l) ** (i - j), rtol=1e-12)


def test_document_start_masks_mask():
    """A -inf log-decay (document start at k) zeroes every L_ij with j < k <= i."""
    ell = np.full((1, 16), -0.1)
    ell[0, 6] = -np.inf
    L = np.exp(oracle.segsum(ell))[0]
    for i in range(16):
        for j in range(i + 1):
            assert (L[i, j] == 0.0) == (j < 6 <= i)


def test_diff_segsum_fails_on_stress_rows():
    """The comparator must be shown failing where the direct form does not."""
    rows = synth.stress_logdecay_rows(2000, 128)
    seg_d = oracle.segsum(rows.astype(np.float64))
    assert violations(seg_d) == 0
    seg_f = oracle.diff_segsum_f32(rows)
    # -inf rows: the subtraction produces NaN (-inf - -inf)
    assert violations(seg_f) > 0


def test_diff_segsum_cancellation_varlen_regime():
    """Per-chunk sums near -1e3: diff segsum loses the small near-diagonal
    entries (error ~ u |cum|, far beyond the summation bound gamma_{Q-1}|seg|),
    while the fp32 values of a direct sum stay inside that bound."""
    rows = synth.varlen_logdecay_rows(500, 128)
    Q = 128
    exact = oracle.segsum(rows.astype(np.float64))
    seg_f = oracle.diff_segsum_f32(rows).astype(np.float64)
    i, j = np.tril_indices(Q, -1)
    gamma = ((Q - 1) * 2.0 ** -24) / (1 - (Q - 1) * 2.0 ** -24)
    err = np.abs(seg_f[:, i, j] - exact[:, i, j])
    bound = gamma * np.abs(exact[:, i, j])
    assert np.count_nonzero(err > bound) > 0
