"""Randomised agreement of the oracle's three forms (hypothesis, CPU only).

For random small shapes, chunk sizes, split lengths, group counts and packed
document layouts, the sequential recurrence, the quadratic (C B^T) o L form and
the block decomposition with split composition agree to fp64 round-off.  The
three are independent implementations of one operator, so a slip in any one of
them (an index, a sign, a missing decay term) shows up as a disagreement.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from mamba_ssd_chunked_scan_gb300 import synth  # noqa: E402


@st.composite
def problems(draw):
    G = draw(st.sampled_from([1, 2]))
    H = G * draw(st.integers(1, 2))
    L = draw(st.integers(1, 40))
    docs = draw(st.booleans())
    lens = None
    batch = draw(st.integers(1, 2))
    if docs:
        batch = 1
        cuts = sorted(draw(st.lists(st.integers(1, max(1, L - 1)), max_size=4, unique=True))) if L > 1 else []
        edges = [0] + cuts + [L]
        lens = [b - a for a, b in zip(edges, edges[1:])]
    p = synth.make_problem(batch=batch, seqlen=L, nheads=H, headdim=draw(st.integers(1, 3)),
                           dstate=draw(st.integers(1, 4)), ngroups=G, chunk=4, dtype="f32",
                           seed=draw(st.integers(0, 10_000)), xbc="unit", dt_dist="softplus_m2", A_dist="exp",
                           with_D=draw(st.booleans()), init_std=draw(st.sampled_from([0.0, 0.5])),
                           doc_lengths=lens)
    chunk = draw(st.sampled_from([1, 2, 3, 8, 16]))
    split = draw(st.sampled_from([0, chunk, 2 * chunk, 5 * chunk]))
    return p, chunk, split


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


@settings(max_examples=60, deadline=None)
@given(problems())
def test_three_forms_agree(case):
    p, chunk, split = case
    y, fin = oracle.ssd_recurrence(p)
    assert rel(oracle.ssd_quadratic(p), y) < 1e-11
    yc, fc = oracle.ssd_chunked(p, chunk, split)
    assert rel(yc, y) < 1e-11
    assert rel(fc, fin) < 1e-11
