"""Pins for the oracle's backward pass: central finite differences of the
(pinned) fp64 forward recurrence.

The loss is <dy, y> + <dfin, final_states>.  For every input the oracle's
gradient, contracted with a random direction of that input alone, must equal
(loss(theta + eps v) - loss(theta - eps v)) / (2 eps); the error of the central
difference is O(eps^2) and far below the bound used.  Separate directions per
input make a dropped term, a wrong sign or a transposed operand in any one
gradient fail its own check.
"""
import numpy as np
import pytest

import oracle
from mamba_ssd_chunked_scan_gb300 import synth

INPUTS = ("x", "dt", "A", "B", "C", "D", "initial_states")
GRAD = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "initial_states": "dinit"}


def problem(seed, **kw):
    args = dict(batch=2, seqlen=23, nheads=4, headdim=3, dstate=5, ngroups=2, chunk=16, dtype="f32",
                seed=seed, xbc="unit", dt_dist="softplus_m2", A_dist="exp", init_std=0.5)
    args.update(kw)
    p = synth.make_problem(**args)
    for n in INPUTS:                       # fp64 copies: the perturbations must not round
        if getattr(p, n) is not None:
            setattr(p, n, getattr(p, n).astype(np.float64))
    return p


def loss(p, dy, dfin):
    y, fin = oracle.ssd_recurrence(p, want_final=True)
    return float(np.sum(dy * y) + np.sum(dfin * fin))


@pytest.mark.parametrize("kw", [dict(), dict(ngroups=1), dict(ngroups=4, nheads=4), dict(with_D=False),
                                dict(init_std=0.0, seqlen=40),
                                dict(batch=1, seqlen=23, doc_lengths=[1, 7, 5, 10]),
                                dict(batch=1, seqlen=30, doc_lengths=[12, 1, 17], init_std=0.0)])
def test_gradients_match_central_differences(kw):
    p = problem(61, **kw)
    rng = np.random.default_rng(5)
    dy = rng.standard_normal((p.batch, p.seqlen, p.nheads, p.headdim))
    dfin = rng.standard_normal((p.nstates, p.nheads, p.headdim, p.dstate))
    g = oracle.ssd_backward(p, dy, dfin)
    if p.initial_states is None:
        p.initial_states = np.zeros((p.nstates, p.nheads, p.headdim, p.dstate))
    eps = 1e-6
    for name in INPUTS:
        base = getattr(p, name)
        if base is None:
            assert g[GRAD[name]] is None
            continue
        v = rng.standard_normal(base.shape)
        setattr(p, name, base + eps * v)
        lp = loss(p, dy, dfin)
        setattr(p, name, base - eps * v)
        lm = loss(p, dy, dfin)
        setattr(p, name, base)
        fd = (lp - lm) / (2 * eps)
        an = float(np.sum(g[GRAD[name]] * v))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_documents_are_independent():
    """Packed documents: each document's gradients equal those of the document
    run alone (no adjoint crosses a boundary), bit for bit."""
    lens = [6, 1, 9, 8]
    p = problem(73, batch=1, seqlen=sum(lens), doc_lengths=lens)
    rng = np.random.default_rng(9)
    dy = rng.standard_normal((1, p.seqlen, p.nheads, p.headdim))
    dfin = rng.standard_normal((len(lens), p.nheads, p.headdim, p.dstate))
    g = oracle.ssd_backward(p, dy, dfin)
    cu = p.cu_seqlens
    for d in range(len(lens)):
        a, b = int(cu[d]), int(cu[d + 1])
        q = synth.SSDProblem(1, b - a, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0, "f32",
                             p.x[:, a:b].copy(), p.dt[:, a:b].copy(), p.A, p.B[:, a:b].copy(), p.C[:, a:b].copy(),
                             p.D, p.initial_states[d:d + 1].copy())
        gd = oracle.ssd_backward(q, dy[:, a:b], dfin[d:d + 1])
        for k in ("dx", "ddt", "dB", "dC"):
            assert np.array_equal(gd[k][0], g[k][0, a:b]), (d, k)
        assert np.array_equal(gd["dinit"][0], g["dinit"][d])


def test_zero_cotangents_give_zero_gradients():
    p = problem(67)
    g = oracle.ssd_backward(p, np.zeros((p.batch, p.seqlen, p.nheads, p.headdim)), None)
    for k, a in g.items():
        assert a is None or not np.any(a), k


def test_final_state_gradient_alone_is_the_decayed_chain():
    """With dy = 0 only the final state carries gradient: the initial state's
    gradient is dfin times the product of every decay, exp(A_h sum_t dt_t)."""
    p = problem(71, with_D=False)
    dfin = np.random.default_rng(3).standard_normal((p.batch, p.nheads, p.headdim, p.dstate))
    g = oracle.ssd_backward(p, np.zeros((p.batch, p.seqlen, p.nheads, p.headdim)), dfin)
    for b in range(p.batch):
        for h in range(p.nheads):
            decay = np.exp(p.A[h] * np.sum(p.dt[b, :, h]))
            np.testing.assert_allclose(g["dinit"][b, h], decay * dfin[b, h], rtol=1e-12, atol=1e-300)
