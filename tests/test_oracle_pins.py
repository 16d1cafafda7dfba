"""Pins for the fp64 oracle: each check ties it to something other than itself.

- two exact forms of the operator (sequential recurrence vs the quadratic
  (C B^T) o L matrix form) agree to fp64 round-off;
- the a_k = 1 special case is unnormalised causal linear attention, brute
  forced here with plain loops;
- the scalar (N = P = 1) case has a closed form in products of decays,
  evaluated here without logarithms;
- a hand-worked three-token example (tests/golden/scalar_three_tokens.txt);
- the block decomposition with split composition equals the recurrence for
  every chunk and split length;
- packed documents equal their stand-alone runs bit for bit;
- a sequence split in two and resumed from the first half's final state
  equals the whole run.
"""
import math
import os

import numpy as np
import pytest

import oracle
from mamba_ssd_chunked_scan_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def small(seed, **kw):
    args = dict(batch=2, seqlen=70, nheads=4, headdim=3, dstate=5, ngroups=2, chunk=16,
                dtype="f32", seed=seed, xbc="unit", dt_dist="softplus_m2", A_dist="exp")
    args.update(kw)
    return synth.make_problem(**args)


@pytest.mark.parametrize("kw", [
    dict(),
    dict(with_D=False),
    dict(init_std=0.7),
    dict(ngroups=1),
    dict(ngroups=4, init_std=0.3),
    dict(batch=1, seqlen=90, doc_lengths=[1, 15, 16, 17, 41], init_std=0.5),
    dict(batch=1, seqlen=90, doc_lengths=[90]),
])
def test_recurrence_equals_quadratic(kw):
    p = small(3, **kw)
    y, _ = oracle.ssd_recurrence(p)
    yq = oracle.ssd_quadratic(p)
    assert rel(y, yq) < 1e-12


def test_linear_attention_special_case():
    """A = 0 and dt = 1 make every decay 1: y_i = sum_{j<=i} (C_i . B_j) x_j."""
    p = small(5, ngroups=1, with_D=False)
    p.A[:] = 0.0
    p.dt[:] = 1.0
    y, _ = oracle.ssd_recurrence(p)
    bsz, L, H, P = p.x.shape
    N = p.dstate
    want = np.zeros_like(y)
    for b in range(bsz):
        for h in range(H):
            for i in range(L):
                for j in range(i + 1):
                    s = 0.0
                    for n in range(N):
                        s += float(p.C[b, i, 0, n]) * float(p.B[b, j, 0, n])
                    want[b, i, h, :] += s * p.x[b, j, h, :].astype(np.float64)
    assert rel(y, want) < 1e-12
    assert rel(oracle.ssd_quadratic(p), want) < 1e-12


def test_scalar_closed_form_products():
    """N = P = 1: y_t = C_t [prod_{k<=t} a_k] h0 + C_t sum_{j<=t} [prod_{k=j+1..t} a_k] dt_j B_j x_j + D x_t."""
    p = small(7, batch=1, seqlen=40, nheads=2, headdim=1, dstate=1, ngroups=1, init_std=1.0)
    y, fin = oracle.ssd_recurrence(p)
    for h in range(2):
        a = [math.exp(float(p.dt[0, t, h]) * float(p.A[h])) for t in range(40)]
        h0 = float(p.initial_states[0, h, 0, 0])
        for t in range(40):
            pre = 1.0
            for k in range(t + 1):
                pre *= a[k]
            acc = pre * h0
            for j in range(t + 1):
                w = 1.0
                for k in range(j + 1, t + 1):
                    w *= a[k]
                acc += w * float(p.dt[0, j, h]) * float(p.B[0, j, 0, 0]) * float(p.x[0, j, h, 0])
            want = float(p.C[0, t, 0, 0]) * acc + float(p.D[h]) * float(p.x[0, t, h, 0])
            assert abs(y[0, t, h, 0] - want) <= 1e-12 * max(1.0, abs(want))
            if t == 39:
                assert abs(fin[0, h, 0, 0] - acc) <= 1e-12 * max(1.0, abs(acc))


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=")
                vals[k.strip()] = [float(t) for t in v.split()]
    return vals


def test_hand_worked_three_tokens():
    g = _read_golden("scalar_three_tokens.txt")
    powers = [math.exp(-k) for k in range(5)]
    want_y = [sum(c * e for c, e in zip(g[f"y{t}"], powers)) for t in range(3)]
    want_h = sum(c * e for c, e in zip(g["h_final"], powers))
    p = synth.make_problem(batch=1, seqlen=3, nheads=1, headdim=1, dstate=1, ngroups=1, chunk=2,
                           dtype="f32", seed=0, with_D=True, init_std=1.0)
    p.x[0, :, 0, 0] = g["x"]
    p.dt[0, :, 0] = g["dt"]
    p.A[0] = g["A"][0]
    p.B[0, :, 0, 0] = g["B"]
    p.C[0, :, 0, 0] = g["C"]
    p.D[0] = g["D"][0]
    p.initial_states[0, 0, 0, 0] = g["h0"][0]
    y, fin = oracle.ssd_recurrence(p)
    np.testing.assert_allclose(y[0, :, 0, 0], want_y, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(fin[0, 0, 0, 0], want_h, rtol=1e-14, atol=1e-14)
    for Q, sl in ((1, 0), (2, 0), (2, 2), (3, 0)):
        yc, fc = oracle.ssd_chunked(p, Q, sl)
        np.testing.assert_allclose(yc[0, :, 0, 0], want_y, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(fc[0, 0, 0, 0], want_h, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(oracle.ssd_quadratic(p)[0, :, 0, 0], want_y, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("Q,split", [(1, 0), (2, 0), (16, 0), (16, 16), (16, 48), (64, 0), (64, 64),
                                     (128, 0)])
def test_chunked_equals_recurrence(Q, split):
    p = small(11, batch=2, seqlen=200, init_std=0.4)
    y, fin = oracle.ssd_recurrence(p)
    yc, fc = oracle.ssd_chunked(p, Q, split)
    assert rel(yc, y) < 1e-12
    assert rel(fc, fin) < 1e-12


@pytest.mark.parametrize("Q,split", [(16, 0), (16, 32), (64, 64)])
def test_chunked_equals_recurrence_varlen(Q, split):
    lens = [1, 15, 16, 17, 31, 33, 63, 64, 60]
    p = small(13, batch=1, seqlen=sum(lens), doc_lengths=lens, init_std=0.4)
    y, fin = oracle.ssd_recurrence(p)
    yc, fc = oracle.ssd_chunked(p, Q, split)
    assert rel(yc, y) < 1e-12
    assert rel(fc, fin) < 1e-12


def test_varlen_equals_separate_documents_bitwise():
    lens = [5, 1, 33, 20, 41]
    p = small(17, batch=1, seqlen=sum(lens), doc_lengths=lens, init_std=0.3)
    y, fin = oracle.ssd_recurrence(p)
    cu = p.cu_seqlens
    for d in range(len(lens)):
        a, b = int(cu[d]), int(cu[d + 1])
        q = synth.SSDProblem(1, b - a, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0, "f32",
                             p.x[:, a:b].copy(), p.dt[:, a:b].copy(), p.A, p.B[:, a:b].copy(),
                             p.C[:, a:b].copy(), p.D, p.initial_states[d:d + 1].copy())
        yd, fd = oracle.ssd_recurrence(q)
        assert np.array_equal(yd[0], y[0, a:b])
        assert np.array_equal(fd[0], fin[d])


def test_resume_from_final_state():
    p = small(19, batch=2, seqlen=96, init_std=0.5)
    y, fin = oracle.ssd_recurrence(p)
    half = 40
    def part(a, b, init):
        return synth.SSDProblem(p.batch, b - a, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0,
                                "f32", p.x[:, a:b].copy(), p.dt[:, a:b].copy(), p.A,
                                p.B[:, a:b].copy(), p.C[:, a:b].copy(), p.D, init)
    y1, f1 = oracle.ssd_recurrence(part(0, half, p.initial_states))
    # handing over the fp64 state exactly replays the same operations
    y2, f2 = oracle.ssd_recurrence(part(half, 96, f1))
    assert np.array_equal(np.concatenate([y1, y2], axis=1), y)
    assert np.array_equal(f2, fin)


def test_document_isolation():
    """Changing one packed document changes no other document's output."""
    lens = [30, 1, 50, 19]
    p = small(23, batch=1, seqlen=sum(lens), doc_lengths=lens)
    y, fin = oracle.ssd_recurrence(p)
    cu = p.cu_seqlens
    q = synth.SSDProblem(**{k: (v.copy() if isinstance(v, np.ndarray) else v)
                            for k, v in vars(p).items()})
    a, b = int(cu[2]), int(cu[3])
    q.x[:, a:b] *= -3.0
    q.B[:, a:b] += 1.0
    q.dt[:, a:b] *= 2.0
    y2, fin2 = oracle.ssd_recurrence(q)
    for d in range(len(lens)):
        s, e = int(cu[d]), int(cu[d + 1])
        same = np.array_equal(y2[0, s:e], y[0, s:e]) and np.array_equal(fin2[d], fin[d])
        assert same == (d != 2)
