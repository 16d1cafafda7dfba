"""Pins for the oracle's decode step (one token from a resident state).

- stepping token by token through a sequence equals the recurrence over the
  whole sequence, bit for bit (the step is the recurrence taken once);
- dt = 0 leaves the state unchanged and reduces y to a matrix-vector product
  (numpy matmul) plus the skip term;
- A = 0 from a zero state gives the rank-one state dt x B^T (numpy outer
  product) and y = dt (B . C) x + D x;
- x = 0 only decays the state: state' = exp(dt A) state, checked per head
  against math.exp.
"""
import math

import numpy as np

import oracle
from mamba_ssd_chunked_scan_gb300 import synth


def inputs(seed, batch=3, H=4, P=5, N=6, G=2, init_std=0.6):
    p = synth.make_problem(batch=batch, seqlen=1, nheads=H, headdim=P, dstate=N, ngroups=G, chunk=16,
                           dtype="f32", seed=seed, xbc="unit", dt_dist="softplus_m2", A_dist="exp",
                           init_std=init_std)
    return (p.initial_states.astype(np.float64), p.x[:, 0].astype(np.float64), p.dt[:, 0].astype(np.float64),
            p.A.astype(np.float64), p.B[:, 0].astype(np.float64), p.C[:, 0].astype(np.float64),
            p.D.astype(np.float64))


def test_steps_equal_recurrence_bitwise():
    p = synth.make_problem(batch=2, seqlen=37, nheads=4, headdim=3, dstate=5, ngroups=2, chunk=16,
                           dtype="f32", seed=41, xbc="unit", dt_dist="softplus_m2", A_dist="exp", init_std=0.5)
    y, fin = oracle.ssd_recurrence(p)
    S = p.initial_states.astype(np.float64)
    for t in range(p.seqlen):
        yt, S = oracle.ssd_step(S, p.x[:, t], p.dt[:, t], p.A, p.B[:, t], p.C[:, t], p.D)
        assert np.array_equal(yt, y[:, t])
    assert np.array_equal(S, fin)


def test_zero_dt_keeps_state():
    S, x, dt, A, B, C, D = inputs(43)
    dt[:] = 0.0
    y, S1 = oracle.ssd_step(S, x, dt, A, B, C, D)
    assert np.array_equal(S1, S)
    H = S.shape[1]
    G = B.shape[1]
    for b in range(S.shape[0]):
        for h in range(H):
            g = h // (H // G)
            want = S[b, h] @ C[b, g] + D[h] * x[b, h]
            np.testing.assert_allclose(y[b, h], want, rtol=1e-13, atol=1e-13)


def test_zero_decay_rate_from_zero_state():
    S, x, dt, A, B, C, D = inputs(47)
    S[:] = 0.0
    A[:] = 0.0
    y, S1 = oracle.ssd_step(S, x, dt, A, B, C, D)
    H, G = S.shape[1], B.shape[1]
    for b in range(S.shape[0]):
        for h in range(H):
            g = h // (H // G)
            np.testing.assert_allclose(S1[b, h], dt[b, h] * np.outer(x[b, h], B[b, g]), rtol=1e-14, atol=1e-15)
            want = dt[b, h] * float(np.dot(B[b, g], C[b, g])) * x[b, h] + D[h] * x[b, h]
            np.testing.assert_allclose(y[b, h], want, rtol=1e-12, atol=1e-14)


def test_zero_input_only_decays():
    S, x, dt, A, B, C, D = inputs(53, init_std=1.0)
    x[:] = 0.0
    y, S1 = oracle.ssd_step(S, x, dt, A, B, C, None)
    for b in range(S.shape[0]):
        for h in range(S.shape[1]):
            a = math.exp(dt[b, h] * A[h])
            np.testing.assert_allclose(S1[b, h], a * S[b, h], rtol=1e-15, atol=0)
