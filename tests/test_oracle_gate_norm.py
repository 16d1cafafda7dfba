"""Pins for the oracle's gated RMS normalisation.

- equals torch's own silu and rms_norm (a library routine), in fp64;
- a group whose gated values are all equal to c maps to c / sqrt(c^2 + eps) * w;
- with eps = 0 the result does not change when y is scaled by a positive factor;
- z = 0 closes the gate (silu(0) = 0) and the output is exactly zero.
"""
import numpy as np
import pytest
import torch

import oracle


def inputs(rows=5, width=48, seed=1):
    r = np.random.default_rng(seed)
    return r.standard_normal((rows, width)), r.standard_normal((rows, width)) * 2, r.uniform(0.5, 1.5, width)


@pytest.mark.parametrize("group", [48, 16, 8])
def test_matches_torch_silu_and_rms_norm(group):
    y, z, w = inputs()
    eps = 1e-5
    got = oracle.gate_norm(y, z, w, group, eps)
    g = torch.from_numpy(y) * torch.nn.functional.silu(torch.from_numpy(z))
    gg = g.reshape(y.shape[0], -1, group)
    ref = torch.nn.functional.rms_norm(gg, (group,), eps=eps).reshape(y.shape) * torch.from_numpy(w)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_constant_group_closed_form():
    rows, width, group, eps = 3, 16, 8, 1e-3
    c = np.array([0.5, -2.0, 3.0])
    z = np.full((rows, width), 1.5)
    y = (c / (1.5 / (1 + np.exp(-1.5))))[:, None] * np.ones((rows, width))   # g = c everywhere
    w = np.linspace(0.5, 2.0, width)
    got = oracle.gate_norm(y, z, w, group, eps)
    want = (c / np.sqrt(c * c + eps))[:, None] * w
    np.testing.assert_allclose(got, want, rtol=1e-12)


def test_scale_invariance_without_eps():
    y, z, w = inputs(seed=3)
    np.testing.assert_allclose(oracle.gate_norm(7.5 * y, z, w, 16, 0.0), oracle.gate_norm(y, z, w, 16, 0.0),
                               rtol=1e-12)


def test_closed_gate_gives_zero():
    y, z, w = inputs(seed=4)
    assert not np.any(oracle.gate_norm(y, np.zeros_like(z), w, 16, 1e-5))
