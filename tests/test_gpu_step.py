"""GPU parity of the decode step (ssd_step) against the fp64 oracle.

Shapes cover every lane layout of the kernel (dstate 16 to 512: segments of
4 to 32 lanes, one to four vectors per lane), ragged row counts, several
groups, both storage types, D present or absent.  The state is fp32 and all
of the step's arithmetic is fp32, so the state is held to the fp32 tolerance
in both storage types; y is held to its storage type's tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

from gpu_helpers import TOL, rel_err, run, to_device

pytestmark = pytest.mark.gpu


def problem(batch, H, P, N, G, dtype, seed, with_D=True, init_std=0.5):
    return synth.make_problem(batch=batch, seqlen=1, nheads=H, headdim=P, dstate=N, ngroups=G, chunk=128,
                              dtype=dtype, seed=seed, with_D=with_D, init_std=init_std)


def step_on_gpu(p, in_place=True):
    d = to_device(p)
    x, B, C = d["x"][:, 0], d["B"][:, 0], d["C"][:, 0]
    state = d["init"].clone()
    out = None if in_place else torch.full_like(state, float("nan"))
    y = ssd.ssd_step(state, x, d["dt"][:, 0], d["A"], B, C, d["D"], state_out=out)
    torch.cuda.synchronize()
    s = state if in_place else out
    return y.float().cpu().numpy().astype(np.float64), s.cpu().numpy().astype(np.float64), s


def check(p):
    y_o, s_o = oracle.ssd_step(p.initial_states, p.x[:, 0], p.dt[:, 0], p.A, p.B[:, 0], p.C[:, 0], p.D)
    y_g, s_g, _ = step_on_gpu(p)
    assert np.isfinite(y_g).all() and np.isfinite(s_g).all()
    assert rel_err(s_g, s_o) <= TOL["f32"], rel_err(s_g, s_o)
    assert rel_err(y_g, y_o) <= TOL[p.dtype], rel_err(y_g, y_o)


@pytest.mark.parametrize("batch,H,P,N,G,dtype", [
    (3, 4, 64, 128, 2, "bf16"),     # 32-lane rows, one vector per lane
    (2, 3, 16, 16, 1, "f32"),       # 4-lane rows
    (5, 8, 64, 64, 4, "bf16"),      # 16-lane rows
    (2, 2, 24, 48, 2, "f32"),       # 12 vectors on 16 lanes; 24 rows: a ragged last pass
    (1, 2, 32, 256, 1, "f32"),      # two vectors per lane
    (2, 2, 8, 512, 2, "bf16"),      # four vectors per lane
    (3, 2, 100, 32, 1, "bf16"),     # 8-lane rows, 100 rows
    (1, 1, 1, 4, 1, "f32"),         # one row of one vector
])
def test_step_parity(batch, H, P, N, G, dtype):
    check(problem(batch, H, P, N, G, dtype, seed=200 + N + P))


def test_step_without_D():
    check(problem(2, 4, 64, 128, 1, "bf16", seed=211, with_D=False))


def test_step_in_place_equals_out_of_place():
    p = problem(4, 6, 64, 128, 2, "bf16", seed=213)
    y1, s1, _ = step_on_gpu(p, in_place=True)
    y2, s2, _ = step_on_gpu(p, in_place=False)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


def test_step_zero_dt_keeps_state_bitwise():
    p = problem(3, 4, 64, 128, 2, "bf16", seed=217)
    p.dt[:] = 0.0
    _, s_g, _ = step_on_gpu(p)
    assert np.array_equal(s_g, p.initial_states.astype(np.float64))


def test_prefill_then_decode_continues_the_sequence():
    """ssd_fwd over the first L tokens (final states), then one ssd_step per
    further token, equals the oracle recurrence over all L + K tokens."""
    L, K = 300, 5
    p = synth.make_problem(batch=2, seqlen=L + K, nheads=8, headdim=64, dstate=128, ngroups=2, chunk=128,
                           dtype="bf16", seed=219, init_std=0.1)
    y_o, f_o = oracle.ssd_recurrence(p)
    d = to_device(p)
    f = ssd.SSDForward(p.batch, L, p.nheads, p.headdim, p.dstate, p.ngroups, 128, 0, 0, torch.bfloat16)
    state = torch.empty((p.batch, p.nheads, p.headdim, p.dstate), dtype=torch.float32, device="cuda")
    y_pre = f(d["x"][:, :L].contiguous(), d["dt"][:, :L].contiguous(), d["A"], d["B"][:, :L].contiguous(),
              d["C"][:, :L].contiguous(), d["D"], d["init"], None, final_states=state)
    assert f.check_status() == 0
    ys = []
    for t in range(L, L + K):
        ys.append(ssd.ssd_step(state, d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"],
                               d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), d["D"]))
    torch.cuda.synchronize()
    y_dec = torch.stack(ys, dim=1).float().cpu().numpy()
    assert rel_err(y_pre.float().cpu().numpy(), y_o[:, :L]) <= TOL["bf16"]
    assert rel_err(y_dec, y_o[:, L:]) <= TOL["bf16"]
    assert rel_err(state.cpu().numpy(), f_o) <= TOL["bf16"]


def test_step_full_size_sampled():
    """The benchmark's decode workload (batch 256, 80 heads, P 64, N 128): the
    whole batch in one launch, outputs of sampled (row, head) pairs against
    the oracle."""
    p = synth.config_decode()
    y_g, s_g, _ = step_on_gpu(p)
    rng = np.random.default_rng(7)
    rows = rng.choice(p.batch, size=6, replace=False)
    for b in rows:
        y_o, s_o = oracle.ssd_step(p.initial_states[b:b + 1], p.x[b:b + 1, 0], p.dt[b:b + 1, 0], p.A,
                                   p.B[b:b + 1, 0], p.C[b:b + 1, 0], p.D)
        assert rel_err(s_g[b:b + 1], s_o) <= TOL["f32"]
        assert rel_err(y_g[b:b + 1], y_o) <= TOL["bf16"]
