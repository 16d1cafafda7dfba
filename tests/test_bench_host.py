"""Host-side accounting of bench.py, checked by hand on CPU."""
from types import SimpleNamespace

import pytest

import bench


def layer(batch=8, seqlen=2048, nheads=80):
    """Shape of the 2.7B-like layer (the accounting reads only the sizes)."""
    return SimpleNamespace(batch=batch, seqlen=seqlen, nheads=nheads, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", initial_states=None, nstates=batch)


def test_compulsory_bytes_of_the_27b_layer():
    # per token: x + y (80 heads x 64 x 2 B each), dt (80 x 4 B), B + C (128 x 2 B each)
    assert bench.compulsory_bytes(layer()) == 16384 * (2 * 80 * 64 * 2 + 80 * 4 + 2 * 128 * 2) == 349175808


def test_compulsory_bytes_with_states():
    # initial states read and final states written: 2 x (nstates, H, P, N) fp32
    p = layer()
    p.initial_states = object()
    assert bench.compulsory_bytes(p) == 349175808 + 2 * 8 * 80 * 64 * 128 * 4


def test_decode_bytes():
    p = layer(batch=8, seqlen=1)
    per_head = 2 * 64 * 128 * 4 + 2 * 64 * 2 + 4
    assert bench.decode_bytes(p) == 8 * 80 * per_head + 8 * 1 * 2 * 128 * 2


def test_bwd_flops_per_token_head():
    mac = 2 * 64 * 128 + 32 * (128 + 64) / 2 + 64 * (2 * 128 + 16) + 128 * (2 * 64 + 32)
    assert bench.bwd_flops(layer(batch=1, seqlen=1, nheads=1)) == pytest.approx(2 * mac) == pytest.approx(114688.0)


@pytest.mark.parametrize("batch,want", [
    (8, 32 * 3),   # 640 units on 152 SMs leave 32, each cut into 4 pieces: 3 continue a sequence
    (2, 8 * 7),    # 160 units leave 8, cut into 8 pieces (64 x 32 KiB fits in 4 MiB): 7 continue
    (1, 0),        # 80 units are fewer than the SMs: no plan
])
def test_tail_pieces_of_the_leftover_unit_plan(batch, want):
    assert bench.tail_pieces(layer(batch=batch), 152) == want


def test_job_rate_counts_every_rank():
    assert bench.job_rate(16384, 4, 2.0) == pytest.approx(4 * 16384 / 2e-3)
