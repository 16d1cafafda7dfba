"""GPU parity of the backward pass (ssd_bwd) against the fp64 oracle.

The oracle differentiates the recurrence token by token, backwards in time,
from stored per-token states; the GPU recomputes chunk-entry states and works
chunk by chunk in matrix form, so the two share nothing but the definition.
Bounds: max |d_gpu - d_oracle| / max |d_oracle| per gradient, 1e-4 for fp32
inputs (fp32 arithmetic, sums over whole chunks and sequences) and 2e-2 for
bf16 inputs (bf16 gradients).
"""
import numpy as np
import pytest
import torch

import oracle
import mamba_ssd_chunked_scan_gb300 as ssd
from mamba_ssd_chunked_scan_gb300 import synth

from gpu_helpers import rel_err, to_device

pytestmark = pytest.mark.gpu

BWD_TOL = {"f32": 1e-4, "bf16": 2e-2}


def cotangents(p, seed, with_dfin=True):
    rng = np.random.default_rng(seed)
    dy = rng.standard_normal((p.batch, p.seqlen, p.nheads, p.headdim)).astype(np.float32)
    if p.dtype == "bf16":
        dy = synth.bf16_to_f32(synth.bf16_bits(dy))
    dfin = rng.standard_normal((p.nstates, p.nheads, p.headdim, p.dstate)).astype(np.float32) if with_dfin else None
    return dy, dfin


def run_bwd(p, dy, dfin, split_len=0):
    d = to_device(p)
    if p.dtype == "bf16":
        dyt = torch.from_numpy(synth.bf16_bits(dy).view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        dyt = torch.from_numpy(dy).cuda()
    dft = None if dfin is None else torch.from_numpy(dfin).cuda()
    g = ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], dyt, d["D"], d["init"], dft, d["cu"],
                    split_len=split_len, check_status=True)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.float().cpu().numpy().astype(np.float64)) for k, v in g.items()}


def check(p, seed=1, with_dfin=True, split_len=0):
    dy, dfin = cotangents(p, seed, with_dfin)
    want = oracle.ssd_backward(p, dy, dfin)
    got = run_bwd(p, dy, dfin, split_len)
    tol = BWD_TOL[p.dtype]
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        if want[k] is None or got[k] is None:
            assert got[k] is None and (want[k] is None or p.cu_seqlens is not None), k
            continue
        assert np.isfinite(got[k]).all(), k
        e = rel_err(got[k], want[k])
        assert e <= tol, f"{k}: {e:.3e} > {tol}"
    return got


@pytest.mark.parametrize("kw", [
    dict(batch=2, seqlen=100, nheads=4, headdim=16, dstate=16, ngroups=2, dtype="f32"),     # Qb 64, ragged
    dict(batch=1, seqlen=200, nheads=2, headdim=64, dstate=128, ngroups=1, dtype="f32"),    # Qb 32
    dict(batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2, dtype="bf16"),
    dict(batch=3, seqlen=37, nheads=6, headdim=32, dstate=64, ngroups=3, dtype="f32"),      # shorter than a chunk
    dict(batch=1, seqlen=130, nheads=2, headdim=8, dstate=256, ngroups=1, dtype="f32"),     # wide state
])
def test_bwd_parity(kw):
    p = synth.make_problem(chunk=128, seed=301, init_std=0.3, **kw)
    check(p)


def test_bwd_without_optional_inputs():
    p = synth.make_problem(batch=2, seqlen=150, nheads=4, headdim=64, dstate=128, ngroups=1, chunk=128,
                           dtype="bf16", seed=303, with_D=False)
    g = check(p, with_dfin=False)
    assert g["dD"] is None


def test_bwd_strong_decay():
    """dt = softplus(N(2, 2)): chunk log-decay sums near -1e3, where many
    decays underflow to zero."""
    p = synth.make_problem(batch=1, seqlen=256, nheads=4, headdim=64, dstate=128, ngroups=1, chunk=128,
                           dtype="f32", seed=305, dt_dist="softplus_n22", init_std=0.2)
    check(p)


def test_bwd_deterministic():
    p = synth.make_problem(batch=2, seqlen=200, nheads=4, headdim=64, dstate=128, ngroups=2, chunk=128,
                           dtype="bf16", seed=307, init_std=0.1)
    dy, dfin = cotangents(p, 3)
    g1, g2 = run_bwd(p, dy, dfin), run_bwd(p, dy, dfin)
    for k in g1:
        assert (g1[k] is None and g2[k] is None) or np.array_equal(g1[k], g2[k]), k


def test_bwd_long_sequence():
    """Many chunks: 2048 tokens of the 2.7B-like head shape."""
    p = synth.make_problem(batch=1, seqlen=2048, nheads=4, headdim=64, dstate=128, ngroups=1, chunk=128,
                           dtype="bf16", seed=309, init_std=0.1)
    check(p)


@pytest.mark.parametrize("lens,kw", [
    ([3, 300, 128, 1, 257, 90, 500], dict(headdim=64, dstate=128, dtype="bf16")),    # tiled instance
    ([32, 1, 31, 64, 33, 2], dict(headdim=64, dstate=128, dtype="f32")),             # ends on chunk edges
    ([10, 1, 50, 39], dict(headdim=16, dstate=32, dtype="f32")),                    # generic instance
])
def test_bwd_packed_documents(lens, kw):
    """Packed documents from zero states: no gradient crosses a boundary."""
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=4, ngroups=2, chunk=128, seed=311,
                           doc_lengths=lens, dt_dist="softplus_n22", **kw)
    check(p, with_dfin=False)


@pytest.mark.parametrize("lens,kw", [
    ([3, 300, 128, 1, 257, 90, 500], dict(headdim=64, dstate=128, dtype="bf16")),    # tensor cores, bf16
    ([700, 129, 1000, 255, 384, 383], dict(headdim=64, dstate=128, dtype="bf16")),   # several chunks each
    ([32, 1, 31, 64, 33, 2], dict(headdim=64, dstate=128, dtype="f32")),             # ends on chunk edges
    ([10, 1, 50, 39], dict(headdim=16, dstate=32, dtype="f32")),                    # generic instance
])
@pytest.mark.parametrize("with_dfin", [True, False])
def test_bwd_packed_documents_with_states(lens, kw, with_dfin):
    """Packed documents, each from its own initial state and with (or without)
    its own final-state gradient, run as (head, document) units whose chunks
    start at the document's first token (bf16 on the tensor cores: a document's
    last chunk runs past its end into padding rows and is written row by row);
    dinit is per document."""
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=4, ngroups=2, chunk=128, seed=315,
                           doc_lengths=lens, A_dist="exp", init_std=0.5, **kw)
    got = check(p, with_dfin=with_dfin)
    assert got["dinit"] is not None and got["dinit"].shape[0] == len(lens)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_packed_documents_final_gradient_only(dtype):
    """Documents from zero states with final-state gradients (no initial
    states given): the same path, dinit not asked for."""
    lens = [70, 1, 200, 33]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=4, headdim=64, dstate=128, ngroups=1, chunk=128,
                           dtype=dtype, seed=317, doc_lengths=lens, A_dist="exp")
    got = check(p)
    assert got["dinit"] is None


@pytest.mark.parametrize("kw", [
    dict(batch=1, seqlen=37, nheads=2, ngroups=1),                          # shorter than a chunk
    dict(batch=2, seqlen=128 * 3 + 5, nheads=6, ngroups=2),                 # ragged, 3 heads per group
    dict(batch=1, seqlen=512, nheads=4, ngroups=4, dt_dist="softplus_n22"),  # strong decay, one head per group
    dict(batch=1, seqlen=256, nheads=32, ngroups=1),                        # 32 heads' shares summed per group
])
def test_bwd_tensor_core_shapes(kw):
    """The tensor-core backward (bf16, P 64, N 128, 128-token chunks) with
    initial and final states."""
    p = synth.make_problem(headdim=64, dstate=128, chunk=128, dtype="bf16", seed=313, init_std=0.3, **kw)
    got = check(p)
    assert got["dinit"] is not None


@pytest.mark.parametrize("split_len", [512, 1024, 0])
@pytest.mark.parametrize("kw", [
    dict(batch=1, seqlen=4096, nheads=4, ngroups=1),                    # one row in splits
    dict(batch=2, seqlen=1000, nheads=2, ngroups=1, init_std=0.3),      # ragged last split, initial states
    dict(batch=1, seqlen=2048, nheads=2, ngroups=2, dt_dist="softplus_n22", init_std=0.3),   # strong decay
])
def test_bwd_sequence_splits(kw, split_len):
    """The tensor-core backward over sequence splits: each split enters from the
    state the forward pass's split scan composes and leaves with the adjoint a
    reverse scan composes from dfin (the reverse aggregates: the same
    contraction with C, dy and prefix decays); the splits run in parallel."""
    p = synth.make_problem(headdim=64, dstate=128, chunk=128, dtype="bf16", seed=319, **kw)
    check(p, split_len=split_len)


@pytest.mark.parametrize("lens", [
    [700, 1, 1200, 300, 1895],     # starts inside splits
    [512, 512, 3072],              # starts on split boundaries (split 512)
])
def test_bwd_sequence_splits_packed_documents(lens):
    """Packed documents (from zero states) over sequence splits: the -inf decay
    of a start also cuts the composed states and adjoints at split boundaries."""
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=4, headdim=64, dstate=128, ngroups=2, chunk=128,
                           dtype="bf16", seed=321, doc_lengths=lens)
    check(p, with_dfin=False, split_len=512)


def test_bwd_splits_agree_with_whole_rows_on_a_long_sequence():
    """A sequence too long for the oracle: the split plan and whole rows
    (split_len = L) give the same gradients within bf16 rounding of the bf16
    outputs and fp32 rounding of the fp32 ones."""
    p = synth.make_problem(batch=1, seqlen=16384, nheads=4, headdim=64, dstate=128, ngroups=1, chunk=128,
                           dtype="bf16", seed=323, A_dist="exp", init_std=0.2)
    dy, dfin = cotangents(p, 5)
    split = run_bwd(p, dy, dfin, split_len=1024)
    whole = run_bwd(p, dy, dfin, split_len=p.seqlen)
    for k, tol in (("dx", 1e-2), ("dB", 1e-2), ("dC", 1e-2), ("ddt", 1e-4), ("dA", 1e-4), ("dD", 1e-4),
                   ("dinit", 1e-4)):
        e = rel_err(split[k], whole[k])
        assert e <= tol, f"{k}: {e:.3e} > {tol}"


def test_bwd_documents_with_states_full_size_sampled():
    """C5's full size (32,768 tokens in 37 packed documents, 48 heads, bf16)
    with every document's initial state and final-state gradient.  Documents
    are independent sequences, so each sampled one (the first, one in the
    middle, the last) is run by the oracle on its own, from its initial state
    and with its final-state gradient, and gives every gradient of its tokens
    and its dinit.  (dA and dD sum over all documents; the smaller cases above
    check them.)"""
    p = synth.config_varlen(init_std=0.2)
    dy, dfin = cotangents(p, 17)
    got = run_bwd(p, dy, dfin)
    cu = p.cu_seqlens
    for d in (0, p.ndocs // 2, p.ndocs - 1):
        t0, t1 = int(cu[d]), int(cu[d + 1])
        q = synth.SSDProblem(1, t1 - t0, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0, p.dtype,
                             p.x[:, t0:t1].copy(), p.dt[:, t0:t1].copy(), p.A, p.B[:, t0:t1].copy(),
                             p.C[:, t0:t1].copy(), p.D, p.initial_states[d:d + 1].copy(), None, f"doc{d}")
        want = oracle.ssd_backward(q, dy[:, t0:t1].copy(), dfin[d:d + 1].copy())
        for k, g in (("dx", got["dx"][:, t0:t1]), ("ddt", got["ddt"][:, t0:t1]), ("dB", got["dB"][:, t0:t1]),
                     ("dC", got["dC"][:, t0:t1]), ("dinit", got["dinit"][d:d + 1])):
            assert np.isfinite(g).all(), (d, k)
            e = rel_err(g, want[k])
            assert e <= BWD_TOL["bf16"], f"document {d} {k}: {e:.3e}"
