"""GPU parity: ssd_fwd through the C ABI against the fp64 oracle.

Bound (per tensor): max |y_gpu - y_oracle| / max |y_oracle| <= 1e-5 for fp32
inputs and <= 2e-2 for bf16 inputs with fp32 accumulation; final states are
held to the same bounds.
"""
import numpy as np
import pytest

import oracle
from mamba_ssd_chunked_scan_gb300 import synth

from gpu_helpers import TOL, rel_err, run

pytestmark = pytest.mark.gpu


def check(p, split_len=None, chunk=None, want_final=True):
    y_o, f_o = oracle.ssd_recurrence(p, want_final=want_final)
    y_g, f_g, _ = run(p, want_final=want_final, split_len=split_len, chunk=chunk)
    tol = TOL[p.dtype]
    ey = rel_err(y_g, y_o)
    assert np.isfinite(y_g).all()
    assert ey <= tol, f"{p.name}: y err {ey:.3e} > {tol}"
    if want_final:
        assert np.isfinite(f_g).all()
        ef = rel_err(f_g, f_o)
        assert ef <= tol, f"{p.name}: final state err {ef:.3e} > {tol}"
    return ey


def test_tiny_fp32_config():
    p = synth.config_tiny_f32()
    check(p)


@pytest.mark.parametrize("chunk", [64, 128])
@pytest.mark.parametrize("split", [0, 128, 256])
def test_fp32_small_with_tail(chunk, split):
    if split % chunk:
        pytest.skip("split_len must be a multiple of chunk")
    p = synth.make_problem(batch=2, seqlen=3 * 128 + 37, nheads=3, headdim=16, dstate=32, ngroups=1,
                           chunk=chunk, dtype="f32", seed=31, xbc="unit", dt_dist="softplus_m2",
                           A_dist="exp", init_std=0.5)
    check(p, split_len=split)


@pytest.mark.parametrize("kw", [
    dict(batch=2, seqlen=5 * 128 + 37, nheads=4, ngroups=2),
    dict(batch=1, seqlen=3 * 128, nheads=2, ngroups=1, init_std=0.1),
    dict(batch=3, seqlen=100, nheads=2, ngroups=2, with_D=False),
    dict(batch=1, seqlen=1, nheads=2, ngroups=1, init_std=0.1),
])
def test_bf16_mamba2_shapes(kw):
    p = synth.make_problem(headdim=64, dstate=128, chunk=128, dtype="bf16", seed=41, **kw)
    check(p)


@pytest.mark.parametrize("split", [128, 512, 1024])
def test_bf16_splits(split):
    p = synth.make_problem(batch=1, seqlen=1500, nheads=3, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=43, init_std=0.1)
    check(p, split_len=split)


@pytest.mark.parametrize("nheads", [3, 4])
@pytest.mark.parametrize("split", [512, 1024])
def test_bf16_split_aggregates_with_states(nheads, split):
    # splits of 4 or more chunks take the tensor-core aggregate kernel: one or two
    # heads per CTA (odd / even heads per group), two batch rows, initial states,
    # a ragged last split
    p = synth.make_problem(batch=2, seqlen=4 * 512 + 300, nheads=nheads, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=44, init_std=0.1)
    check(p, split_len=split)


@pytest.mark.parametrize("nheads", [3, 4])
def test_bf16_split_aggregates_packed_documents(nheads):
    # documents that start on a split start, on a chunk start and inside chunks, of
    # length 1 up to a whole split, with splits of 4 chunks
    lens = [1, 511, 512, 3, 509, 130, 1024, 77, 300]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=nheads, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=46, dt_dist="softplus_n22", doc_lengths=lens)
    check(p, split_len=512)


@pytest.mark.parametrize("split", [0, 256])
@pytest.mark.parametrize("init", [0.0, 0.2])
def test_bf16_varlen_edges(split, init):
    # documents of length 1, a chunk-1, chunk, chunk+1, one ending on a split boundary
    lens = [1, 127, 128, 129, 127, 1, 256, 75]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=2, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=47, dt_dist="softplus_n22",
                           doc_lengths=lens, init_std=init)
    check(p, split_len=split)


@pytest.mark.parametrize("decay", ["slow", "fast"])
@pytest.mark.parametrize("nheads", [3, 4])
@pytest.mark.parametrize("split", [0, 256, 512])
def test_bf16_packed_documents_with_init_states(nheads, split, decay):
    # every document brings its own initial state, on the tensor-core kernel: several
    # documents start inside one chunk (lengths 1 to 5), others on a chunk start, on a
    # split start (splits of 2 chunks take the full kernel's aggregate mode, of 4 chunks
    # the split-aggregate kernel), or run over several splits.  "slow": per-token decay
    # near 0.98, so the initial states' decayed terms carry most of y over tens of
    # tokens and reach the final states; "fast": the packed-varlen stress decays
    lens = [5, 1, 2, 40, 3, 77, 128, 300, 17, 129, 256, 1, 600, 4, 130]
    dist = dict(dt_dist="loguniform", A_dist="exp") if decay == "slow" else dict(dt_dist="softplus_n22")
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=nheads, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=48, doc_lengths=lens, init_std=1.0, **dist)
    check(p, split_len=split)
    import mamba_ssd_chunked_scan_gb300 as ssd
    f = ssd.SSDForward(1, p.seqlen, nheads, 64, 128, 1, 128, split, p.ndocs)
    fam, launches, ns = f.plan(True, True)
    assert fam == 1 and launches == (4 if ns > 1 else 1)


def test_varlen_init_no_leakage():
    """Changing the initial states of the other documents leaves a target
    document's y and final state bit-identical."""
    lens = [70, 200, 77, 300]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=2, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=62, doc_lengths=lens, init_std=0.5, A_dist="exp")
    y1, f1, _ = run(p, split_len=128)
    q = synth.SSDProblem(**{k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in vars(p).items()})
    q.initial_states[[0, 2, 3]] *= -3.0
    y2, f2, _ = run(q, split_len=128)
    a, b, c = int(p.cu_seqlens[1]), int(p.cu_seqlens[2]), int(p.cu_seqlens[3])
    assert np.array_equal(y1[:, a:b], y2[:, a:b])
    assert np.array_equal(f1[1], f2[1])
    # the changed initial states do reach their own documents
    assert not np.array_equal(y1[:, :a], y2[:, :a])
    assert not np.array_equal(y1[:, c], y2[:, c])
    assert not np.array_equal(f1[3], f2[3])


def test_fp32_varlen_with_init():
    lens = [3, 60, 64, 65, 1, 40]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=2, headdim=16, dstate=16, ngroups=1,
                           chunk=64, dtype="f32", seed=53, xbc="unit", dt_dist="softplus_m2",
                           A_dist="exp", doc_lengths=lens, init_std=0.5)
    check(p, split_len=64)


def test_varlen_no_leakage():
    """Perturbing other documents leaves a target document's y and final state
    bit-identical."""
    lens = [200, 77, 300]
    p = synth.make_problem(batch=1, seqlen=sum(lens), nheads=2, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=59, doc_lengths=lens)
    y1, f1, _ = run(p, split_len=128)
    q = synth.SSDProblem(**{k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in vars(p).items()})
    a, b = int(p.cu_seqlens[1]), int(p.cu_seqlens[2])
    for name in ("x", "B", "C"):
        arr = getattr(q, name)
        arr[:, :a] = synth.bf16_to_f32(synth.bf16_bits(arr[:, :a] * -2.0))
        arr[:, b:] = synth.bf16_to_f32(synth.bf16_bits(arr[:, b:] + 0.5))
    q.dt[:, :a] *= 3.0
    y2, f2, _ = run(q, split_len=128)
    assert np.array_equal(y1[:, a:b], y2[:, a:b])
    assert np.array_equal(f1[1], f2[1])
    assert not np.array_equal(y1[:, :a], y2[:, :a])


def test_resume_continuation():
    """final_states of the first half, fed as initial_states of the second,
    reproduce the whole run (within the bf16 bound)."""
    p = synth.make_problem(batch=2, seqlen=512, nheads=2, headdim=64, dstate=128, ngroups=1,
                           chunk=128, dtype="bf16", seed=61, init_std=0.1)
    y_o, f_o = oracle.ssd_recurrence(p)
    def part(a, b, init):
        return synth.SSDProblem(p.batch, b - a, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0,
                                "bf16", p.x[:, a:b].copy(), p.dt[:, a:b].copy(), p.A, p.B[:, a:b].copy(),
                                p.C[:, a:b].copy(), p.D, init)
    y1, f1, _ = run(part(0, 256, p.initial_states))
    y2, f2, _ = run(part(256, 512, f1.astype(np.float32)))
    assert rel_err(np.concatenate([y1, y2], axis=1), y_o) <= TOL["bf16"]
    assert rel_err(f2, f_o) <= TOL["bf16"]


def test_deterministic():
    p = synth.make_problem(batch=1, seqlen=700, nheads=4, headdim=64, dstate=128, ngroups=2, chunk=128,
                           dtype="bf16", seed=67)
    y1, f1, _ = run(p, split_len=256)
    y2, f2, _ = run(p, split_len=256)
    assert np.array_equal(y1, y2) and np.array_equal(f1, f2)


def test_mamba2_shape_uses_tensor_core_kernel():
    import mamba_ssd_chunked_scan_gb300 as ssd
    f = ssd.SSDForward(2, 256, 4, 64, 128, 2, 128, 0, 0)
    fam, launches, ns = f.plan()
    assert fam == 1 and launches == 1 and ns == 1
    f32 = ssd.SSDForward(2, 256, 4, 16, 16, 2, 64, 0, 0, dtype=__import__("torch").float32)
    assert f32.plan()[0] == 0
