"""The C ABI without a GPU: the library builds and loads, exports every
symbol include/ssd.h declares, and rejects bad arguments before launching
anything (these calls never touch the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mamba_ssd_chunked_scan_gb300 import build
    build.build()
    from mamba_ssd_chunked_scan_gb300 import _lib
    return _lib


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "ssd.h")).read()
    return re.findall(r"SSD_API\s+[\w\s\*]+?\b(ssd_\w+)\s*\(", src)


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 7
    assert set(names) == set(L.EXPORTS)
    for n in names:
        assert hasattr(L.lib, n), n


def params(L, **kw):
    d = dict(batch=8, seqlen=2048, nheads=80, headdim=64, dstate=128, ngroups=1, chunk=128,
             split_len=0, ndocs=0, dtype=1)
    d.update(kw)
    return L.make_params(**d)


def test_workspace_size_and_plan(L):
    p = params(L)
    # one split: the status header only (with a GPU present, also the leftover-unit plan's
    # piece log-decays and states), always inside the 8 MiB allocation-free scratch
    for q in (p, params(L, batch=2), params(L, batch=4, nheads=48), params(L, batch=16, seqlen=1024, nheads=64,
                                                                           ngroups=8)):
        assert L.workspace_size(q) == 256 or 256 < L.workspace_size(q) < int(4.01 * (1 << 20))
        assert L.workspace_size(q) <= 8 << 20
    fam, launches, ns = L.plan(p)
    assert ns == 1 and launches >= 1
    p = params(L, batch=1, seqlen=65536, nheads=32, split_len=2048)
    fam, launches, ns = L.plan(p)
    assert ns == 32
    assert L.workspace_size(p) >= 256 + 32 * 32 * (4 + 64 * 128 * 4)
    # split_len >= seqlen is one split
    assert L.plan(params(L, batch=1, seqlen=1000, nheads=2, split_len=1024))[2] == 1


@pytest.mark.parametrize("kw,code", [
    (dict(chunk=256), 2), (dict(chunk=0), 1), (dict(chunk=100), 2), (dict(ngroups=3), 1),
    (dict(split_len=100), 1), (dict(batch=0), 1), (dict(dtype=7), 1), (dict(ndocs=3, batch=2), 1),
    (dict(headdim=12), 2),
])
def test_invalid_params(L, kw, code):
    p = params(L, **kw)
    assert L.workspace_size(p) == 0
    rc = L.lib.ssd_fwd(ctypes.byref(p), *([ctypes.c_void_p(0x1000)] * 10), ctypes.c_void_p(0x1000),
                       1 << 20, None)
    assert rc == code


def test_invalid_pointers_rejected_before_launch(L):
    p = params(L, batch=1, seqlen=256, nheads=2)
    ok = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    args = [ok, ok, ok, ok, ok, None, None, None, ctypes.c_void_p(0x30000), None]
    def call(a, wsb=4096, w=ws):
        return L.lib.ssd_fwd(ctypes.byref(p), *a, w, wsb, None)
    bad = list(args); bad[0] = None                       # x missing
    assert call(bad) == 1
    bad = list(args); bad[0] = ctypes.c_void_p(0x10008)   # x not 16-byte aligned
    assert call(bad) == 1
    bad = list(args); bad[8] = ok                         # y aliases x
    assert call(bad) == 1
    bad = list(args); bad[7] = ok                         # cu_seqlens with ndocs == 0
    assert call(bad) == 1
    assert call(args, wsb=100) == 3                       # workspace too small
    assert call(args, w=None) == 3                        # workspace missing
    assert L.lib.ssd_segsum_dump(None, 10, 128, None, None, None, None, None) == 1
    assert L.lib.ssd_segsum_dump(ok, 10, 96, None, None, None, None, None) == 1


def test_status_strings(L):
    assert L.lib.ssd_status_string(0) == b"SSD_OK"
    assert L.lib.ssd_status_string(5) == b"SSD_ERR_TIMEOUT"
    assert L.lib.ssd_status_string(99) == b"SSD_ERR_UNKNOWN"


def wave_fill(units, sms=152):
    return units / (-(-units // sms) * sms)


def test_plan_packed_documents_with_init_states(L):
    # the bf16 Mamba-2 head shape runs packed documents with initial states on the
    # tensor-core kernel; a split plan adds one launch (the documents' initial states
    # in the split aggregates, before their composition)
    p = params(L, batch=1, seqlen=4096, nheads=8, split_len=1024, ndocs=5)
    assert L.plan(p, True, True) == (1, 4, 4)
    assert L.plan(p, False, True) == (1, 3, 4)
    assert L.plan(params(L, batch=1, seqlen=4096, nheads=8, split_len=4096, ndocs=5), True, True) == (1, 1, 1)
    # fp32 stays on the SIMT kernel
    assert L.plan(params(L, batch=1, seqlen=4096, nheads=8, split_len=1024, ndocs=5, dtype=0), True, True)[0] == 0


@pytest.mark.parametrize("batch,seqlen,nheads,want", [
    (1, 32768, 48, 6),     # packed varlen config: 7 splits would run 3 waves, 6 fill 2 to 95 %
    (1, 16384, 64, 7),     # 448 units, 98 % of 3 waves
    (2, 256, 4, 1),        # too short to split (splits keep at least 4 chunks)
    (2, 1000, 3, 2),       # as many 4-chunk splits as the length allows
    (8, 2048, 80, 1),      # at least as many units as SMs: one split
    (2, 2048, 80, 1),      # 160 units: one split (the leftover-unit plan evens the waves)
])
def test_automatic_split_plan(L, batch, seqlen, nheads, want):
    p = params(L, batch=batch, seqlen=seqlen, nheads=nheads, ngroups=1)
    fam, launches, ns = L.plan(p)
    assert ns == want
    nchunks = -(-seqlen // 128)
    if ns > 1:
        # the chosen count is the smallest in its range whose units fill their waves to 95 %,
        # or the best fill when none does; splits keep at least 4 chunks
        assert -(-nchunks // ns) >= 4 or ns == nchunks // 4
        lo = -(-152 // (batch * nheads))
        if wave_fill(batch * nheads * ns) < 0.95:
            hi = min(-(-4 * 152 // (batch * nheads)), nchunks // 4)
            assert all(wave_fill(batch * nheads * k) <= wave_fill(batch * nheads * ns) for k in range(lo, hi + 1))
        else:
            assert all(wave_fill(batch * nheads * k) < 0.95 for k in range(lo, ns))


def step_args(L, **kw):
    """ssd_step arguments with distinct, 256-byte aligned fake device addresses
    (every case below is rejected before anything touches the device)."""
    base = 1 << 40
    d = dict(batch=4, nheads=8, headdim=64, dstate=128, ngroups=2, dtype=1,
             state_in=base, state_out=base, x=base + (1 << 30), dt=base + (2 << 30), A=base + (3 << 30),
             B=base + (4 << 30), C=base + (5 << 30), D=base + (6 << 30), y=base + (7 << 30), stream=None)
    d.update(kw)
    return d


def call_step(L, d):
    vp = ctypes.c_void_p
    return L.lib.ssd_step(d["batch"], d["nheads"], d["headdim"], d["dstate"], d["ngroups"], d["dtype"],
                          *(vp(d[k]) if d[k] is not None else None
                            for k in ("state_in", "state_out", "x", "dt", "A", "B", "C", "D", "y", "stream")))


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), 1), (dict(nheads=0), 1), (dict(ngroups=3), 1), (dict(dtype=5), 1),
    (dict(dstate=6), 2), (dict(dstate=1024), 2), (dict(headdim=4096), 2), (dict(batch=1 << 28, nheads=8), 2),
    (dict(x=None), 1), (dict(state_in=None), 1), (dict(y=None), 1),
    (dict(state_out=(1 << 40) + 8), 1),                    # misaligned state
    (dict(state_out=(1 << 40) + 4096), 1),                 # partial overlap with state_in
    (dict(y=(1 << 40) + (1 << 30)), 1),                    # y == x
    (dict(dt=(1 << 40) + (2 << 30) + 2), 1),               # misaligned dt
])
def test_step_invalid_args(L, kw, code):
    assert call_step(L, step_args(L, **kw)) == code


def test_bwd_workspace_size(L):
    # status header + chunk-entry states + dB, dC shares + dA, dD shares; the bf16
    # Mamba-2 head shape runs the tensor-core backward (128-token chunks, bf16
    # shares), fp32 the CUDA-core one (32-token chunks, fp32 shares)
    shares = 2 * 2 * 1000 * 4 * 128
    n = L.lib.ssd_bwd_workspace_size(ctypes.byref(params(L, batch=2, seqlen=1000, nheads=4)))
    assert n >= 256 + 2 * 4 * 8 * 64 * 128 * 4 + 2 * shares + 2 * 8 * 4
    n = L.lib.ssd_bwd_workspace_size(ctypes.byref(params(L, batch=2, seqlen=1000, nheads=4, dtype=0)))
    assert n >= 256 + 2 * 4 * 32 * 64 * 128 * 4 + 4 * shares + 2 * 8 * 4
    assert L.lib.ssd_bwd_workspace_size(ctypes.byref(params(L, ndocs=3, batch=1))) > 0    # packed documents
    # packed documents with per-document states: (head, document) units, each document in chunks
    # from its first token (one more chunk per document at most), a dA and a dD share per unit; the
    # bf16 Mamba-2 head shape on the tensor cores (128-token chunks, bf16 shares), fp32 on CUDA
    # cores (32-token chunks, fp32 shares)
    pd = params(L, batch=1, seqlen=1000, nheads=4, ndocs=3)
    nd = L.lib.ssd_bwd_workspace_size_doc_states(ctypes.byref(pd))
    assert nd >= 256 + 4 * (8 + 3) * 64 * 128 * 4 + 2 * (1000 * 4 * 128 * 2) + 2 * 4 * 3 * 4
    pf = params(L, batch=1, seqlen=1000, nheads=4, ndocs=3, dtype=0)
    nf = L.lib.ssd_bwd_workspace_size_doc_states(ctypes.byref(pf))
    assert nf >= 256 + 4 * (32 + 3) * 64 * 128 * 4 + 2 * (1000 * 4 * 128 * 4) + 2 * 4 * 3 * 4
    assert nf == L.lib.ssd_bwd_workspace_size(ctypes.byref(pf))   # (CUDA cores: document units either way)
    assert L.lib.ssd_bwd_workspace_size_doc_states(ctypes.byref(params(L, batch=2, seqlen=1000))) == 0   # no documents
    assert L.lib.ssd_bwd_workspace_size(ctypes.byref(params(L, headdim=128, dstate=128))) == 0   # P * N > 8192


@pytest.mark.parametrize("case,code", [("docs_dinit", 3), ("docs_no_cu", 1), ("null_dx", 1), ("alias", 1),
                                       ("misaligned", 1), ("no_ws", 3)])
def test_bwd_invalid_args(L, case, code):
    base = 1 << 40
    ptr = {k: base + (i << 30) for i, k in enumerate(
        ("x", "dt", "A", "B", "C", "D", "dy", "dx", "ddt", "dA", "dB", "dC", "ws"))}
    p = params(L, batch=2, seqlen=256, nheads=4)
    cu, dinit = None, None
    if case == "docs_dinit":     # per-document states need ssd_bwd_workspace_size_doc_states() bytes
        p = params(L, batch=1, seqlen=256, nheads=4, ndocs=2)
        cu, dinit = base + (40 << 30), base + (41 << 30)
    if case == "docs_no_cu":     # ndocs without cu_seqlens
        p = params(L, batch=1, seqlen=256, nheads=4, ndocs=2)
    if case == "null_dx":
        ptr["dx"] = None
    if case == "alias":
        ptr["dB"] = ptr["B"]
    if case == "misaligned":
        ptr["ddt"] += 4
    nbytes = L.lib.ssd_bwd_workspace_size(ctypes.byref(p))
    if case == "no_ws":
        ptr["ws"], nbytes = None, 0
    vp = ctypes.c_void_p
    v = lambda k: None if ptr[k] is None else vp(ptr[k])
    rc = L.lib.ssd_bwd(ctypes.byref(p), v("x"), v("dt"), v("A"), v("B"), v("C"), v("D"), None,
                       None if cu is None else vp(cu), v("dy"), None, v("dx"), v("ddt"), v("dA"), v("dB"),
                       v("dC"), None, None if dinit is None else vp(dinit), v("ws"), nbytes, None)
    assert rc == code


def test_fwd_timed_rejects_missing_outputs(L):
    p = params(L)
    n = ctypes.c_int(0)
    ms = (ctypes.c_float * 4)()
    vp = ctypes.c_void_p
    args = [ctypes.byref(p)] + [vp(1 << 40)] * 10 + [vp(1 << 41), 256, None]
    assert L.lib.ssd_fwd_timed(*args, None, 4, ctypes.byref(n)) == 1
    assert L.lib.ssd_fwd_timed(*args, ms, 0, ctypes.byref(n)) == 1
    assert L.lib.ssd_fwd_timed(*args, ms, 4, None) == 1


@pytest.mark.parametrize("kw,code", [
    (dict(rows=0), 1), (dict(width=50), 1), (dict(dtype=3), 1), (dict(eps=-1.0), 1), (dict(eps=float("nan")), 1),
    (dict(group_size=12, width=48), 2), (dict(group_size=16384, width=16384), 2), (dict(y=None), 1),
    (dict(out=(1 << 40) + 8), 1), (dict(weight=(1 << 40) + (2 << 30) + 4), 1),
])
def test_gate_norm_invalid_args(L, kw, code):
    d = dict(rows=4, width=64, group_size=16, dtype=1, y=1 << 40, z=(1 << 40) + (1 << 30),
             weight=(1 << 40) + (2 << 30), eps=1e-5, out=(1 << 40) + (3 << 30))
    d.update(kw)
    vp = ctypes.c_void_p
    ptr = lambda k: None if d[k] is None else vp(d[k])
    rc = L.lib.ssd_gate_norm(d["rows"], d["width"], d["group_size"], d["dtype"], ptr("y"), ptr("z"), ptr("weight"),
                             d["eps"], ptr("out"), None)
    assert rc == code


def test_fault_inject_argument_checks(L):
    """The fault-injection test aid rejects a wait cap below 4096 rounds and
    problems without device waits (the fp32 SIMT kernel) before any launch."""
    ok = ctypes.c_void_p(0x1000)
    p = params(L)
    assert L.lib.ssd_fwd_fault_inject(ctypes.byref(p), *([ok] * 10), ok, 1 << 20, 100, None) == 1
    p32 = params(L, batch=1, seqlen=256, nheads=2, headdim=16, dstate=16, chunk=64, dtype=0)
    ptrs = [ctypes.c_void_p(0x100000 * (k + 1)) for k in range(10)]   # distinct, aligned, never dereferenced
    ptrs[7] = None                                                     # no cu_seqlens
    assert L.lib.ssd_fwd_fault_inject(ctypes.byref(p32), *ptrs, ok, 1 << 20, 1 << 14, None) == 2


def test_check_status_where_without_workspace(L):
    where = ctypes.c_uint32(7)
    assert L.lib.ssd_check_status_where(None, None, ctypes.byref(where)) == 3 and where.value == 0
