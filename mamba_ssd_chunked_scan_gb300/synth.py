"""Seeded synthetic inputs for the SSD forward pass.

This module only draws random tensors with the shapes and distributions of the
Mamba-2 SSD workloads; it holds none of the method's arithmetic. Both the CUDA
path and the fp64 oracle consume exactly the bytes produced here: bf16
workloads are rounded to bf16 (round-to-nearest-even) once, here, and the
oracle reads the same rounded values widened exactly to fp64.

Layouts follow the multi-head SSM layout (Batch, Sequence, Heads, Head_dim) of
"State Space Duality and Mamba-2", section "Multi-Head SSM Patterns":

    x, y            (batch, L, H, P)
    dt              (batch, L, H)       fp32, already softplus-ed (>= 0)
    A, D            (H,)                fp32, A < 0
    B, C            (batch, L, G, N)
    initial_states  (batch or ndocs, H, P, N) fp32
    cu_seqlens      (ndocs + 1,) int32  (packed batch of one row)

Every tensor has its own random stream, derived from (seed, tensor id), so a
change to one distribution never shifts another tensor's values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# tensor ids of the per-tensor random streams
_TID = {"x": 1, "dt": 2, "A": 3, "B": 4, "C": 5, "D": 6, "init": 7, "docs": 8}


def _rng(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), _TID[name]]))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the exactly equal fp32 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _softplus(v: np.ndarray) -> np.ndarray:
    # numerically safe log(1 + e^v); input-distribution shaping only
    return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


@dataclasses.dataclass
class SSDProblem:
    """One synthetic SSD forward problem (host arrays)."""

    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    split_len: int
    dtype: str                      # "f32" or "bf16": storage type of x, B, C, y
    x: np.ndarray                   # fp32 values (already bf16-exact for bf16)
    dt: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: Optional[np.ndarray] = None
    initial_states: Optional[np.ndarray] = None
    cu_seqlens: Optional[np.ndarray] = None
    name: str = ""

    @property
    def ndocs(self) -> int:
        return 0 if self.cu_seqlens is None else len(self.cu_seqlens) - 1

    @property
    def nstates(self) -> int:
        """Leading extent of initial_states / final_states."""
        return self.ndocs if self.cu_seqlens is not None else self.batch

    def storage(self, name: str) -> np.ndarray:
        """The array as it is handed to the library: bf16 bits or fp32."""
        a = getattr(self, name)
        if name in ("x", "B", "C") and self.dtype == "bf16":
            return bf16_bits(a)
        return a

    def tokens(self) -> int:
        return self.batch * self.seqlen


def _finish(p: SSDProblem) -> SSDProblem:
    if p.dtype == "bf16":
        for n in ("x", "B", "C"):
            setattr(p, n, bf16_to_f32(bf16_bits(getattr(p, n))))
    for n in ("x", "dt", "A", "B", "C", "D", "initial_states"):
        a = getattr(p, n)
        if a is not None:
            setattr(p, n, np.ascontiguousarray(a, dtype=np.float32))
    if p.cu_seqlens is not None:
        p.cu_seqlens = np.ascontiguousarray(p.cu_seqlens, dtype=np.int32)
    return p


def geometric_doc_lengths(seed: int, total: int, ndocs: int, mean: float) -> np.ndarray:
    """Document lengths for a packed row: ndocs-1 lengths ~ Geometric(1/mean)
    on {1, 2, ...}, redrawn as a set until their sum leaves at least one token,
    and a last document that takes the remainder."""
    g = _rng(seed, "docs")
    while True:
        lens = g.geometric(1.0 / mean, size=ndocs - 1).astype(np.int64)
        if lens.sum() <= total - 1:
            break
    return np.concatenate([lens, [total - lens.sum()]]).astype(np.int64)


def cu_from_lengths(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int32)


def make_problem(*, batch: int, seqlen: int, nheads: int, headdim: int, dstate: int,
                 ngroups: int = 1, chunk: int = 128, split_len: int = 0, dtype: str = "bf16",
                 seed: int = 0, xbc: str = "scaled", dt_dist: str = "loguniform",
                 A_dist: str = "uniform", with_D: bool = True, init_std: float = 0.0,
                 doc_lengths=None, name: str = "") -> SSDProblem:
    """Draw one problem.

    xbc:     "unit"    x, B, C ~ N(0, 1)
             "scaled"  x, B, C ~ N(0, 1) / sqrt(dstate)
    dt_dist: "softplus_m2"   dt = softplus(N(0,1) - 2)
             "loguniform"    dt = exp(U(ln 1e-3, ln 1e-1))  (softplus of the
                             inverse-softplus init is the identity)
             "softplus_n22"  dt = softplus(N(2, 2))
    A_dist:  "exp"      A = -exp(U(0, 1.5))
             "uniform"  A = -U(1, 16)
    """
    T = batch * seqlen
    H, P, N, G = nheads, headdim, dstate, ngroups
    scale = 1.0 if xbc == "unit" else 1.0 / math.sqrt(N)
    x = _rng(seed, "x").standard_normal((batch, seqlen, H, P), dtype=np.float32) * scale
    B = _rng(seed, "B").standard_normal((batch, seqlen, G, N), dtype=np.float32) * scale
    C = _rng(seed, "C").standard_normal((batch, seqlen, G, N), dtype=np.float32) * scale
    gd = _rng(seed, "dt")
    if dt_dist == "softplus_m2":
        dt = _softplus(gd.standard_normal((batch, seqlen, H)) - 2.0)
    elif dt_dist == "loguniform":
        dt = np.exp(gd.uniform(math.log(1e-3), math.log(1e-1), size=(batch, seqlen, H)))
    elif dt_dist == "softplus_n22":
        dt = _softplus(gd.normal(2.0, 2.0, size=(batch, seqlen, H)))
    else:
        raise ValueError(dt_dist)
    ga = _rng(seed, "A")
    if A_dist == "exp":
        A = -np.exp(ga.uniform(0.0, 1.5, size=H))
    elif A_dist == "uniform":
        A = -ga.uniform(1.0, 16.0, size=H)
    else:
        raise ValueError(A_dist)
    D = _rng(seed, "D").standard_normal(H).astype(np.float32) if with_D else None
    cu = None
    nst = batch
    if doc_lengths is not None:
        assert batch == 1 and int(np.sum(doc_lengths)) == seqlen
        cu = cu_from_lengths(doc_lengths)
        nst = len(doc_lengths)
    init = None
    if init_std > 0:
        init = _rng(seed, "init").standard_normal((nst, H, P, N), dtype=np.float32) * init_std
    del T
    return _finish(SSDProblem(batch, seqlen, H, P, N, G, chunk, split_len, dtype, x, dt, A, B, C,
                              D, init, cu, name))


# The five workloads (sizes, distributions and seeds of the Mamba-2 SSD
# configurations).  Config k (1-based) uses seed k-1.
def config_tiny_f32() -> SSDProblem:
    return make_problem(batch=1, seqlen=256, nheads=2, headdim=16, dstate=16, ngroups=1, chunk=64,
                        dtype="f32", seed=0, xbc="unit", dt_dist="softplus_m2", A_dist="exp",
                        with_D=False, name="tiny_f32_b1_L256_H2_P16_N16_Q64")


def config_27b(batch: int = 8, seqlen: int = 2048) -> SSDProblem:
    return make_problem(batch=batch, seqlen=seqlen, nheads=80, headdim=64, dstate=128, ngroups=1,
                        chunk=128, dtype="bf16", seed=1,
                        name=f"mamba2_2.7b_layer_b{batch}_L{seqlen}_H80_P64_N128_G1_Q128")


SWEEP_POINTS = ((16, 1024), (8, 2048), (4, 4096), (2, 8192), (1, 16384))
SWEEP_SPLITS = (1, 4, 16)   # split_len in units of chunk


def config_sweep(batch: int, seqlen: int, split_chunks: int = 1) -> SSDProblem:
    return make_problem(batch=batch, seqlen=seqlen, nheads=64, headdim=64, dstate=128, ngroups=8,
                        chunk=128, split_len=128 * split_chunks, dtype="bf16", seed=2,
                        name=f"sweep_b{batch}_L{seqlen}_H64_G8_split{128 * split_chunks}")


def config_long(seqlen: int = 65536, split_len: int = 2048) -> SSDProblem:
    return make_problem(batch=1, seqlen=seqlen, nheads=32, headdim=64, dstate=128, ngroups=1,
                        chunk=128, split_len=split_len, dtype="bf16", seed=3, init_std=0.1,
                        name=f"long_b1_L{seqlen}_H32_split{split_len}")


def config_varlen(total: int = 32768, ndocs: int = 37, nheads: int = 48, init_std: float = 0.0) -> SSDProblem:
    """Packed documents; with init_std > 0 every document also has its own
    initial state (and the bench then asks for every final state)."""
    lens = geometric_doc_lengths(4, total, ndocs, 900.0)
    return make_problem(batch=1, seqlen=total, nheads=nheads, headdim=64, dstate=128, ngroups=1,
                        chunk=128, dtype="bf16", seed=4, dt_dist="softplus_n22", doc_lengths=lens,
                        init_std=init_std,
                        name=f"varlen_T{total}_docs{ndocs}_H{nheads}" + ("_states" if init_std > 0 else ""))


def stress_logdecay_rows(nrows: int, length: int, seed: int = 100) -> np.ndarray:
    """Rows of per-token log-decays for the segsum stability check: half the
    tokens strongly decaying (-U(5, 20)), half nearly neutral (-10^U(-9,-4)),
    2% exact zeros and 1% -inf (document starts)."""
    g = np.random.default_rng(np.random.SeedSequence([seed, 11]))
    big = -g.uniform(5.0, 20.0, size=(nrows, length))
    tiny = -np.power(10.0, g.uniform(-9.0, -4.0, size=(nrows, length)))
    pick = g.random((nrows, length))
    ell = np.where(pick < 0.5, big, tiny)
    u = g.random((nrows, length))
    ell = np.where(u < 0.02, 0.0, ell)
    ell = np.where((u >= 0.02) & (u < 0.03), -np.inf, ell)
    return ell.astype(np.float32)


def varlen_logdecay_rows(nrows: int, length: int, seed: int = 101) -> np.ndarray:
    """Rows of dt * A with the packed-varlen stress distribution
    (dt = softplus(N(2, 2)), A = -U(1, 16)); per-chunk sums reach about -1e3."""
    g = np.random.default_rng(np.random.SeedSequence([seed, 12]))
    dt = _softplus(g.normal(2.0, 2.0, size=(nrows, length))).astype(np.float32)
    A = (-g.uniform(1.0, 16.0, size=(nrows, 1))).astype(np.float32)
    return (dt * A).astype(np.float32)


def config_decode(batch: int = 256) -> SSDProblem:
    """One decode step of the 2.7B-like layer: one token per batch row from a
    resident state (seqlen 1 with initial states)."""
    return make_problem(batch=batch, seqlen=1, nheads=80, headdim=64, dstate=128, ngroups=1, chunk=128,
                        dtype="bf16", seed=5, init_std=0.1, name=f"decode_b{batch}_H80_P64_N128_G1")
