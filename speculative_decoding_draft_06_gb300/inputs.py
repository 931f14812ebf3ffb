"""Seeded synthetic inputs for DARTree supertree builds.

This module only draws random numbers and lays them out. It holds none of the
method's arithmetic (no head step, no softmax, no selection), so the CPU oracle
and the CUDA path can both be fed from it without sharing any computation.

What it stands in for (the pages measure on trained Qwen3 drafters over public
suites, which are not used here):

* ``z[r, d, :]`` stands in for the diffusion drafter's position-wise marginals
  ("DARTree: Teaching a Chain-Trained Corrector to Think in Trees", Core
  Mechanism: one drafter forward gives L position-wise distributions).  Each
  row is ``sigma * N(0, 1) + log Zipf_s(rank)`` scattered through a seeded
  permutation of the vocabulary, in fp32.
* ``A [H, H]``, ``E [V, H]``, ``Wout [V, H]`` are the weights of the synthetic
  correction head ``s' = tanh(A s + E[tok])``, ``logits = z_d + s' Wout^T``
  (the pages never give the head's architecture).  Entries are
  ``N(0, 1/H)``; in bf16 workloads they are rounded to bf16 (round to nearest
  even) and kept as raw 16-bit patterns (``uint16``).
* ``state0 [R, H]`` is each request's head state at the verified prefix,
  ``N(0, 1)`` in fp32.

Seeding: ``numpy.random.SeedSequence(seed)`` is split into fixed children per
tensor and per row chunk, so the arrays do not depend on how many threads
generate them.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK_ROWS = 4096  # rows per independently seeded chunk of a weight matrix


@dataclasses.dataclass(frozen=True)
class Workload:
    """One supertree-build workload: shapes, budgets and the input recipe."""

    name: str
    V: int          # vocabulary size
    H: int          # head state width
    D: int          # draft depth (number of head calls)
    W: int          # layer width (frontier size kept per depth)
    K: int          # children expanded per frontier node
    B: int          # verification budget (Top-B)
    beta: float     # depth bonus, <= 0
    bf16: bool      # weights in bf16 (True) or fp32 (False)
    R: int = 1      # independent requests built in one call
    zipf_s: float = 1.1
    sigma: float = 2.0
    seed: int = 0

    def frontier_sizes(self) -> list[int]:
        """|F_1..F_D| with |F_0| = 1 and |F_d| = min(W, K |F_{d-1}|)."""
        f, out = 1, []
        for _ in range(self.D):
            f = min(self.W, self.K * f)
            out.append(f)
        return out

    def pool_size(self) -> int:
        return sum(self.frontier_sizes())

    def head_rows(self) -> list[int]:
        """Rows that go through the head at each depth: R * |F_{d-1}|."""
        prev = [1] + self.frontier_sizes()[:-1]
        return [self.R * f for f in prev]

    def candidates_per_build(self) -> int:
        """Children scored per call: R * sum_d K |F_{d-1}|."""
        return sum(self.K * m for m in self.head_rows())

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _base_seed(index: int) -> int:
    return 20261202 + 1000 * index


# The five workloads of the build.  Shapes follow Qwen3-4B / Qwen3-8B
# (vocabulary 151936, hidden 2560 / 4096).
CONFIGS: dict[str, Workload] = {
    "tiny": Workload("tiny", V=32000, H=256, D=8, W=4, K=4, B=16, beta=0.0,
                     bf16=False, zipf_s=1.1, sigma=2.0, seed=_base_seed(0)),
    "q4b": Workload("q4b", V=151936, H=2560, D=16, W=8, K=8, B=64, beta=0.0,
                    bf16=True, zipf_s=1.1, sigma=2.0, seed=_base_seed(1)),
    "q8b": Workload("q8b", V=151936, H=4096, D=16, W=16, K=16, B=128,
                    beta=-0.1, bf16=True, zipf_s=1.0, sigma=3.0,
                    seed=_base_seed(2)),
    "batch": Workload("batch", V=151936, H=4096, D=16, W=8, K=8, B=64,
                      beta=0.0, bf16=True, R=32, zipf_s=1.1, sigma=2.0,
                      seed=_base_seed(3)),
    "wide": Workload("wide", V=151936, H=4096, D=16, W=64, K=32, B=256,
                     beta=-0.5, bf16=True, zipf_s=1.2, sigma=2.0,
                     seed=_base_seed(4)),
}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits.

    Input preparation only (the weights are *given* in bf16).  Inputs here
    are finite, so no NaN handling is needed.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (b >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _normal_matrix(ss: np.random.SeedSequence, rows: int, cols: int,
                   scale: float, bf16: bool) -> np.ndarray:
    """rows x cols of N(0, scale^2), chunked by rows with fixed child seeds."""
    n_chunks = (rows + _CHUNK_ROWS - 1) // _CHUNK_ROWS
    children = ss.spawn(n_chunks)
    out = np.empty((rows, cols), dtype=np.uint16 if bf16 else np.float32)

    def fill(c: int) -> None:
        r0 = c * _CHUNK_ROWS
        r1 = min(rows, r0 + _CHUNK_ROWS)
        g = np.random.Generator(np.random.PCG64(children[c]))
        blk = g.standard_normal((r1 - r0, cols), dtype=np.float32)
        blk *= np.float32(scale)
        out[r0:r1] = to_bf16_bits(blk) if bf16 else blk

    if n_chunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def zipf_log_probs(V: int, s: float) -> np.ndarray:
    """log p_s(k) for ranks k = 1..V, p_s(k) = k^-s / sum_k' k'^-s (fp64)."""
    k = np.arange(1, V + 1, dtype=np.float64)
    logw = -s * np.log(k)
    m = logw.max()
    return logw - (m + np.log(np.exp(logw - m).sum()))


def make_base_logits(w: Workload, ss: np.random.SeedSequence) -> np.ndarray:
    """z[R, D, V] fp32: per (request, depth) seeded permutation of Zipf + noise."""
    logp = zipf_log_probs(w.V, w.zipf_s)
    z = np.empty((w.R, w.D, w.V), dtype=np.float32)
    kids = ss.spawn(w.R * w.D)

    def fill(i: int) -> None:
        r, d = divmod(i, w.D)
        g = np.random.Generator(np.random.PCG64(kids[i]))
        perm = g.permutation(w.V)
        noise = g.standard_normal(w.V, dtype=np.float64)
        row = np.empty(w.V, dtype=np.float64)
        row[perm] = w.sigma * noise + logp
        z[r, d] = row.astype(np.float32)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(w.R * w.D)))
    return z


def make_inputs(w: Workload, *, zero_wout: bool = False) -> dict:
    """All inputs of one build call, on the host.

    Returns a dict with ``z`` [R,D,V] f32, ``state0`` [R,H] f32 and the head
    ``A`` [H,H], ``E`` [V,H], ``Wout`` [V,H] (uint16 bf16 bits or f32).
    ``zero_wout`` replaces Wout by zeros (the uncorrected-tree special case).
    """
    root = np.random.SeedSequence(w.seed)
    s_w, s_z, s_s = root.spawn(3)
    s_a, s_e, s_o = s_w.spawn(3)
    scale = 1.0 / np.sqrt(w.H)
    A = _normal_matrix(s_a, w.H, w.H, scale, w.bf16)
    E = _normal_matrix(s_e, w.V, w.H, scale, w.bf16)
    if zero_wout:
        Wout = np.zeros((w.V, w.H), dtype=np.uint16 if w.bf16 else np.float32)
    else:
        Wout = _normal_matrix(s_o, w.V, w.H, scale, w.bf16)
    z = make_base_logits(w, s_z)
    g = np.random.Generator(np.random.PCG64(s_s))
    state0 = g.standard_normal((w.R, w.H), dtype=np.float32)
    return {"z": z, "state0": state0, "A": A, "E": E, "Wout": Wout}


def small_workload(seed: int, *, V: int, H: int, D: int, W: int, K: int,
                   B: int, beta: float = 0.0, bf16: bool = True, R: int = 1,
                   zipf_s: float = 1.1, sigma: float = 2.0) -> Workload:
    """A parity-test workload of arbitrary (small) shape."""
    return Workload(f"small-{seed}", V=V, H=H, D=D, W=W, K=K, B=B, beta=beta,
                    bf16=bf16, R=R, zipf_s=zipf_s, sigma=sigma,
                    seed=90000 + seed)


# ------------------------------------------------ verification consumer

@dataclasses.dataclass(frozen=True)
class VerifyShape:
    """One attention layer of a synthetic target over prefix + draft tree.
    Qwen3-8B attention shape: 32 query heads, 8 key/value heads, head dim 128
    (Hq * dh = 4096 = the hidden size, so the layer's output feeds an output
    projection of the head's shape)."""
    Lp: int = 2048
    Hq: int = 32
    Hkv: int = 8
    dh: int = 128
    seed: int = 20261202 + 7000


def make_verify_inputs(R: int, B: int, s: VerifyShape) -> dict:
    """Seeded synthetic Q [R,B+1,Hq,dh], prefix Kp/Vp [R,Lp,Hkv,dh] and tree
    Kt/Vt [R,B,Hkv,dh], all N(0,1) rounded to bf16 bits."""
    root = np.random.SeedSequence(s.seed + 31 * R + B)
    kids = root.spawn(5)
    shapes = [(R, B + 1, s.Hq, s.dh), (R, s.Lp, s.Hkv, s.dh), (R, s.Lp, s.Hkv, s.dh),
              (R, B, s.Hkv, s.dh), (R, B, s.Hkv, s.dh)]
    out = {}
    for name, ss, shp in zip(("Q", "Kp", "Vp", "Kt", "Vt"), kids, shapes):
        rows = int(np.prod(shp[:-1]))
        out[name] = _normal_matrix(ss, max(rows, 1), shp[-1], 1.0, True)[:rows].reshape(shp)
    return out


def random_tree(g: np.random.Generator, B: int, n_out: int | None = None) -> dict:
    """A random rooted tree in canonical form: parent ranks before their
    children (parent -1 = the root), distinct tokens among siblings; rows
    at or beyond n_out are empty (parent/token -1, depth 0)."""
    n_out = B if n_out is None else n_out
    parent = np.full(B, -1, np.int32)
    token = np.full(B, -1, np.int32)
    depth = np.zeros(B, np.int32)
    for n in range(n_out):
        parent[n] = -1 if n == 0 or g.random() < 0.2 else int(g.integers(0, n))
        sib = int(np.count_nonzero(parent[:n] == parent[n]))
        token[n] = 1000 * (parent[n] + 1) + sib
        depth[n] = 1 if parent[n] < 0 else depth[parent[n]] + 1
    return {"parent": parent, "token": token, "depth": depth, "n_out": n_out}
