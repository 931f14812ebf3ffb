"""Independent brute-force references used to pin the oracle.

Nothing here is shared with the oracle's C code or the CUDA path.  The head
stand-in is evaluated in numpy float64 (bf16 rounding through torch's own
bf16 conversion), and trees are enumerated path by path, recomputing every
state and score from scratch along each path -- no batching, no frontier
slots, no pool indices.
"""
from __future__ import annotations

import itertools

import numpy as np
import torch


def q(x: np.ndarray, bf16: bool) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    if not bf16:
        return x
    return torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float32).numpy()


def weights_f64(w: np.ndarray, bf16: bool) -> np.ndarray:
    if bf16:
        return (w.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return w.astype(np.float64)


class Head:
    """The synthetic correction head, evaluated one path at a time."""

    def __init__(self, inp: dict, r: int, bf16: bool, markov: bool = False):
        self.bf16 = bf16
        self.z = inp["z"][r].astype(np.float64)
        self.s0 = inp["state0"][r]
        # the Markov head is the A = 0 case of the recurrence
        self.A = np.zeros(inp["A"].shape) if markov else weights_f64(inp["A"], bf16)
        self.E = weights_f64(inp["E"], bf16)
        self.Wout = weights_f64(inp["Wout"], bf16)

    def root_state(self) -> np.ndarray:
        return q(self.s0, self.bf16)

    def step(self, s: np.ndarray, tok: int) -> np.ndarray:
        u = self.A @ s.astype(np.float64) + self.E[tok]
        return q(np.tanh(u).astype(np.float32), self.bf16)

    def row(self, s: np.ndarray, d: int):
        """(fp32 logits, fp64 log-sum-exp) of the depth-d distribution."""
        ell = (self.z[d - 1] + self.Wout @ s.astype(np.float64)).astype(np.float32)
        e = ell.astype(np.float64)
        m = e.max()
        return ell, m + np.log(np.exp(e - m).sum())

    def children(self, s: np.ndarray, d: int, K: int):
        """Top-K (token, fp32 logp) by (logit desc, token asc)."""
        ell, lse = self.row(s, d)
        order = np.argsort(-ell.astype(np.float64), kind="stable")[:K]
        return [(int(t), np.float32(np.float64(ell[t]) - lse)) for t in order]

    def children_base(self, s: np.ndarray, d: int, K: int):
        """Base-logit candidates: the top-K tokens of z_d, scored by the
        corrected logits at those tokens and normalised over the K; ordered
        by (corrected logit desc, token asc)."""
        z = self.z[d - 1]
        cand = np.argsort(-z, kind="stable")[:K]
        ell = (z[cand] + self.Wout[cand] @ s.astype(np.float64)).astype(np.float32)
        e = ell.astype(np.float64)
        lse = e.max() + np.log(np.exp(e - e.max()).sum())
        order = sorted(range(K), key=lambda j: (-float(ell[j]), int(cand[j])))
        return [(int(cand[j]), np.float32(e[j] - lse)) for j in order]


def enumerate_tree(head: Head, D: int, K: int, base: bool = False) -> list[dict]:
    """Every path of length 1..D through top-K children, with its score
    (children from the base-logit candidates when ``base``)."""
    out = []
    children = head.children_base if base else head.children

    def rec(path, state, score, d):
        if d > D:
            return
        for tok, logp in children(state, d, K):
            sc = np.float32(score + logp)
            p = path + (tok,)
            out.append({"path": p, "score": float(sc), "depth": d})
            if d < D:
                rec(p, head.step(state, tok), sc, d + 1)

    rec((), head.root_state(), np.float32(0.0), 1)
    return out


def pool_paths(parent: np.ndarray, token: np.ndarray) -> list[tuple]:
    """Token path of every pool node, following parent links."""
    paths = []
    for n in range(len(parent)):
        p, seq = n, []
        while p >= 0:
            seq.append(int(token[p]))
            p = int(parent[p])
        paths.append(tuple(reversed(seq)))
    return paths


def k_best_sums(per_depth_logp: list[np.ndarray], W: int) -> list[np.ndarray]:
    """Exhaustive: for each depth d, all sums of one value per depth 1..d,
    sorted descending and cut to W.  Values are accumulated in fp32 in depth
    order, exactly like a cumulative path score."""
    out = []
    for d in range(1, len(per_depth_logp) + 1):
        sums = []
        for combo in itertools.product(*[range(len(x)) for x in per_depth_logp[:d]]):
            s = np.float32(0.0)
            for dd, j in enumerate(combo):
                s = np.float32(s + per_depth_logp[dd][j])
            sums.append(float(s))
        out.append(np.sort(np.array(sums))[::-1][:W])
    return out
