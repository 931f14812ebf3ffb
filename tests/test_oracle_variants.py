"""Pins for the oracle's build variants (no GPU): the Markov correction
head, base-logit candidates and the sequential best-first baseline.

Each is tied to something other than the oracle's own code: the brute-force
path enumerator of tests/bruteforce.py (numpy, one path at a time), library
sorts and log-softmax, exhaustive k-best sums, closed forms (a K = V
candidate set is the whole vocabulary), and the equivalence of the
best-first build with the depth-wise build's Top-B when the beam prunes
nothing (Lemma 1 of "Technische Samenvatting: DARTree", Methodologie 2).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import bruteforce as bf


def _pool_vs_enumeration(o, ref, w):
    last = sorted((e for e in ref if e["depth"] == w.D), key=lambda e: -e["score"])
    ref = [e for e in ref if e["depth"] < w.D] + last[: w.W]
    paths = bf.pool_paths(o["pool_parent"], o["pool_token"])
    assert len(paths) == len(ref) == w.pool_size()
    got = {p: float(s) for p, s in zip(paths, o["pool_score"])}
    for e in ref:
        assert abs(got[e["path"]] - e["score"]) <= 1e-6, e["path"]


# ------------------------------------------------------------ Markov head

@pytest.mark.parametrize("bf16", [False, True])
def test_markov_construction_equals_bruteforce_with_zero_A(bf16):
    w = I.small_workload(700 + bf16, V=40, H=8, D=3, W=9, K=3, B=20, beta=-0.1, bf16=bf16)
    inp = I.make_inputs(w)
    o = oracle.build_tree(inp, 0, w.D, w.W, w.K, bf16, markov=True)
    ref = bf.enumerate_tree(bf.Head(inp, 0, bf16, markov=True), w.D, w.K)
    _pool_vs_enumeration(o, ref, w)


def test_markov_state_is_a_function_of_the_token():
    w = I.small_workload(710, V=30, H=16, D=4, W=12, K=4, B=20, bf16=True)
    inp = I.make_inputs(w)
    E = bf.weights_f64(inp["E"], True)
    for tok in (0, 7, 29):
        for par in (np.zeros(16, np.float32), np.ones(16, np.float32)):
            s = oracle.state_step(None, inp["E"], par, tok, True)
            want = bf.q(np.tanh(E[tok]).astype(np.float32), True)
            assert np.array_equal(s, want)
    # two kept nodes of a depth with the same token get the same head row
    o = oracle.build_tree(inp, 0, w.D, w.W, w.K, True, markov=True)
    F = [1] + w.frontier_sizes()
    off = 0
    for d in range(1, w.D):
        toks = o["pool_token"][off:off + F[d]]
        for a in range(F[d]):
            for b in range(a + 1, F[d]):
                if toks[a] == toks[b]:
                    assert o["row_lse"][d, a] == o["row_lse"][d, b]
                    assert np.array_equal(o["row_tok"][d, a], o["row_tok"][d, b])
        off += F[d]
    # and the recurrent head is a different tree on the same inputs
    r = oracle.build_tree(inp, 0, w.D, w.W, w.K, True)
    assert not np.array_equal(r["row_lse"][1:], o["row_lse"][1:])


# ------------------------------------------------- base-logit candidates

@pytest.mark.parametrize("bf16,markov", [(False, False), (True, False), (True, True)])
def test_base_candidates_equal_bruteforce_enumeration(bf16, markov):
    w = I.small_workload(720 + 2 * bf16 + markov, V=50, H=8, D=3, W=16, K=4, B=30,
                         beta=-0.3, bf16=bf16)
    inp = I.make_inputs(w)
    o = oracle.build_tree(inp, 0, w.D, w.W, w.K, bf16, markov=markov, cand_base=True)
    ref = bf.enumerate_tree(bf.Head(inp, 0, bf16, markov=markov), w.D, w.K, base=True)
    _pool_vs_enumeration(o, ref, w)


def test_base_candidates_are_the_base_top_k_and_normalise_over_K():
    w = I.small_workload(730, V=200, H=16, D=4, W=6, K=5, B=20, bf16=True)
    inp = I.make_inputs(w)
    o = oracle.build_tree(inp, 0, w.D, w.W, w.K, True, cand_base=True)
    F = [1] + w.frontier_sizes()
    for d in range(w.D):
        z = torch.from_numpy(inp["z"][0, d].astype(np.float64))
        top = set(torch.sort(z, descending=True, stable=True).indices[:w.K].tolist())
        for i in range(F[d]):
            assert set(o["row_tok"][d, i].tolist()) == top
            p = np.exp(o["row_logp"][d, i].astype(np.float64))
            assert abs(p.sum() - 1.0) <= 1e-6
            assert np.all(np.diff(o["row_logp"][d, i]) <= 0)


@pytest.mark.parametrize("seed,D,W,K", [(1, 4, 5, 3), (2, 3, 7, 4)])
def test_base_candidates_with_zero_wout_are_k_best_sums(seed, D, W, K):
    w = I.small_workload(740 + seed, V=60, H=8, D=D, W=W, K=K, B=8, bf16=True)
    inp = I.make_inputs(w, zero_wout=True)
    o = oracle.build_tree(inp, 0, D, W, K, True, cand_base=True)
    per_depth = []
    for d in range(D):
        z = torch.from_numpy(inp["z"][0, d].astype(np.float64))
        top = torch.sort(z, descending=True, stable=True).indices[:K]
        per_depth.append(torch.log_softmax(z[top], 0).numpy().astype(np.float32))
    want = bf.k_best_sums(per_depth, W)
    for d in range(1, D + 1):
        got = np.sort(o["pool_score"][o["pool_depth"] == d])[::-1]
        assert np.allclose(got, want[d - 1], atol=2e-6, rtol=0)


def test_base_candidates_with_K_equal_V_are_the_corrected_build():
    # all V tokens are candidates: the restricted normalisation is the full
    # softmax and the corrected top-K is every token
    w = I.small_workload(750, V=12, H=8, D=3, W=20, K=12, B=30, bf16=False)
    inp = I.make_inputs(w)
    a = oracle.build_tree(inp, 0, w.D, w.W, w.K, False, cand_base=True)
    b = oracle.build_tree(inp, 0, w.D, w.W, w.K, False)
    assert np.array_equal(a["pool_token"], b["pool_token"])
    assert np.array_equal(a["pool_parent"], b["pool_parent"])
    assert np.allclose(a["pool_score"], b["pool_score"], atol=1e-6, rtol=0)
    assert np.allclose(a["row_lse"], b["row_lse"], atol=1e-9, rtol=0, equal_nan=True)


def test_cand_row_against_torch():
    g = np.random.default_rng(9)
    V, H, K = 300, 16, 7
    z = g.standard_normal(V).astype(np.float32)
    Wout = (g.standard_normal((V, H)) / 4).astype(np.float32)
    s = g.standard_normal(H).astype(np.float32)
    cand = g.choice(V, K, replace=False).astype(np.int32)
    tok, val, lse = oracle.cand_row(z, Wout, s, cand, False)
    ell = torch.from_numpy(z.astype(np.float64)) + torch.from_numpy(Wout.astype(np.float64)) @ \
        torch.from_numpy(s.astype(np.float64))
    sub = ell[torch.from_numpy(cand.astype(np.int64))].float().double()
    assert abs(lse - torch.logsumexp(sub, 0).item()) <= 1e-12
    order = sorted(range(K), key=lambda j: (-float(sub[j]), int(cand[j])))
    assert np.array_equal(tok, cand[order])
    assert np.array_equal(val, sub[order].float().numpy())


# ----------------------------------------------- sequential best-first

BF_CASES = [
    dict(V=40, H=8, D=3, W=9, K=3, B=12, beta=-0.1, bf16=False),
    dict(V=64, H=16, D=4, W=8, K=2, B=15, beta=-0.5, bf16=True),
    dict(V=30, H=8, D=2, W=5, K=5, B=25, beta=0.0, bf16=True),
]


@pytest.mark.parametrize("case", range(len(BF_CASES)))
def test_bestfirst_pops_the_best_prefixes_of_the_full_tree(case):
    c = BF_CASES[case]
    w = I.small_workload(760 + case, **c)
    inp = I.make_inputs(w)
    o = oracle.bestfirst(inp, 0, w.D, w.K, w.B, w.beta, w.bf16)
    ref = bf.enumerate_tree(bf.Head(inp, 0, w.bf16), w.D, w.K)
    keys = sorted(((float(np.float32(np.float32(e["score"]) +
                                     np.float32(np.float32(w.beta) * np.float32(e["depth"])))),
                    e["depth"], e["path"], e["score"]) for e in ref),
                  key=lambda t: (-t[0], t[1]))
    n = min(w.B, len(ref))
    assert o["n_out"] == n
    got = bf.pool_paths(o["parent"][:n], o["token"][:n])
    assert got == [t[2] for t in keys[:n]]
    assert np.allclose(o["score"][:n], [t[3] for t in keys[:n]], atol=1e-6, rtol=0)
    # one call for the root plus one per popped node that was expanded
    expanded = [q for q in range(n - 1) if o["depth"][q] < w.D]
    assert o["calls"] == 1 + len(expanded)
    assert sorted(r for r in o["call_rank"] if r >= 0) == expanded


@pytest.mark.parametrize("case", range(len(BF_CASES)))
def test_bestfirst_equals_depthwise_topb_without_beam_pruning(case):
    c = dict(BF_CASES[case])
    c["W"] = c["K"] ** c["D"]       # every depth complete: the beam prunes nothing
    w = I.small_workload(770 + case, **c)
    inp = I.make_inputs(w)
    o = oracle.bestfirst(inp, 0, w.D, w.K, w.B, w.beta, w.bf16)
    t = oracle.build_request(inp, 0, w.D, w.W, w.K, w.B, w.beta, w.bf16)["tree"]
    assert o["n_out"] == t["n_out"]
    for k in ("parent", "token", "depth"):
        assert np.array_equal(o[k], t[k]), k
    assert np.array_equal(o["score"].view(np.uint32), t["score"].view(np.uint32))
    assert np.array_equal(o["mask"], t["mask"])


def test_bestfirst_depth_one_is_the_root_top_k():
    w = I.small_workload(780, V=50, H=8, D=1, W=4, K=6, B=10, bf16=False)
    inp = I.make_inputs(w)
    o = oracle.bestfirst(inp, 0, 1, w.K, w.B, -0.2, False)
    ell, lse = oracle.logits_row(inp["z"][0, 0], inp["Wout"], inp["state0"][0], False)
    order = np.argsort(-ell.astype(np.float64), kind="stable")[:w.K]
    assert o["calls"] == 1 and o["n_out"] == w.K
    assert np.array_equal(o["token"][:w.K], order)
    assert np.all(o["parent"][:w.K] == -1) and np.all(o["token"][w.K:] == -1)


def test_bestfirst_forcing_with_own_rows_and_states_is_identity():
    w = I.small_workload(790, V=40, H=8, D=4, W=8, K=3, B=14, beta=-0.2, bf16=True)
    inp = I.make_inputs(w)
    a = oracle.bestfirst(inp, 0, w.D, w.K, w.B, w.beta, True)
    b = oracle.bestfirst(inp, 0, w.D, w.K, w.B, w.beta, True, force_tok=a["row_tok"],
                         force_logp=a["row_logp"], force_state=a["call_state"])
    for k in ("parent", "token", "depth", "score", "mask", "call_rank"):
        assert np.array_equal(a[k], b[k]), k


def test_bestfirst_markov_head_equals_bruteforce():
    w = I.small_workload(795, V=30, H=8, D=3, W=9, K=3, B=10, beta=-0.1, bf16=True)
    inp = I.make_inputs(w)
    o = oracle.bestfirst(inp, 0, w.D, w.K, w.B, w.beta, True, markov=True)
    ref = bf.enumerate_tree(bf.Head(inp, 0, True, markov=True), w.D, w.K)
    keys = sorted(((float(np.float32(np.float32(e["score"]) +
                                     np.float32(np.float32(w.beta) * np.float32(e["depth"])))),
                    e["depth"], e["path"]) for e in ref), key=lambda t: (-t[0], t[1]))
    assert bf.pool_paths(o["parent"][:w.B], o["token"][:w.B]) == [t[2] for t in keys[:w.B]]
