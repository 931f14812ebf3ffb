"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: the definition of
bf16 rounding and torch's own conversion, closed forms of the head on
hand-built weights, library log-sum-exp / stable sort, brute-force
enumeration of every path, exhaustive k-best sums, a plain greedy loop,
Lemma 1 (global Top-B == sequential best-first heap for beta <= 0), the
ancestor-closure and mask invariants, and the weather/storm example.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------- bf16 rounding

def test_round_bf16_definition_cases():
    # spacing of bf16 at 1.0 is 2^-7; exact halves go to the even neighbour
    assert oracle.round_bf16(1.0) == 1.0
    assert oracle.round_bf16(1.0 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6
    assert oracle.round_bf16(1.0 + 2 ** -8 + 2 ** -20) == 1.0 + 2 ** -7
    assert oracle.round_bf16(-(1.0 + 3 * 2 ** -8)) == -(1.0 + 2 ** -6)
    assert oracle.round_bf16(float("inf")) == float("inf")
    assert math.isnan(oracle.round_bf16(float("nan")))


def test_round_bf16_matches_torch():
    g = np.random.default_rng(5)
    x = np.concatenate([g.standard_normal(20000).astype(np.float32),
                        (g.standard_normal(2000) * 1e-39).astype(np.float32),
                        (g.standard_normal(2000) * 1e30).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in x], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------ head closed forms

def test_logits_row_closed_form_single_column():
    # Wout[v, h] = c_v if h == h0 else 0 and s = a e_h0  =>  ell_v = z_v + a c_v
    V, H, h0, a = 37, 5, 3, 0.75
    g = np.random.default_rng(1)
    z = g.standard_normal(V).astype(np.float32)
    c = g.standard_normal(V).astype(np.float32)
    Wout = np.zeros((V, H), np.float32)
    Wout[:, h0] = c
    s = np.zeros(H, np.float32)
    s[h0] = a
    ell, lse = oracle.logits_row(z, Wout, s, bf16=False)
    want = (z.astype(np.float64) + a * c.astype(np.float64)).astype(np.float32)
    assert np.array_equal(ell, want)
    e = want.astype(np.float64)
    assert abs(lse - (e.max() + math.log(np.exp(e - e.max()).sum()))) < 1e-12


def test_logits_row_bf16_weights_are_widened_exactly():
    V, H = 9, 4
    Wf = np.array([[1.0, -2.0, 0.5, 0.0]] * V, np.float32) * np.arange(1, V + 1)[:, None]
    Wb = I.to_bf16_bits(Wf)           # these values are exact in bf16
    z = np.zeros(V, np.float32)
    s = np.array([1.0, 1.0, 2.0, 7.0], np.float32)
    ell, _ = oracle.logits_row(z, Wb, s, bf16=True)
    assert np.array_equal(ell, (Wf @ s).astype(np.float32))  # = 0 * v exactly
    s2 = np.array([1.0, 0.0, 0.0, 0.0], np.float32)
    ell2, _ = oracle.logits_row(z, Wb, s2, bf16=True)
    assert np.array_equal(ell2, np.arange(1, V + 1, dtype=np.float32))


def test_state_step_closed_form_permutation():
    # A = permutation matrix P (A[h, pi(h)] = 1) => u_h = s[pi(h)] + E[tok, h]
    H, V = 6, 4
    pi = np.array([2, 0, 5, 1, 3, 4])
    A = np.zeros((H, H), np.float32)
    A[np.arange(H), pi] = 1.0
    g = np.random.default_rng(2)
    E = g.standard_normal((V, H)).astype(np.float32)
    s = g.standard_normal(H).astype(np.float32)
    for tok in range(V):
        out = oracle.state_step(A, E, s, tok, bf16=False)
        want = np.tanh(s[pi].astype(np.float64) + E[tok].astype(np.float64)).astype(np.float32)
        assert np.array_equal(out, want)
    # bf16: the result is rounded to bf16 after the tanh
    out = oracle.state_step(I.to_bf16_bits(A), I.to_bf16_bits(E), s, 1, bf16=True)
    Eb = I.bf16_bits_to_f32(I.to_bf16_bits(E)).astype(np.float64)
    want = bf.q(np.tanh(s[pi].astype(np.float64) + Eb[1]).astype(np.float32), True)
    assert np.array_equal(out, want)


# ------------------------------------------- log-softmax / top-K vs torch

def test_lse_and_topk_against_torch():
    w = I.small_workload(3, V=777, H=48, D=1, W=1, K=1, B=1, bf16=True)
    inp = I.make_inputs(w)
    s = bf.q(inp["state0"][0], True)
    ell, lse = oracle.logits_row(inp["z"][0, 0], inp["Wout"], s, bf16=True)
    t = torch.from_numpy(ell.astype(np.float64))
    assert abs(lse - torch.logsumexp(t, 0).item()) < 1e-12
    assert abs(np.exp(ell.astype(np.float64) - lse).sum() - 1.0) < 1e-12
    for K in (1, 5, 32, 777):
        tok, val, gap = oracle.topk_row(ell, K)
        ref = torch.sort(t, descending=True, stable=True).indices[:K].numpy()
        assert np.array_equal(tok, ref)
        assert np.array_equal(val, ell[ref])
        if K < 777:
            nxt = torch.sort(t, descending=True, stable=True).indices[K].item()
            assert gap == np.float32(ell[ref[-1]] - ell[nxt])
        else:
            assert gap == float("inf")


def test_topk_ties_break_on_lower_token():
    ell = np.array([0.5, 2.0, 2.0, -np.inf, 2.0, 0.5, -np.inf], np.float32)
    tok, val, _ = oracle.topk_row(ell, 5)
    assert list(tok) == [1, 2, 4, 0, 5]
    tok, val, _ = oracle.topk_row(ell, 7)
    assert list(tok) == [1, 2, 4, 0, 5, 3, 6]


# ------------------------------------------------- brute-force construction

BRUTE_CASES = [
    dict(V=24, H=6, D=3, W=9, K=3, B=20, beta=0.0, bf16=False),
    dict(V=40, H=8, D=3, W=4, K=2, B=14, beta=-0.2, bf16=True),
    dict(V=64, H=16, D=4, W=8, K=2, B=30, beta=-1.0, bf16=True),
    dict(V=17, H=4, D=2, W=5, K=5, B=30, beta=-0.05, bf16=False),
    dict(V=50, H=12, D=4, W=27, K=3, B=40, beta=0.0, bf16=False),
]


@pytest.mark.parametrize("case", range(len(BRUTE_CASES)))
def test_construction_equals_bruteforce_enumeration(case):
    c = BRUTE_CASES[case]
    assert c["W"] >= c["K"] ** (c["D"] - 1)     # no pruning before depth D
    w = I.small_workload(100 + case, **c)
    inp = I.make_inputs(w)
    o = oracle.build_request(inp, 0, w.D, w.W, w.K, w.B, w.beta, w.bf16)
    ref = bf.enumerate_tree(bf.Head(inp, 0, w.bf16), w.D, w.K)
    # depths < D are complete; at depth D only the best W paths survive
    last = sorted((e for e in ref if e["depth"] == w.D), key=lambda e: -e["score"])
    ref = [e for e in ref if e["depth"] < w.D] + last[: w.W]
    paths = bf.pool_paths(o["pool_parent"], o["pool_token"])
    assert len(paths) == len(ref) == w.pool_size()
    got = {p: (float(s), int(d)) for p, s, d in zip(paths, o["pool_score"], o["pool_depth"])}
    for e in ref:
        s, d = got[e["path"]]
        assert d == e["depth"] == len(e["path"])
        assert abs(s - e["score"]) <= 1e-6
    # within a depth the pool is in rank order (score desc)
    for d in range(1, w.D + 1):
        sc = o["pool_score"][o["pool_depth"] == d]
        assert np.all(np.diff(sc) <= 0)
    # Top-B selects the B best keys among all enumerated prefixes
    keys = sorted(((np.float32(e["score"] + np.float32(np.float32(w.beta) * e["depth"])),
                    e["depth"], e["path"]) for e in ref),
                  key=lambda t: (-t[0], t[1]))
    want = {t[2] for t in keys[: min(w.B, len(ref))]}
    tr = o["tree"]
    sel = bf.pool_paths(tr["parent"][: tr["n_out"]], tr["token"][: tr["n_out"]])
    assert set(sel) == want and tr["rc"] == 0


def test_pool_size_closed_form():
    for (D, W, K, P) in [(8, 4, 4, 32), (16, 8, 8, 128), (16, 16, 16, 256),
                         (16, 64, 32, 32 + 64 * 15), (3, 9, 3, 3 + 9 + 9)]:
        assert oracle.pool_size(D, W, K) == P


# ------------------------------------------ uncorrected tree: k-best sums

@pytest.mark.parametrize("seed,D,W,K", [(1, 4, 5, 3), (2, 3, 7, 4), (3, 5, 4, 2)])
def test_zero_wout_tree_is_k_best_sums(seed, D, W, K):
    w = I.small_workload(200 + seed, V=60, H=8, D=D, W=W, K=K, B=8, bf16=True)
    inp = I.make_inputs(w, zero_wout=True)
    o = oracle.build_tree(inp, 0, D, W, K, True)
    per_depth = []
    for d in range(D):
        z = torch.from_numpy(inp["z"][0, d].astype(np.float64))
        lp = torch.log_softmax(z, 0)
        top = torch.sort(z, descending=True, stable=True).indices[:K]
        per_depth.append(lp[top].numpy().astype(np.float32))
        # every branch proposes the same K tokens: those of z_d
        F = [1] + w.frontier_sizes()
        for i in range(F[d]):
            assert np.array_equal(o["row_tok"][d, i], top.numpy())
    want = bf.k_best_sums(per_depth, W)
    for d in range(1, D + 1):
        got = np.sort(o["pool_score"][o["pool_depth"] == d])[::-1]
        assert np.allclose(got, want[d - 1], atol=2e-6, rtol=0)


# ------------------------------------------------------ W = 1 greedy chain

@pytest.mark.parametrize("bf16", [False, True])
def test_width_one_is_greedy_corrected_chain(bf16):
    w = I.small_workload(300 + bf16, V=120, H=16, D=6, W=1, K=4, B=6, bf16=bf16)
    inp = I.make_inputs(w)
    o = oracle.build_tree(inp, 0, w.D, 1, w.K, bf16)
    head = bf.Head(inp, 0, bf16)
    s, score, toks, scores = head.root_state(), np.float32(0), [], []
    for d in range(1, w.D + 1):
        ell, lse = head.row(s, d)
        t = int(np.argmax(ell))               # first (lowest) index among ties
        score = np.float32(score + np.float32(np.float64(ell[t]) - lse))
        toks.append(t)
        scores.append(float(score))
        s = head.step(s, t)
    assert list(o["pool_token"]) == toks
    assert list(o["pool_parent"]) == [-1] + list(range(w.D - 1))
    assert np.allclose(o["pool_score"], scores, atol=1e-6, rtol=0)


# ---------------------------------------- top-K inside the beam (K >= W)

def test_topk_candidates_lose_nothing_when_K_ge_W():
    w = I.small_workload(400, V=90, H=12, D=4, W=3, K=5, B=6, bf16=True)
    inp = I.make_inputs(w)
    o = oracle.build_tree(inp, 0, w.D, w.W, w.K, True)
    head = bf.Head(inp, 0, True)
    paths = bf.pool_paths(o["pool_parent"], o["pool_token"])
    frontier = [((), head.root_state(), np.float32(0.0))]
    off = 0
    for d in range(1, w.D + 1):
        allc = []
        for i, (p, s, sc) in enumerate(frontier):
            ell, lse = head.row(s, d)
            for v in range(w.V):
                allc.append((np.float32(sc + np.float32(np.float64(ell[v]) - lse)), i, v))
        allc.sort(key=lambda t: (-t[0], t[1], t[2]))
        fd = w.frontier_sizes()[d - 1]
        best = allc[:fd]
        for q, (c, i, v) in enumerate(best):
            assert paths[off + q] == frontier[i][0] + (v,)
            assert abs(o["pool_score"][off + q] - c) <= 1e-6
        frontier = [(frontier[i][0] + (v,), head.step(frontier[i][1], v), c)
                    for (c, i, v) in best]
        off += fd


# ----------------------------------------------------- Lemma 1 and pruning

def _random_pool(g, n_roots, n_nodes, tie_prob):
    """A random pool: scores never increase along a path (log-probs <= 0),
    with exact ties (log-prob 0) at probability tie_prob, in depth-major
    order like the construction produces."""
    parent, depth, score = [], [], []
    frontier = []
    for _ in range(n_roots):
        parent.append(-1); depth.append(1)
        score.append(np.float32(-g.exponential()))
        frontier.append(len(parent) - 1)
    while len(parent) < n_nodes:
        nxt = []
        for p in frontier:
            for _ in range(g.integers(0, 3)):
                if len(parent) >= n_nodes:
                    break
                lp = 0.0 if g.random() < tie_prob else -g.exponential()
                parent.append(p); depth.append(depth[p] + 1)
                score.append(np.float32(score[p] + np.float32(lp)))
                nxt.append(len(parent) - 1)
        if not nxt:
            break
        frontier = nxt
    return (np.array(parent, np.int32), np.array(depth, np.int32),
            np.array(score, np.float32))


@pytest.mark.parametrize("beta", [0.0, -0.05, -0.3, -2.0])
def test_lemma1_topb_equals_best_first_heap_random_pools(beta):
    g = np.random.default_rng(11)
    for trial in range(60):
        pp, pd, ps = _random_pool(g, int(g.integers(1, 6)), int(g.integers(2, 120)),
                                  tie_prob=0.3 if trial % 2 else 0.0)
        pt = np.arange(len(pp), dtype=np.int32)
        for B in (1, 3, 17, 500):
            tb = oracle.topb(pp, pt, pd, ps, B, beta)
            heap = oracle.heap_prune(pp, pd, ps, B, beta)
            assert tb["rc"] == 0
            assert np.array_equal(tb["order"][: tb["n_out"]], heap)


@pytest.mark.parametrize("beta", [0.0, -0.1, -0.5])
def test_lemma1_on_constructed_supertrees(beta):
    for seed in range(4):
        w = I.small_workload(500 + seed, V=200, H=16, D=5, W=6, K=4, B=12,
                             beta=beta, bf16=bool(seed % 2))
        inp = I.make_inputs(w)
        o = oracle.build_request(inp, 0, w.D, w.W, w.K, w.B, w.beta, w.bf16)
        heap = oracle.heap_prune(o["pool_parent"], o["pool_depth"], o["pool_score"],
                                 w.B, w.beta)
        assert np.array_equal(o["tree"]["order"][: o["tree"]["n_out"]], heap)


def test_positive_depth_bonus_breaks_lemma1():
    # a (depth 1, -1.0) -> b (depth 2, -1.1); c (depth 1, -1.05); beta = +1:
    # keys a 0.0, b 0.9, c -0.05.  Top-1 = {b} is not ancestor-closed, and
    # the heap (which can only pop a root first) disagrees.
    pp = np.array([-1, -1, 0], np.int32)
    pd = np.array([1, 1, 2], np.int32)
    ps = np.array([-1.0, -1.05, -1.1], np.float32)
    pt = np.array([10, 11, 12], np.int32)
    tb = oracle.topb(pp, pt, pd, ps, 1, 1.0)
    assert tb["rc"] == oracle.ORC_ERR_CLOSURE
    tb2 = oracle.topb(pp, pt, pd, ps, 2, 1.0)
    assert tb2["rc"] == oracle.ORC_ERR_ORDER
    heap = oracle.heap_prune(pp, pd, ps, 2, 1.0)
    assert list(heap) == [0, 2] and list(tb2["order"]) == [2, 0]
    # the same pool with beta <= 0 is fine
    assert oracle.topb(pp, pt, pd, ps, 2, 0.0)["rc"] == 0


def test_topb_hand_worked_example():
    # pool (depth-major): 0:a(d1,-0.5) 1:b(d1,-1.0) 2:a.x(d2,-0.7) 3:a.y(d2,-2.0)
    # 4:b.z(d2,-1.2) 5:a.x.w(d3,-0.9); beta = -0.25 -> keys
    # a -0.75, b -1.25, ax -1.2, ay -2.5, bz -1.7, axw -1.65
    # order: a, ax, b, axw, bz, ay
    pp = np.array([-1, -1, 0, 0, 1, 2], np.int32)
    pt = np.array([7, 8, 9, 10, 11, 12], np.int32)
    pd = np.array([1, 1, 2, 2, 2, 3], np.int32)
    ps = np.array([-0.5, -1.0, -0.7, -2.0, -1.2, -0.9], np.float32)
    tb = oracle.topb(pp, pt, pd, ps, 4, -0.25)
    assert tb["n_out"] == 4 and tb["rc"] == 0
    assert list(tb["order"]) == [0, 2, 1, 5]
    assert list(tb["parent"]) == [-1, 0, -1, 1]
    assert list(tb["token"]) == [7, 9, 8, 12]
    assert list(tb["depth"]) == [1, 2, 1, 3]
    assert list(tb["mask"][:, 0]) == [0b0001, 0b0011, 0b0100, 0b1011]
    tb = oracle.topb(pp, pt, pd, ps, 8, -0.25)      # B > P: all six, padded
    assert tb["n_out"] == 6
    assert list(tb["parent"][6:]) == [-1, -1] and list(tb["token"][6:]) == [-1, -1]
    assert list(tb["mask"][6:, 0]) == [0, 0]


def _check_tree_invariants(tr, B):
    n = tr["n_out"]
    words = (B + 31) // 32
    assert tr["mask"].shape == (B, words)
    for i in range(n):
        p = tr["parent"][i]
        assert p < i
        row = tr["mask"][i]
        bits = sum(bin(int(x)).count("1") for x in row)
        assert bits == tr["depth"][i]                      # self + ancestors
        assert (row[i // 32] >> (i % 32)) & 1
        for j in range(i + 1, B):                          # lower-triangular
            assert not (row[j // 32] >> (j % 32)) & 1
        want = np.zeros(words, np.uint32) if p < 0 else tr["mask"][p].copy()
        want[i // 32] |= np.uint32(1 << (i % 32))
        assert np.array_equal(row, want)
        if p >= 0:
            assert tr["depth"][p] == tr["depth"][i] - 1
        else:
            assert tr["depth"][i] == 1


@pytest.mark.parametrize("seed", range(4))
def test_selected_tree_is_ancestor_closed_and_mask_is_consistent(seed):
    w = I.small_workload(600 + seed, V=150, H=16, D=6, W=5, K=3, B=[7, 19, 33, 40][seed],
                         beta=[0.0, -0.1, -1.0, -0.01][seed], bf16=True)
    inp = I.make_inputs(w)
    o = oracle.build_request(inp, 0, w.D, w.W, w.K, w.B, w.beta, w.bf16)
    assert o["tree"]["rc"] == 0
    assert o["tree"]["n_out"] == min(w.B, w.pool_size())
    _check_tree_invariants(o["tree"], w.B)


def test_exactly_D_head_calls():
    for D in (1, 2, 7):
        w = I.small_workload(700 + D, V=80, H=8, D=D, W=3, K=2, B=4, bf16=False)
        o = oracle.build_tree(I.make_inputs(w), 0, D, 3, 2, False)
        assert o["calls"] == D


def test_teacher_forcing_with_own_choice_is_identity():
    w = I.small_workload(800, V=120, H=16, D=5, W=4, K=3, B=9, bf16=True)
    inp = I.make_inputs(w)
    a = oracle.build_tree(inp, 0, w.D, w.W, w.K, True)
    b = oracle.build_tree(inp, 0, w.D, w.W, w.K, True,
                          force_slot=a["own_slot"], force_tok=a["own_tok"])
    for k in ("pool_parent", "pool_token", "pool_depth", "pool_score", "own_slot",
              "own_tok", "own_score"):
        assert np.array_equal(a[k], b[k]), k
    assert np.all(b["force_margin"] >= 0)


def test_state_forcing_with_own_states_is_identity():
    w = I.small_workload(802, V=150, H=16, D=4, W=4, K=3, B=9, bf16=True)
    inp = I.make_inputs(w)
    a = oracle.build_tree(inp, 0, w.D, w.W, w.K, True)
    # the oracle's own head states, depth by depth, from its own frontier
    st = np.zeros((w.D, w.W, w.H), np.float32)
    rows = [bf.q(inp["state0"][0], True)]
    off, sizes = 0, w.frontier_sizes()
    for d in range(w.D):
        for i, s in enumerate(rows):
            st[d, i] = s
        fd = sizes[d]
        rows = [oracle.state_step(inp["A"], inp["E"], rows[a["own_slot"][off + q]],
                                  int(a["own_tok"][off + q]), True) for q in range(fd)]
        off += fd
    b = oracle.build_tree(inp, 0, w.D, w.W, w.K, True, force_state=st)
    for k in ("pool_parent", "pool_token", "pool_score", "row_lse", "row_logp"):
        assert np.array_equal(a[k], b[k], equal_nan=k.startswith("row")), k


def test_teacher_forcing_scores_an_off_beam_choice():
    w = I.small_workload(801, V=120, H=16, D=3, W=2, K=2, B=4, bf16=False)
    inp = I.make_inputs(w)
    a = oracle.build_tree(inp, 0, w.D, w.W, w.K, False)
    fs, ft = a["own_slot"].copy(), a["own_tok"].copy()
    ft[1] = (ft[1] + 7) % w.V                     # force a token outside top-K
    b = oracle.build_tree(inp, 0, w.D, w.W, w.K, False, force_slot=fs, force_tok=ft)
    head = bf.Head(inp, 0, False)
    ell, lse = head.row(head.root_state(), 1)
    assert b["pool_token"][1] == ft[1]
    assert abs(b["pool_score"][1] - np.float32(np.float64(ell[ft[1]]) - lse)) <= 1e-6
    assert b["force_margin"][1] < 0


# ------------------------------------------------ one depth on its own

@pytest.mark.parametrize("bf16,cand_base", [(False, False), (True, False), (True, True)])
def test_depth_replays_every_depth_of_a_build(bf16, cand_base):
    """orc_depth called alone, with a depth's input states and the previous
    frontier's scores, gives bit for bit what that depth gave inside the
    build (the build is pinned by brute force above)."""
    w = I.small_workload(810 + 2 * bf16 + cand_base, V=150, H=16, D=4, W=5, K=3, B=9,
                         bf16=bf16)
    inp = I.make_inputs(w)
    g = np.random.default_rng(3)
    st = np.tanh(g.standard_normal((w.D, w.W, w.H))).astype(np.float32)
    st = bf.q(st, bf16)
    a = oracle.build_tree(inp, 0, w.D, w.W, w.K, bf16, force_state=st, cand_base=cand_base)
    sizes, off, F, prev = w.frontier_sizes(), 0, 1, np.zeros(1, np.float32)
    for d in range(1, w.D + 1):
        fd = sizes[d - 1]
        o = oracle.depth(inp["z"][0, d - 1], inp["Wout"], st[d - 1, :F], prev, w.W, w.K, bf16,
                         cand_base=cand_base)
        sl = slice(off, off + fd)
        for k in ("own_slot", "own_tok", "own_score"):
            assert np.array_equal(o[k], a[k][sl]), (d, k)
        assert np.array_equal(o["sel_score"], a["pool_score"][sl])
        assert np.array_equal(o["sel_logp"], a["pool_logp"][sl])
        assert np.array_equal(o["row_lse"], a["row_lse"][d - 1, :F])
        assert np.array_equal(o["row_tok"], a["row_tok"][d - 1, :F])
        assert np.array_equal(o["row_logp"], a["row_logp"][d - 1, :F])
        assert np.array_equal(o["w_cut"], a["w_cut"][d - 1])
        prev, off, F = o["sel_score"], off + fd, fd


def test_depth_from_given_rows_equals_bruteforce():
    """Arbitrary frontier states and scores: the rows are the brute-force
    head's top-K children, the own top-W is the best fd of all F*K
    candidates score_i + logp_ij (fp32), ties on the lower index."""
    V, H, K, W, F = 70, 8, 4, 6, 3
    w = I.small_workload(820, V=V, H=H, D=2, W=W, K=K, B=4, bf16=False)
    inp = I.make_inputs(w)
    head = bf.Head(inp, 0, False)
    g = np.random.default_rng(9)
    st = np.tanh(g.standard_normal((F, H))).astype(np.float32)
    score = (-np.abs(g.standard_normal(F)) * 3).astype(np.float32)
    o = oracle.depth(inp["z"][0, 1], inp["Wout"], st, score, W, K, False)
    cands = []
    for i in range(F):
        ch = head.children(st[i], 2, K)
        assert [t for t, _ in ch] == o["row_tok"][i].tolist()
        assert np.allclose([lp for _, lp in ch], o["row_logp"][i], atol=1e-6, rtol=0)
        cands += [(np.float32(score[i] + lp), i * K + j, t) for j, (t, lp) in enumerate(ch)]
    best = sorted(cands, key=lambda c: (-float(c[0]), c[1]))
    fd = min(W, F * K)
    assert o["own_slot"].tolist() == [c[1] // K for c in best[:fd]]
    assert o["own_tok"].tolist() == [c[2] for c in best[:fd]]
    assert np.allclose(o["own_score"], [c[0] for c in best[:fd]], atol=2e-6, rtol=0)
    assert abs(o["w_cut"][1] - best[fd][0]) <= 2e-6
    # no forcing: the kept frontier is the own one, log-probs as in the rows
    assert np.array_equal(o["sel_slot"], o["own_slot"])
    for q in range(fd):
        j = o["row_tok"][o["sel_slot"][q]].tolist().index(o["sel_tok"][q])
        assert o["sel_logp"][q] == o["row_logp"][o["sel_slot"][q], j]
    # a forced frontier is scored from the given scores
    fs = np.array([2, 0, 1, 2, 0, 1], np.int32)
    ft = np.array([int(o["row_tok"][s_, 1]) for s_ in fs], np.int32)
    f = oracle.depth(inp["z"][0, 1], inp["Wout"], st, score, W, K, False, force_slot=fs,
                     force_tok=ft)
    for q in range(fd):
        assert f["sel_score"][q] == np.float32(score[fs[q]] + o["row_logp"][fs[q], 1])
        assert f["force_margin"][q] >= 0


def test_path_scores_are_per_path_fp32_sums():
    g = np.random.default_rng(4)
    P = 60
    parent = np.array([-1 if n < 3 or g.random() < 0.1 else int(g.integers(0, n))
                       for n in range(P)], np.int32)
    logp = (-np.abs(g.standard_normal(P)) * 2).astype(np.float32)
    got = oracle.path_scores(parent, logp)
    for n in range(P):
        path, u = [], n
        while u >= 0:
            path.append(u)
            u = int(parent[u])
        s_ = np.float32(0.0)
        for u in reversed(path):                 # root side first
            s_ = np.float32(s_ + logp[u])
        assert got[n] == s_, n
    bad = parent.copy()
    bad[5] = 7
    with pytest.raises(RuntimeError):
        oracle.path_scores(bad, logp)


# ------------------------------------------- the weather / storm example

def _weather_inputs(zero_wout=False):
    gdn = json.load(open(os.path.join(GOLDEN, "weather_storm.json")))
    vocab = gdn["vocab"]
    tid = {t: i for i, t in enumerate(vocab)}
    V, H, D = len(vocab), 2, len(gdn["marginals"])
    z = np.full((1, D, V), np.log(1e-6), np.float32)
    for d, m in enumerate(gdn["marginals"]):
        for t, p in m.items():
            z[0, d, tid[t]] = np.float32(np.log(p))
    g, alpha, c = 4.0, 3.0, 3.0
    sign = {"the": 1, "weather": 1, "lovely": 1, "a": -1, "storm": -1, "coming": -1}
    E = np.zeros((V, H), np.float32)
    Wout = np.zeros((V, H), np.float32)
    for t, s in sign.items():
        E[tid[t]] = [s * g, -s * g]
        if t in ("weather", "storm", "lovely", "coming") and not zero_wout:
            Wout[tid[t]] = [s * c, -s * c]
    inp = {"z": z, "state0": np.zeros((1, H), np.float32),
           "A": (alpha * np.eye(H)).astype(np.float32), "E": E, "Wout": Wout}
    return gdn, vocab, inp


def test_weather_storm_corrected_tree_keeps_only_coherent_paths():
    gdn, vocab, inp = _weather_inputs()
    D, W, K = 4, 2, 2
    o = oracle.build_tree(inp, 0, D, W, K, False)
    paths = bf.pool_paths(o["pool_parent"], o["pool_token"])
    last = [tuple(vocab[t] for t in p) for p, d in zip(paths, o["pool_depth"]) if d == D]
    assert set(last) == {tuple(p) for p in gdn["coherent_paths"]}
    for p, s, d in zip(paths, o["pool_score"], o["pool_depth"]):
        if d == D:
            assert abs(s - math.log(0.5)) < 1e-3       # each has joint prob 1/2
    assert tuple(gdn["incoherent_example"][:2]) not in {
        tuple(vocab[t] for t in p) for p in paths}


def test_weather_storm_uncorrected_tree_assembles_incoherent_path():
    gdn, vocab, inp = _weather_inputs(zero_wout=True)
    o = oracle.build_tree(inp, 0, 4, 2, 2, False)
    paths = {tuple(vocab[t] for t in p)
             for p in bf.pool_paths(o["pool_parent"], o["pool_token"])}
    assert tuple(gdn["incoherent_example"][:2]) in paths
    coherent = {tuple(p) for p in gdn["coherent_paths"]}
    deepest = {p for p in paths if len(p) == 4}
    assert deepest and not deepest <= coherent     # an incoherent sentence kept
