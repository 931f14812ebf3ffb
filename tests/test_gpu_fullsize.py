"""Parity at the five full workload sizes, in the launch configuration the
bench times (dartree_build on a created stream, so the captured graph).

The oracle cannot build the large trees in test time, so these tests check
(a) properties that hold at any size -- exactly D head calls, pool layout,
every score = parent score + that row's log-prob (one fp32 add), every
kept frontier = the top-W of the GPU's own candidates under the total
order, Top-B / compaction / mask bit-exact against the oracle on the GPU's
pool and equal to the best-first heap (Lemma 1) -- and (b) sampled head rows
recomputed by the oracle along the GPU's own paths (states from scratch,
full-vocabulary logits, log-sum-exp and top-K).  The tiny workload (fp32) is
compared in full with the teacher-forced oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import gpu_util as gu
from tests import parity

pytestmark = pytest.mark.gpu


def _run(w):
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx = gu.make_ctx(w)
    s = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    kw = dict(D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta, out=out, stream=s)
    for _ in range(2):                      # capture, then a replay
        ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], **kw)
    ctx.sync(s)
    res = {"pool": {k: v.numpy() for k, v in ctx.get_pool(w.R, w.pool_size()).items()},
           "tree": {k: v.cpu().numpy() for k, v in out.items()}, "rows": []}
    F = 1
    for d, fd in enumerate(w.frontier_sizes(), 1):
        res["rows"].append({k: v.numpy() for k, v in ctx.get_rows(d, w.R * F, w.K).items()})
        F = fd
    res["states"], F = [], 1
    for d, fd in enumerate(w.frontier_sizes(), 1):
        res["states"].append(ctx.get_states(d, w.R * F))
        F = fd
    res["head_calls"] = ctx.head_calls()
    ctx.close()
    return inp, res


def _check_properties(w, res):
    assert res["head_calls"] == w.D
    sizes = w.frontier_sizes()
    for r in range(w.R):
        pool, rows, tree = gu.split_request(res, w, r)
        slot, tok, _ = parity.forced_frontier(pool, w.D, w.W, w.K)
        off_prev, off, F = 0, 0, 1
        score_prev = np.zeros(1, np.float32)
        for d in range(1, w.D + 1):
            fd = sizes[d - 1]
            rw = rows[d - 1]
            # candidates of this depth from the GPU's own rows, total order
            c = (score_prev[:, None] + rw["logp"]).astype(np.float32)      # [F, K] fp32 add
            order = sorted(range(F * w.K), key=lambda e: (-float(c.flat[e]), e))[:fd]
            sl = slice(off, off + fd)
            assert np.array_equal(slot[sl], [e // w.K for e in order]), d
            assert np.array_equal(tok[sl], [rw["tok"].flat[e] for e in order]), d
            assert np.array_equal(pool["score"][sl].view(np.uint32),
                                  np.array([c.flat[e] for e in order], np.float32).view(np.uint32))
            score_prev = pool["score"][sl]
            off_prev, off, F = off, off + fd, fd
        ref = oracle.topb(pool["parent"], pool["token"], pool["depth"], pool["score"], w.B, w.beta)
        assert ref["rc"] == 0 and int(tree["n_out"]) == ref["n_out"]
        for k in ("parent", "token", "depth"):
            assert np.array_equal(tree[k], ref[k]), k
        assert np.array_equal(tree["mask"].reshape(ref["mask"].shape).view(np.uint32), ref["mask"])
        heap = oracle.heap_prune(pool["parent"], pool["depth"], pool["score"], w.B, w.beta)
        assert np.array_equal(ref["order"][:ref["n_out"]], heap)


def _check_sampled_rows(inp, w, res, samples):
    """Head rows recomputed by the oracle from the GPU's own states (the
    input of that head call), and the state steps that produced them."""
    tol = parity.TOL[w.bf16]
    offs = np.concatenate([[0], np.cumsum(w.frontier_sizes())])
    for (r, d, i) in samples:
        pool, rows, _ = gu.split_request(res, w, r)
        states = gu.request_states(res, w, r)
        s = states[d - 1][i]
        if d == 1:
            want = inp["state0"][r].astype(np.float32)
            if w.bf16:
                want = np.array([oracle.round_bf16(float(x)) for x in want], np.float32)
            assert np.array_equal(s, want)
        else:
            node = int(offs[d - 2]) + i                 # frontier slot i of depth d-1
            par = int(pool["parent"][node])
            ps = states[d - 2][0] if par < 0 else states[d - 2][par - int(offs[d - 3])]
            ref = oracle.state_step(inp["A"], inp["E"], ps, int(pool["token"][node]), w.bf16)
            ulp = np.spacing(np.abs(ref)) * (2 ** 16 if w.bf16 else 1)
            assert np.all(np.abs(s - ref) <= ulp + (2e-5 if w.bf16 else 2e-6)), (r, d, i)
        ell, lse = oracle.logits_row(inp["z"][r, d - 1], inp["Wout"], s, w.bf16)
        tk, val, gap = oracle.topk_row(ell, w.K)
        g_lse, g_tok, g_lp = rows[d - 1]["lse"][i], rows[d - 1]["tok"][i], rows[d - 1]["logp"][i]
        assert abs(g_lse - lse) <= 1e-4, (r, d, i, g_lse, lse)
        if gap >= parity.NEAR_TIE:
            assert set(g_tok.tolist()) == set(tk.tolist()), (r, d, i)
        ref_lp = (ell[g_tok].astype(np.float64) - lse).astype(np.float32)
        assert np.max(np.abs(g_lp - ref_lp)) <= min(tol, 1e-4), (r, d, i)
        assert np.all(np.diff(ell[g_tok]) <= parity.NEAR_TIE)


def test_tiny_full_oracle_parity():
    w = I.CONFIGS["tiny"]
    inp, res = _run(w)
    _check_properties(w, res)
    pool, rows, tree = gu.split_request(res, w, 0)
    rep = parity.compare_request(inp, 0, w.D, w.W, w.K, w.B, w.beta, w.bf16, pool, rows, tree,
                                 gpu_states=gu.request_states(res, w, 0))
    assert rep["near_ties"] <= 1


@pytest.mark.parametrize("name", ["q4b", "q8b", "wide", "batch"])
def test_full_size_properties_and_sampled_rows(name):
    w = I.CONFIGS[name]
    inp, res = _run(w)
    _check_properties(w, res)
    last = w.frontier_sizes()[-2]
    samples = [(0, 1, 0), (0, 2, 0), (0, 2, min(3, w.frontier_sizes()[0] - 1)),
               (0, w.D, last - 1)]
    if w.R > 1:
        samples += [(w.R - 1, 1, 0), (w.R // 2, w.D // 2, 1)]
    _check_sampled_rows(inp, w, res, samples)


# ------------------------------------------------ build variants at full size

def _run_variant(w, **variant):
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx = gu.make_ctx(w)
    s = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    kw = dict(D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta, out=out, stream=s, **variant)
    for _ in range(2):
        ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], **kw)
    ctx.sync(s)
    return inp, ctx, out


@pytest.mark.parametrize("variant", [dict(head="markov"), dict(candidates="base")])
def test_q8b_depthwise_variants_properties_and_sampled_rows(variant):
    w = I.CONFIGS["q8b"]
    inp, ctx, out = _run_variant(w, **variant)
    res = {"pool": {k: v.numpy() for k, v in ctx.get_pool(w.R, w.pool_size()).items()},
           "tree": {k: v.cpu().numpy() for k, v in out.items()}, "rows": [], "states": []}
    F = 1
    for d, fd in enumerate(w.frontier_sizes(), 1):
        res["rows"].append({k: v.numpy() for k, v in ctx.get_rows(d, w.R * F, w.K).items()})
        res["states"].append(ctx.get_states(d, w.R * F))
        F = fd
    res["head_calls"] = ctx.head_calls()
    ctx.close()
    _check_properties(w, res)
    markov = variant.get("head") == "markov"
    base = variant.get("candidates") == "base"
    pool, rows, _ = gu.split_request(res, w, 0)
    states = gu.request_states(res, w, 0)
    offs = np.concatenate([[0], np.cumsum(w.frontier_sizes())])
    tol = parity.TOL[True]
    for (d, i) in [(1, 0), (2, 3), (w.D, 15)]:
        s = states[d - 1][i]
        if d >= 2:                         # the state step that produced this row
            node = int(offs[d - 2]) + i
            par = int(pool["parent"][node])
            ps = states[d - 2][0] if par < 0 else states[d - 2][par - int(offs[d - 3])]
            ref = oracle.state_step(None if markov else inp["A"], inp["E"], ps,
                                    int(pool["token"][node]), True)
            ulp = np.spacing(np.abs(ref)) * 2 ** 16
            assert np.all(np.abs(s - ref) <= ulp + 2e-5), (d, i)
        g_lse, g_tok, g_lp = rows[d - 1]["lse"][i], rows[d - 1]["tok"][i], rows[d - 1]["logp"][i]
        if base:
            z = torch.from_numpy(inp["z"][0, d - 1].astype(np.float64))
            cand = torch.sort(z, descending=True, stable=True).indices[:w.K].numpy()
            assert set(g_tok.tolist()) == set(cand.tolist()), (d, i)
            tk, val, lse = oracle.cand_row(inp["z"][0, d - 1], inp["Wout"], s, cand, True)
            ref_lp = {int(t): float(np.float64(v) - lse) for t, v in zip(tk, val)}
        else:
            ell, lse = oracle.logits_row(inp["z"][0, d - 1], inp["Wout"], s, True)
            tk, _, gap = oracle.topk_row(ell, w.K)
            if gap >= parity.NEAR_TIE:
                assert set(g_tok.tolist()) == set(tk.tolist()), (d, i)
            ref_lp = {int(t): float(np.float64(ell[t]) - lse) for t in g_tok}
        assert abs(g_lse - lse) <= 1e-4, (d, i, g_lse, lse)
        assert max(abs(float(lp) - ref_lp[int(t)]) for t, lp in zip(g_tok, g_lp)) <= min(tol, 1e-4)


def test_q8b_bestfirst_properties_and_sampled_calls():
    w = I.CONFIGS["q8b"]
    inp, ctx, out = _run_variant(w, expansion="bestfirst")
    assert ctx.head_calls() == w.B
    t = {k: v.cpu().numpy()[0] for k, v in out.items()}
    n = int(t["n_out"])
    assert n == w.B
    calls = {}
    for c in sorted({0, 1, 2, n // 2, n - 1}):
        calls[c] = ({k: v.numpy()[0] for k, v in ctx.get_rows(c + 1, 1, w.K).items()},
                    ctx.get_states(c + 1, 1)[0])
    all_rows = [{k: v.numpy()[0] for k, v in ctx.get_rows(c + 1, 1, w.K).items()}
                for c in range(n)]
    ctx.close()
    beta = np.float32(w.beta)
    key = (t["score"][:n] + beta * t["depth"][:n].astype(np.float32)).astype(np.float32)
    assert np.all(np.diff(key) <= 0)                    # pops in best-first order
    for q in range(n):
        pr = int(t["parent"][q])
        assert pr < q
        assert t["depth"][q] == (1 if pr < 0 else t["depth"][pr] + 1)
        # its score is its parent's plus the log-prob its parent's call gave it
        row = all_rows[pr + 1]
        j = int(np.flatnonzero(row["tok"] == t["token"][q])[0])
        base = np.float32(0.0) if pr < 0 else t["score"][pr]
        assert np.float32(base + row["logp"][j]) == t["score"][q]
    words = (w.B + 31) // 32
    mask = t["mask"].reshape(w.B, words).view(np.uint32)
    for q in range(n):
        anc, u = set(), q
        while u >= 0:
            anc.add(u)
            u = int(t["parent"][u])
        bits = {j for j in range(w.B) if mask[q, j // 32] >> (j % 32) & 1}
        assert bits == anc
    for c, (row, s) in calls.items():          # sampled calls from the GPU's own states
        if c >= 1 and t["depth"][c - 1] >= w.D:
            continue
        d_child = 1 if c == 0 else int(t["depth"][c - 1]) + 1
        ell, lse = oracle.logits_row(inp["z"][0, d_child - 1], inp["Wout"], s, True)
        tk, _, gap = oracle.topk_row(ell, w.K)
        assert abs(row["lse"] - lse) <= 1e-4, (c, row["lse"], lse)
        if gap >= parity.NEAR_TIE:
            assert set(row["tok"].tolist()) == set(tk.tolist()), c
