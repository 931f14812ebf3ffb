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
