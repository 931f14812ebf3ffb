"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small cases span several 128-row vocabulary tiles with a ragged tail, every
padded head-row count (16 .. 256), single and multiple requests, fp32 and
bf16 weights.  Comparison rule (tests/parity.py): structure bit-exact except
counted near-ties (< 1e-4), scores within 2e-3 (bf16) / 1e-5 (fp32); Top-B,
compaction and mask bit-exact on the GPU's pool.
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

SMALL = [
    # (name, workload kwargs)
    ("f32-ragged", dict(V=1000, H=64, D=4, W=4, K=4, B=12, beta=0.0, bf16=False)),
    ("f32-wide", dict(V=777, H=40, D=3, W=20, K=7, B=40, beta=-0.3, bf16=False)),
    ("bf16-n16", dict(V=3000, H=128, D=5, W=8, K=8, B=30, beta=0.0, bf16=True)),
    ("bf16-n32", dict(V=2049, H=192, D=4, W=32, K=6, B=64, beta=-0.1, bf16=True)),
    ("bf16-n64", dict(V=1500, H=64, D=3, W=64, K=32, B=100, beta=-0.5, bf16=True)),
    ("bf16-n128", dict(V=1300, H=128, D=3, W=100, K=5, B=128, beta=-0.05, bf16=True)),
    # frontiers of 33..64 (the 64-key warp fold of the top-W), two requests
    ("bf16-w48", dict(V=900, H=64, D=5, W=48, K=3, B=60, beta=-0.2, bf16=True, R=2)),
    ("bf16-batch", dict(V=1100, H=64, D=4, W=8, K=8, B=40, beta=0.0, bf16=True, R=32)),
    # z rows of the requests at an odd stride (3 * 1101 floats): unaligned loads
    ("bf16-batch-odd", dict(V=1101, H=128, D=3, W=8, K=4, B=30, beta=-0.2, bf16=True, R=20)),
    ("bf16-k1w1", dict(V=500, H=64, D=6, W=1, K=1, B=6, beta=0.0, bf16=True)),
    ("bf16-bigB", dict(V=700, H=64, D=3, W=6, K=3, B=200, beta=-1.0, bf16=True, R=2)),
    # the build limits: W = 256 (256-row head calls on CTA pairs, a top-W over
    # 8192 candidates), K = 32, B = 1024 <= P = 1056
    ("bf16-max", dict(V=1500, H=64, D=5, W=256, K=32, B=1024, beta=-0.05, bf16=True)),
    # fp32 at the limits, B above the pool (P = 800)
    ("f32-max", dict(V=700, H=32, D=4, W=256, K=32, B=1024, beta=0.0, bf16=False)),
    # fp32, three requests of 4 rows: the state contraction rides on the head
    # call (two state tiles, the second ragged) and each request's selection
    # finishes its own rows
    ("f32-multi", dict(V=1000, H=200, D=4, W=4, K=3, B=10, beta=-0.1, bf16=False, R=3)),
]


@pytest.mark.parametrize("idx", range(len(SMALL)), ids=[s[0] for s in SMALL])
def test_build_matches_oracle_small(idx):
    name, kw = SMALL[idx]
    w = I.small_workload(500 + idx, **kw)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx = gu.make_ctx(w)
    res = gu.run_build(ctx, w, dev)
    assert res["head_calls"] == w.D
    tot = {"near_ties": 0, "topk_near_ties": 0}
    for r in range(w.R):
        pool, rows, tree = gu.split_request(res, w, r)
        rep = parity.compare_request(inp, r, w.D, w.W, w.K, w.B, w.beta, w.bf16, pool, rows, tree,
                                     gpu_states=gu.request_states(res, w, r))
        for k in tot:
            tot[k] += rep[k]
    # near-ties must stay rare on random data
    assert tot["near_ties"] <= max(2, w.R // 4)
    ctx.close()


@pytest.mark.parametrize("name", ["bf16-n16", "bf16-batch", "f32-ragged"])
def test_build_with_the_row_group_merge_matches_oracle(monkeypatch, name):
    """The per-row group merge (every CTA list folded), forced here instead
    of the merge through the row bound, gives the same trees."""
    monkeypatch.setenv("DARTREE_MERGE_BOUND", "0")
    test_build_matches_oracle_small([s[0] for s in SMALL].index(name))


@pytest.mark.parametrize("name", ["bf16-n16", "bf16-batch", "bf16-k1w1", "f32-ragged",
                                  "f32-multi"])
def test_build_with_the_global_row_hand_over_matches_oracle(monkeypatch, name):
    """The row blocks of a request handing their results to the selection
    through global memory and an arrival count (instead of a thread-block
    cluster and the leader's shared memory) give the same trees."""
    monkeypatch.setenv("DARTREE_MERGE_CLUSTER", "0")
    test_build_matches_oracle_small([s[0] for s in SMALL].index(name))


@pytest.mark.parametrize("name", ["bf16-n16", "bf16-n32", "bf16-batch", "f32-ragged",
                                  "f32-multi"])
def test_build_with_the_merge_fold_top_w_matches_oracle(monkeypatch, name):
    """The top-W by warp merge folds (instead of rank counting) gives the
    same trees."""
    monkeypatch.setenv("DARTREE_RANK_MAX", "0")
    test_build_matches_oracle_small([s[0] for s in SMALL].index(name))


@pytest.mark.parametrize("name", ["f32-ragged", "f32-multi"])
def test_build_with_a_separate_state_step_matches_oracle(monkeypatch, name):
    """fp32 builds of at most 16 rows with the state step as its own kernel
    (instead of folded into the head call and the selection) give the same
    trees."""
    monkeypatch.setenv("DARTREE_F32_FOLD", "0")
    test_build_matches_oracle_small([s[0] for s in SMALL].index(name))


@pytest.mark.parametrize("name", ["bf16-n16", "bf16-w48", "bf16-batch", "bf16-max", "f32-max",
                                  "bf16-bigB"])
def test_build_with_radix_select_matches_oracle(monkeypatch, name):
    """Top-W and Top-B by block radix select (instead of merge folds and
    bitonic sorts) give the same trees."""
    monkeypatch.setenv("DARTREE_RADIX", "1")
    test_build_matches_oracle_small([s[0] for s in SMALL].index(name))


@pytest.mark.parametrize("cap", ["0", "40"])
@pytest.mark.parametrize("name", ["bf16-n32", "bf16-n64", "bf16-batch", "f32-wide"])
def test_build_with_small_bound_key_buffers_matches_oracle(monkeypatch, name, cap):
    """The merge through the row bound with a small staging buffer: with none,
    every key of the lists that reach the bound is folded straight from
    memory (the path taken when more keys reach it than the buffer holds);
    with 40, rows with 6..40 keys at or above the bound are folded by all
    warps and a tree, rows with more straight from memory."""
    monkeypatch.setenv("DARTREE_MERGE_SURV_CAP", cap)
    test_build_matches_oracle_small([s[0] for s in SMALL].index(name))


@pytest.mark.parametrize("merge_bound", ["0", "1"])
def test_build_with_two_ctas_per_sm_merges_row_groups(monkeypatch, merge_bound):
    """Two head-call CTAs per SM: more than 160 CTA partials per row, so the
    per-row group merge runs in several group blocks and combines them; the
    merge through the row bound reads all pairs in one block per row."""
    monkeypatch.setenv("DARTREE_TC_CTAS_PER_SM", "2")
    monkeypatch.setenv("DARTREE_MERGE_BOUND", merge_bound)
    w = I.small_workload(590, V=30000, H=64, D=3, W=6, K=5, B=20, beta=-0.1, bf16=True)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx = gu.make_ctx(w)
    res = gu.run_build(ctx, w, dev)
    pool, rows, tree = gu.split_request(res, w, 0)
    rep = parity.compare_request(inp, 0, w.D, w.W, w.K, w.B, w.beta, w.bf16, pool, rows, tree,
                                 gpu_states=gu.request_states(res, w, 0))
    assert rep["near_ties"] <= 2
    ctx.close()


def test_two_runs_are_bit_identical():
    w = I.small_workload(7, V=2500, H=128, D=4, W=16, K=8, B=40, beta=-0.1, bf16=True, R=2)
    dev = dtl.weights_to_device(I.make_inputs(w), True)
    ctx = gu.make_ctx(w)
    a = gu.run_build(ctx, w, dev)
    b = gu.run_build(ctx, w, dev)
    for k in a["tree"]:
        assert np.array_equal(a["tree"][k], b["tree"][k]), k
    for k in a["pool"]:
        assert np.array_equal(a["pool"][k], b["pool"][k]), k
    ctx.close()


@pytest.mark.parametrize("bf16,M,K", [(True, 5, 8), (True, 16, 16), (True, 40, 4),
                                      (True, 65, 32), (True, 129, 1), (True, 200, 8),
                                      (True, 256, 32), (False, 3, 4), (False, 70, 9)])
def test_head_topk_matches_oracle_rows(bf16, M, K):
    w = I.small_workload(11 + M, V=2600, H=128 if bf16 else 96, D=1, W=1, K=K, B=1, bf16=bf16)
    inp = I.make_inputs(w)
    g = np.random.default_rng(M)
    S = np.tanh(g.standard_normal((M, w.H))).astype(np.float32)
    if bf16:
        S = I.bf16_bits_to_f32(I.to_bf16_bits(S))
    z = inp["z"][0, 0]
    ctx = gu.make_ctx(w, max_K=K)
    Wd = dtl.weights_to_device(inp, bf16)["Wout"]
    Sd = torch.from_numpy(I.to_bf16_bits(S)).view(torch.int16).cuda() if bf16 \
        else torch.from_numpy(S).cuda()
    out = ctx.head_topk(Sd, torch.from_numpy(z).cuda(), Wd, K=K)
    ctx.sync()
    tol = parity.TOL[bf16]
    for m in range(M):
        ell, lse = oracle.logits_row(z, inp["Wout"], S[m], bf16)
        tok, val, gap = oracle.topk_row(ell, K)
        assert abs(out["lse"][m].item() - lse) <= tol
        gt = out["tok"][m].cpu().numpy()
        if gap >= parity.NEAR_TIE:
            assert set(gt.tolist()) == set(tok.tolist())
        lp = out["logp"][m].cpu().numpy()
        ref = (ell[gt].astype(np.float64) - lse).astype(np.float32)
        assert np.max(np.abs(lp - ref)) <= tol
        assert np.all(np.diff(ell[gt]) <= parity.NEAR_TIE)
    ctx.close()


@pytest.mark.parametrize("mode", ["nv128", "nv256", "pair"])
@pytest.mark.parametrize("M,K", [(130, 8), (256, 3), (200, 16)])
def test_head_rows_tile_widths_match_oracle(monkeypatch, mode, M, K):
    """The row-major head kernel -- one CTA with 128- or 256-entry vocabulary
    tiles (the latter with one accumulator), or CTA pairs with the two-CTA
    MMA -- against the oracle rows."""
    monkeypatch.setenv("DARTREE_ROWS_PAIR", "1" if mode == "pair" else "0")
    monkeypatch.setenv("DARTREE_ROWS_NV", "256" if mode == "nv256" else "128")
    _check_head_rows(M, K, seed=M + len(mode))


@pytest.mark.parametrize("half", ["0", "1"])
@pytest.mark.parametrize("M,K", [(1, 4), (40, 32), (64, 8), (64, 17)])
def test_head_rows_with_at_most_64_rows_match_oracle(monkeypatch, half, M, K):
    """The one-CTA row-major kernel with 64-row state boxes (the other 64
    TMEM lanes hold whatever the stage held and are never read) or full
    128-row boxes."""
    monkeypatch.setenv("DARTREE_ROWS_MIN", "1")
    monkeypatch.setenv("DARTREE_ROWS_HALF_S", half)
    _check_head_rows(M, K, seed=1000 + M + int(half))


def _check_head_rows(M, K, seed):
    w = I.small_workload(60 + M + K, V=1900, H=192, D=1, W=1, K=K, B=1, bf16=True)
    inp = I.make_inputs(w)
    g = np.random.default_rng(seed)
    S = I.bf16_bits_to_f32(I.to_bf16_bits(np.tanh(g.standard_normal((M, w.H))).astype(np.float32)))
    z = inp["z"][0, 0]
    ctx = gu.make_ctx(w, max_K=K)
    Wd = dtl.weights_to_device(inp, True)["Wout"]
    Sd = torch.from_numpy(I.to_bf16_bits(S)).view(torch.int16).cuda()
    out = ctx.head_topk(Sd, torch.from_numpy(z).cuda(), Wd, K=K)
    ctx.sync()
    for m in range(M):
        ell, lse = oracle.logits_row(z, inp["Wout"], S[m], True)
        tok, _, gap = oracle.topk_row(ell, K)
        assert abs(out["lse"][m].item() - lse) <= parity.TOL[True]
        gt = out["tok"][m].cpu().numpy()
        if gap >= parity.NEAR_TIE:
            assert set(gt.tolist()) == set(tok.tolist())
        assert np.all(np.diff(ell[gt]) <= parity.NEAR_TIE)
    ctx.close()


@pytest.mark.parametrize("bf16,M", [(True, 7), (True, 64), (True, 256), (False, 5), (False, 33)])
def test_state_step_matches_oracle(bf16, M):
    H = 256 if bf16 else 64
    w = I.small_workload(21 + M, V=300, H=H, D=1, W=1, K=1, B=1, bf16=bf16)
    inp = I.make_inputs(w)
    g = np.random.default_rng(M)
    S = np.tanh(g.standard_normal((M, H))).astype(np.float32)
    if bf16:
        S = I.bf16_bits_to_f32(I.to_bf16_bits(S))
    tok = g.integers(0, w.V, M).astype(np.int32)
    dev = dtl.weights_to_device(inp, bf16)
    ctx = gu.make_ctx(w, max_W=256 if M > 1 else 1)
    Sd = torch.from_numpy(I.to_bf16_bits(S)).view(torch.int16).cuda() if bf16 \
        else torch.from_numpy(S).cuda()
    out = ctx.state_step(Sd, torch.from_numpy(tok).cuda(), dev["A"], dev["E"])
    ctx.sync()
    got = out.cpu()
    got = I.bf16_bits_to_f32(got.view(torch.int16).numpy().view(np.uint16)) if bf16 else got.numpy()
    flips = 0
    for m in range(M):
        ref = oracle.state_step(inp["A"], inp["E"], S[m], int(tok[m]), bf16)
        if bf16:
            # equal up to one bf16 rounding step: the fp32 accumulation (vs
            # fp64) and tanhf move u by ~1e-6 absolute, which can cross a bf16
            # rounding boundary; near zero that is more than one bf16 ulp, so
            # an absolute term bounds it there
            d = np.abs(got[m] - ref)
            ulp = np.spacing(np.abs(ref).astype(np.float32)) * 2 ** 16
            assert np.all(d <= ulp + 2e-5), (m, float(d.max()))
            flips += int(np.count_nonzero(d))
        else:
            assert np.max(np.abs(got[m] - ref)) <= 2e-6
    if bf16:
        assert flips <= 0.01 * M * H
    ctx.close()


@pytest.mark.parametrize("radix", ["0", "1"])
def test_prune_matches_oracle_bit_exact(monkeypatch, radix):
    monkeypatch.setenv("DARTREE_RADIX", radix)
    g = np.random.default_rng(3)
    R, D, W, K = 3, 6, 12, 4
    w = I.small_workload(31, V=200, H=64, D=D, W=W, K=K, B=64, bf16=True, R=R)
    ctx = gu.make_ctx(w, max_B=512)
    P = dtl.pool_size(D, W, K)
    # random pools with the construction's shape: parents in the previous depth
    sizes = dtl.frontier_sizes(D, W, K)
    par = np.empty((R, P), np.int32)
    dep = np.empty((R, P), np.int32)
    sco = np.empty((R, P), np.float32)
    for r in range(R):
        off_prev, off = 0, 0
        for d, fd in enumerate(sizes, 1):
            prev = sizes[d - 2] if d > 1 else 1
            p = -np.ones(fd, np.int32) if d == 1 else \
                (off_prev + g.integers(0, prev, fd)).astype(np.int32)
            par[r, off:off + fd] = p
            dep[r, off:off + fd] = d
            base = np.zeros(fd, np.float32) if d == 1 else sco[r, p]
            lp = -g.exponential(size=fd).astype(np.float32)
            lp[g.random(fd) < 0.2] = 0.0                      # exact ties
            sco[r, off:off + fd] = base + lp
            off_prev, off = off, off + fd
    tok = g.integers(0, 200, (R, P)).astype(np.int32)
    for B, beta in [(1, 0.0), (17, -0.1), (64, 0.0), (200, -2.0), (512, -0.3)]:
        out = ctx.prune(*(torch.from_numpy(a).cuda() for a in (par, tok, dep, sco)), B=B,
                        beta=beta)
        ctx.sync()
        for r in range(R):
            ref = oracle.topb(par[r], tok[r], dep[r], sco[r], B, beta)
            assert ref["rc"] == 0
            assert out["n_out"][r].item() == ref["n_out"]
            for k in ("parent", "token", "depth"):
                assert np.array_equal(out[k][r].cpu().numpy(), ref[k]), (B, k)
            assert np.array_equal(out["score"][r].cpu().numpy().view(np.uint32),
                                  ref["score"].view(np.uint32))
            assert np.array_equal(out["mask"][r].cpu().numpy().view(np.uint32), ref["mask"])
    ctx.close()


def test_invalid_arguments_are_rejected_before_launch():
    w = I.small_workload(41, V=500, H=64, D=3, W=4, K=4, B=8, bf16=True)
    dev = dtl.weights_to_device(I.make_inputs(w), True)
    ctx = gu.make_ctx(w)
    args = (dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"])
    for bad in [dict(beta=0.5), dict(K=5), dict(D=4), dict(B=0), dict(W=0)]:
        kw = dict(D=3, W=4, K=4, B=8, beta=0.0)
        kw.update(bad)
        with pytest.raises((dtl.DartreeError, ValueError)):
            ctx.build(*args, **kw)
    ctx.close()


def test_nonfinite_base_logits_raise_a_device_check():
    w = I.small_workload(42, V=500, H=64, D=3, W=4, K=4, B=8, bf16=True)
    inp = I.make_inputs(w)
    inp["z"][0, 1, 17] = np.nan
    dev = dtl.weights_to_device(inp, True)
    ctx = gu.make_ctx(w)
    ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], D=3, W=4, K=4, B=8,
              beta=0.0)
    assert ctx.sync_status() == 4      # DARTREE_ERR_DEVICE_CHECK
    assert ctx.sync_status() == 0      # the check word is cleared
    ctx.close()


def test_neg_inf_logits_are_allowed_and_ordered_by_token():
    # only 3 finite logits per depth, K = 5: the -inf tokens fill the list by id
    w = I.small_workload(43, V=300, H=64, D=2, W=5, K=5, B=10, bf16=True)
    inp = I.make_inputs(w, zero_wout=True)
    z = np.full_like(inp["z"], -np.inf)
    for t, v in ((10, 1.0), (20, 2.0), (30, 3.0)):
        z[0, :, t] = v
    inp["z"] = z
    dev = dtl.weights_to_device(inp, True)
    ctx = gu.make_ctx(w)
    res = gu.run_build(ctx, w, dev)
    r1 = res["rows"][0]
    assert list(r1["tok"][0]) == [30, 20, 10, 0, 1]
    assert np.isinf(r1["logp"][0][3:]).all()
    ctx.close()
