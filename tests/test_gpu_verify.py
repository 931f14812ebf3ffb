"""GPU parity of the verification consumer: tree attention over prefix +
draft tree with the ancestor mask (dartree_tree_attention), the longest
accepted prefix (dartree_accept), and the whole verify step on a built tree
(attention -> output projection argmax -> acceptance)."""
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


def ancestor_mask(parent, n_out, B):
    """Mask rows of a canonical tree (test-side, from parent ranks)."""
    words = (B + 31) // 32
    m = np.zeros((B, words), np.uint32)
    for n in range(n_out):
        if parent[n] >= 0:
            m[n] = m[parent[n]]
        m[n, n // 32] |= np.uint32(1 << (n % 32))
    return m


def _cuda16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def attn_tol(Vp, Vt):
    """Softmax weights are rounded to bf16 (relative error <= 2^-9 each) and
    renormalised by their own sum, so each output is a convex combination of
    the visible values whose weights are within a factor 1 +- 2^-8 of the
    exact ones: |O - O_ref| <= 2^-8 max|v|, plus fp32 accumulation."""
    vmax = max(float(np.abs(I.bf16_bits_to_f32(Vp)).max(initial=0.0)),
               float(np.abs(I.bf16_bits_to_f32(Vt)).max(initial=0.0)))
    return 2.0 ** -8 * vmax * 1.01 + 1e-5


ATTN_CASES = [  # R, B, Lp, Hq, Hkv
    (1, 1, 0, 8, 8),
    (2, 7, 5, 4, 2),
    (1, 64, 100, 32, 8),
    (2, 130, 300, 8, 2),
    (1, 256, 64, 16, 4),
    (1, 40, 1000, 2, 1),
    (1, 40, 3000, 2, 1),      # long key ranges: the keys are split over CTAs
    (1, 130, 4000, 8, 2),
    (2, 16, 8000, 4, 2),
    (1, 50, 700, 12, 4),      # g = 3 and 6 do not divide a tile's 128 rows: the
    (1, 30, 2500, 6, 1),      # threads stage the query tile (else TMA boxes of nodes x heads)
]


@pytest.mark.parametrize("split", ["auto", "none", "2", "4", "5", "7", "8"])
@pytest.mark.parametrize("case", range(len(ATTN_CASES)))
def test_tree_attention_parity(monkeypatch, case, split):
    """The key splits: as the launch chooses them, none, or forced small
    split sizes (DARTREE_ATTN_SPLIT_MIN: key tiles per split at least), so
    that clusters of 2 to 8 CTAs exchange and combine their rows (the
    combine is instantiated per split count)."""
    if split == "none":
        monkeypatch.setenv("DARTREE_ATTN_SPLIT_MIN", "100000")
    elif split != "auto":
        monkeypatch.setenv("DARTREE_ATTN_SPLIT_MIN", "1")
        monkeypatch.setenv("DARTREE_ATTN_MAX_SPLIT", split)
    R, B, Lp, Hq, Hkv = ATTN_CASES[case]
    shape = I.VerifyShape(Lp=Lp, Hq=Hq, Hkv=Hkv, dh=128, seed=4000 + case)
    x = I.make_verify_inputs(R, B, shape)
    g = np.random.default_rng(case)
    trees = [I.random_tree(g, B, int(g.integers(max(1, B // 2), B + 1))) for _ in range(R)]
    masks = np.stack([ancestor_mask(t["parent"], t["n_out"], B) for t in trees])
    scale = 128 ** -0.5
    K, VT = dtl.kv_cache(*(_cuda16(x[k]) for k in ("Kp", "Vp", "Kt", "Vt")))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dtl.tree_attention(_cuda16(x["Q"]), K, VT,
                             torch.from_numpy(masks.view(np.int32)).cuda(), Lp=Lp, scale=scale,
                             err=err)
    assert int(err.item()) == 0                       # no pipeline wait ran out
    O = out["O"].cpu().numpy()
    O16 = out["O16"].cpu().numpy().view(np.uint16)
    assert np.array_equal(O16, I.to_bf16_bits(O))     # the bf16 copy is O rounded
    tol = attn_tol(x["Vp"], x["Vt"])
    for r in range(R):
        ref = oracle.tree_attention(x["Q"][r], x["Kp"][r], x["Vp"][r], x["Kt"][r], x["Vt"][r],
                                    masks[r], scale, True)
        err = np.abs(O[r] - ref)
        assert err.max() <= tol, (r, float(err.max()), tol)
        assert err.mean() <= tol / 8                  # typical errors are far below the bound


@pytest.mark.parametrize("seed", range(4))
def test_accept_parity(seed):
    g = np.random.default_rng(50 + seed)
    R, B = 3, 200
    trees = [I.random_tree(g, B, int(g.integers(1, B + 1))) for _ in range(R)]
    pred = np.empty((R, B + 1), np.int32)
    for r, t in enumerate(trees):
        for u in range(-1, B):
            kids = np.flatnonzero(t["parent"][:t["n_out"]] == u)
            pred[r, u + 1] = (t["token"][g.choice(kids)] if len(kids) and g.random() < 0.85
                              else 999999)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()  # noqa: E731
    got = dtl.accept(cu(np.stack([t["parent"] for t in trees])),
                     cu(np.stack([t["token"] for t in trees])),
                     cu(np.array([t["n_out"] for t in trees])), cu(pred), max_len=B)
    ln, nodes, bonus = (got[k].cpu().numpy() for k in ("len", "nodes", "bonus"))
    for r, t in enumerate(trees):
        ref = oracle.accept(t["parent"], t["token"], t["n_out"], pred[r])
        assert ln[r] == ref["len"] and bonus[r] == ref["bonus"]
        assert np.array_equal(nodes[r, :ln[r]], ref["nodes"]) and np.all(nodes[r, ln[r]:] == -1)


def test_verify_step_on_a_built_tree():
    """Build a tree, run the target layer with its mask, take the target's
    greedy tokens through an output projection (the head-call kernel with
    K = 1 and zero base logits) and accept -- each stage against the oracle
    on the GPU's own inputs to that stage."""
    w = I.small_workload(890, V=3000, H=128, D=4, W=6, K=4, B=24, beta=-0.2, bf16=True)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, True)
    ctx = gu.make_ctx(w)
    tree = ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W,
                     K=w.K, B=w.B, beta=w.beta)
    ctx.sync()
    ctx.close()
    t = {k: v.cpu().numpy() for k, v in tree.items()}
    shape = I.VerifyShape(Lp=77, Hq=8, Hkv=2, dh=128, seed=4100)
    x = I.make_verify_inputs(1, w.B, shape)
    K, VT = dtl.kv_cache(*(_cuda16(x[k]) for k in ("Kp", "Vp", "Kt", "Vt")))
    out = dtl.tree_attention(_cuda16(x["Q"]), K, VT, tree["mask"], Lp=shape.Lp,
                             scale=128 ** -0.5)
    mask = t["mask"][0].view(np.uint32)
    ref = oracle.tree_attention(x["Q"][0], x["Kp"][0], x["Vp"][0], x["Kt"][0], x["Vt"][0], mask,
                                128 ** -0.5, True)
    assert np.abs(out["O"].cpu().numpy()[0] - ref).max() <= attn_tol(x["Vp"], x["Vt"])
    # the target's output projection: U [V, Hq*dh], greedy token per row
    H2 = shape.Hq * shape.dh
    U = I.make_inputs(w.replace(H=H2, D=1, seed=w.seed + 1))["Wout"]
    tgt = dtl.DARTree(w.V, H2, max_D=1, max_W=w.B + 1, max_K=1, max_B=1, bf16=True)
    S = out["O16"].reshape(w.B + 1, H2).contiguous()
    zero = torch.zeros(w.V, dtype=torch.float32, device="cuda")
    Ud = torch.from_numpy(U.view(np.int16)).cuda()
    rows = tgt.head_topk(S, zero, Ud, K=1)
    torch.cuda.synchronize()
    tgt.close()
    pred = rows["tok"].cpu().numpy()[:, 0].astype(np.int32)
    S_h = I.bf16_bits_to_f32(S.cpu().numpy().view(np.uint16))
    for i in range(w.B + 1):
        ell, _ = oracle.logits_row(np.zeros(w.V, np.float32), U, S_h[i], True)
        tk, _, gap = oracle.topk_row(ell, 1)
        assert pred[i] == tk[0] or gap < parity.NEAR_TIE, (i, pred[i], tk[0], gap)
    # acceptance on the GPU's predictions, bit-exact
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()  # noqa: E731
    acc = dtl.accept(tree["parent"], tree["token"], tree["n_out"], cu(pred[None]), max_len=w.D)
    r = oracle.accept(t["parent"][0], t["token"][0], int(t["n_out"][0]), pred)
    assert int(acc["len"][0]) == r["len"] and int(acc["bonus"][0]) == r["bonus"]
    assert np.array_equal(acc["nodes"][0, :r["len"]].cpu().numpy(), r["nodes"])
