"""The blocked weight layout (DARTREE_LAYOUT_BLOCKS: Wout in blocks of 128
rows x 64 columns, each block one contiguous piece): dartree_block_weights
against a numpy restatement of the layout, and builds that read the blocked
projection against the same builds on the row-major one -- every state,
row result, pool entry and tree output bit for bit (the head call streams
the projection in exactly these blocks either way) -- for the default
build, the Markov head, base-logit candidates, the best-first baseline, the
unit head call and the full-size q8b build; a layout switch on a reused
buffer re-captures the build's graph."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def blocked_reference(W: np.ndarray) -> np.ndarray:
    """Block (b, k) = rows 128 b.., columns 64 k.. at element (b H/64 + k) 8192."""
    V, H = W.shape
    nb = -(-V // 128)
    P = np.zeros((nb * 128, H), W.dtype)
    P[:V] = W
    return P.reshape(nb, 128, H // 64, 64).transpose(0, 2, 1, 3).reshape(nb * 128, H)


@pytest.mark.parametrize("V,H", [(1000, 64), (1024, 128), (129, 256), (3001, 192)])
def test_block_weights_matches_the_layout(V, H):
    g = np.random.default_rng(V + H)
    W = g.integers(-32768, 32767, size=(V, H), dtype=np.int16)
    out = dtl.block_weights(torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    assert out.shape == (-(-V // 128) * 128, H)
    assert np.array_equal(out.cpu().numpy(), blocked_reference(W))
    assert dtl.load().dartree_blocked_weight_bytes(V, H) == out.numel() * 2


def _all_results(ctx, w, out):
    res = {"tree": {k: v.cpu().numpy() for k, v in out.items()},
           "pool": {k: v.numpy() for k, v in ctx.get_pool(w.R, w.pool_size()).items()}}
    F = 1
    for d, fd in enumerate(w.frontier_sizes(), 1):
        res[f"rows{d}"] = {k: v.numpy() for k, v in ctx.get_rows(d, w.R * F, w.K).items()}
        res[f"states{d}"] = {"s": np.asarray(ctx.get_states(d, w.R * F))}
        F = fd
    return res


def _build(w, dev, layout, variant=None, blocked=None):
    variant = variant or {}
    ctx = gu.make_ctx(w)
    ctx.set_weight_layout(layout)
    Wout = dev["Wout"] if layout == "rows" else (blocked if blocked is not None
                                                  else dtl.block_weights(dev["Wout"]))
    s = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    for _ in range(2):  # capture, then a replay
        ctx.build(dev["z"], dev["state0"], None if variant.get("head") == "markov" else dev["A"],
                  dev["E"], Wout, D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta, out=out, stream=s,
                  **variant)
    ctx.sync(s)
    if variant.get("expansion") == "bestfirst":
        res = {"tree": {k: v.cpu().numpy() for k, v in out.items()}}
        for c in range(w.B):
            res[f"rows{c}"] = {k: v.numpy() for k, v in ctx.get_rows(c + 1, w.R, w.K).items()}
            res[f"states{c}"] = {"s": np.asarray(ctx.get_states(c + 1, w.R))}
    else:
        res = _all_results(ctx, w, out)
    ctx.close()
    return res


def _same(a, b, what):
    assert a.keys() == b.keys()
    for part in a:
        for k in a[part]:
            assert np.array_equal(np.asarray(a[part][k]), np.asarray(b[part][k])), (what, part, k)


CASES = [
    ("n16", dict(V=3000, H=128, D=5, W=8, K=8, B=30, beta=0.0), {}),
    ("n64-rows", dict(V=1500, H=64, D=3, W=64, K=32, B=100, beta=-0.5), {}),
    ("pair-256", dict(V=1500, H=64, D=3, W=256, K=8, B=200, beta=-0.05), {}),
    ("ragged-batch", dict(V=1101, H=128, D=3, W=8, K=4, B=30, beta=-0.2, R=20), {}),
    ("markov", dict(V=3000, H=128, D=4, W=6, K=4, B=20, beta=-0.2), dict(head="markov")),
    ("base", dict(V=1237, H=64, D=5, W=5, K=3, B=17, beta=0.0, R=3), dict(candidates="base")),
    ("bestfirst", dict(V=3000, H=128, D=4, W=1, K=4, B=20, beta=-0.2), dict(expansion="bestfirst")),
]


@pytest.mark.parametrize("idx", range(len(CASES)), ids=[c[0] for c in CASES])
def test_blocked_build_bit_identical(idx):
    name, kw, variant = CASES[idx]
    w = I.small_workload(950 + idx, bf16=True, **kw)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    _same(_build(w, dev, "rows", variant), _build(w, dev, "blocks", variant), name)


def test_blocked_head_call_bit_identical():
    w = I.small_workload(960, V=2049, H=192, D=2, W=32, K=6, B=40, beta=0.0, bf16=True)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    g = np.random.default_rng(3)
    S = torch.from_numpy(I.to_bf16_bits(np.tanh(g.standard_normal((32, w.H))).astype(np.float32))
                         ).view(torch.int16).cuda()
    z = dev["z"][:, 0].contiguous()
    got = {}
    for layout in ("rows", "blocks"):
        ctx = gu.make_ctx(w)
        ctx.set_weight_layout(layout)
        Wout = dev["Wout"] if layout == "rows" else dtl.block_weights(dev["Wout"])
        r = ctx.head_topk(S, z, Wout, K=w.K, rows_per_req=32, z_req_stride=w.V)
        ctx.sync()
        got[layout] = {k: v.cpu().numpy() if torch.is_tensor(v) else np.asarray(v)
                       for k, v in r.items()}
        ctx.close()
    _same({"r": got["rows"]}, {"r": got["blocks"]}, "head_topk")


def test_layout_switch_on_a_reused_buffer_recaptures():
    """The same device buffer holds the row-major, then the blocked matrix
    (V a multiple of 128: the same size): the layout is part of the graph's
    key, so the second build re-encodes the projection's tensor map."""
    w = I.small_workload(961, V=2048, H=128, D=4, W=8, K=4, B=20, beta=0.0, bf16=True)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    buf = dev["Wout"].clone()
    blocked = dtl.block_weights(dev["Wout"])
    ctx = gu.make_ctx(w)
    s = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    trees = []
    for layout in ("rows", "blocks", "rows"):
        with torch.cuda.stream(s):
            buf.copy_(dev["Wout"] if layout == "rows" else blocked)
        ctx.set_weight_layout(layout)
        for _ in range(2):
            ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], buf, D=w.D, W=w.W, K=w.K,
                      B=w.B, beta=w.beta, out=out, stream=s)
        ctx.sync(s)
        trees.append({k: v.cpu().numpy() for k, v in out.items()})
    ctx.close()
    for t in trees[1:]:
        _same({"t": trees[0]}, {"t": t}, "switch")


def test_layout_errors():
    w = I.small_workload(962, V=1000, H=64, D=2, W=4, K=4, B=8, beta=0.0, bf16=False)
    ctx = gu.make_ctx(w)
    with pytest.raises(dtl.DartreeError, match="UNSUPPORTED"):
        ctx.set_weight_layout("blocks")
    assert dtl.load().dartree_set_weight_layout(ctx._h, 7) == 1  # INVALID_ARG
    ctx.close()
    assert dtl.load().dartree_blocked_weight_bytes(1000, 100) == 0
    with pytest.raises(ValueError):
        dtl.block_weights(torch.zeros(10, 100, dtype=torch.int16, device="cuda"))


def test_blocked_full_size_q8b():
    w = I.CONFIGS["q8b"]
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    _same(_build(w, dev, "rows"), _build(w, dev, "blocks"), "q8b")
