"""The host-buffer build (inputs copied in, the later depths' base logits on a
second stream under the head calls -- in one copy, or per depth when they
are large -- the tree copied out) gives the same trees as the device-buffer
build on the same inputs, bit for bit: with and without graph capture, and
on repeated calls (graph replay)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = [
    ("bf16-r3", dict(V=2100, H=128, D=4, W=8, K=6, B=24, beta=-0.1, bf16=True, R=3)),
    ("f32-r1", dict(V=1000, H=64, D=5, W=4, K=4, B=12, beta=0.0, bf16=False)),
    ("bf16-d1", dict(V=900, H=64, D=1, W=4, K=4, B=4, beta=0.0, bf16=True, R=2)),
    # 4 MB of base logits per depth: one copy and one event per depth
    ("bf16-big-z", dict(V=131072, H=64, D=4, W=4, K=4, B=12, beta=0.0, bf16=True, R=8)),
]


@pytest.mark.parametrize("graph", ["1", "0"])
@pytest.mark.parametrize("idx", range(len(CASES)), ids=[c[0] for c in CASES])
def test_build_host_matches_device_build(monkeypatch, idx, graph):
    monkeypatch.setenv("DARTREE_GRAPH", graph)
    name, kw = CASES[idx]
    w = I.small_workload(700 + idx, **kw)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx = gu.make_ctx(w)
    want = gu.run_build(ctx, w, dev)["tree"]
    zh = torch.from_numpy(inp["z"]).pin_memory()
    sh = torch.from_numpy(inp["state0"]).pin_memory()
    s = torch.cuda.Stream()
    for rep in range(3):  # capture, then replays
        oh = ctx.alloc_tree(w.R, w.B, device="cpu", pin=True)
        ctx.build_host(zh, sh, dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W, K=w.K, B=w.B,
                       beta=w.beta, out_host=oh, stream=s)
        for k, v in want.items():
            got = oh[k].numpy()
            assert np.array_equal(got, np.asarray(v)), (name, rep, k)
    ctx.close()


def test_build_host_sees_new_inputs_each_call():
    """The staging is refilled every call: a second call with other base
    logits (same host buffer, new contents) builds the other tree."""
    w = I.small_workload(710, V=1500, H=128, D=4, W=8, K=4, B=16, beta=0.0, bf16=True, R=2)
    inp = I.make_inputs(w)
    inp2 = I.make_inputs(w.replace(seed=w.seed + 1))
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx = gu.make_ctx(w)
    zh = torch.from_numpy(inp["z"].copy()).pin_memory()
    sh = torch.from_numpy(inp["state0"]).pin_memory()
    s = torch.cuda.Stream()
    trees = []
    for z in (inp["z"], inp2["z"], inp["z"]):
        zh.copy_(torch.from_numpy(z))
        oh = ctx.alloc_tree(w.R, w.B, device="cpu", pin=True)
        ctx.build_host(zh, sh, dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W, K=w.K, B=w.B,
                       beta=w.beta, out_host=oh, stream=s)
        trees.append({k: v.numpy().copy() for k, v in oh.items()})
    assert all(np.array_equal(trees[0][k], trees[2][k]) for k in trees[0])
    assert not all(np.array_equal(trees[0][k], trees[1][k]) for k in trees[0])
    ctx.close()
