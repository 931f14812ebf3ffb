"""CUDA-graph replay of a build: the captured launches re-read their inputs
and give the same bits as eager launches, and still match the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import gpu_util as gu
from tests import parity

pytestmark = pytest.mark.gpu


def _fetch(ctx, w, out):
    P = dtl.pool_size(w.D, w.W, w.K)
    return {"pool": {k: v.numpy() for k, v in ctx.get_pool(w.R, P).items()},
            "tree": {k: v.cpu().numpy() for k, v in out.items()}}


def test_graph_replay_reads_new_inputs_and_matches_eager():
    w = I.small_workload(61, V=2300, H=128, D=5, W=12, K=6, B=40, beta=-0.2, bf16=True, R=2)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, True)
    ctx = gu.make_ctx(w)
    s = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    args = (dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"])
    kw = dict(D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta, out=out, stream=s)
    ctx.build(*args, **kw)                       # captured and launched
    ctx.sync(s)
    first = _fetch(ctx, w, out)
    # new inputs in the same buffers, then a replay
    z2 = I.make_inputs(w.replace(seed=w.seed + 1))["z"]
    dev["z"].copy_(torch.from_numpy(z2))
    torch.cuda.synchronize()
    ctx.build(*args, **kw)
    ctx.sync(s)
    replay = _fetch(ctx, w, out)
    assert not np.array_equal(first["pool"]["token"], replay["pool"]["token"])
    # eager launches on the legacy stream from the same inputs
    eager_out = ctx.build(*args[:5], D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta)
    ctx.sync()
    eager = _fetch(ctx, w, eager_out)
    for part in ("pool", "tree"):
        for k in eager[part]:
            assert np.array_equal(eager[part][k], replay[part][k]), (part, k)
    # and the replayed build still matches the oracle
    inp["z"] = z2
    res = gu.run_build(ctx, w, dev)
    for r in range(w.R):
        pool, rows, tree = gu.split_request(res, w, r)
        parity.compare_request(inp, r, w.D, w.W, w.K, w.B, w.beta, True, pool, rows, tree)
    ctx.close()
