"""GPU parity of the build variants against the oracle (dartree_build_ex):
the Markov correction head, base-logit candidates and the sequential
best-first baseline, on small seeded workloads that span several vocabulary
tiles and a ragged tail."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import gpu_util as gu
from tests import parity

pytestmark = pytest.mark.gpu

DEPTHWISE = [
    dict(V=3000, H=128, D=4, W=6, K=4, B=20, beta=-0.2, bf16=True),
    dict(V=1237, H=64, D=5, W=5, K=3, B=17, beta=0.0, bf16=True, R=3),
    dict(V=2000, H=64, D=4, W=4, K=4, B=12, beta=-0.1, bf16=False),
    dict(V=20000, H=256, D=3, W=16, K=8, B=40, beta=-0.3, bf16=True, R=2),
]


def _build(w, dev, **variant):
    ctx = gu.make_ctx(w)
    s = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    for _ in range(2):  # capture, then a replay
        ctx.build(dev["z"], dev["state0"], None if variant.get("head") == "markov" else dev["A"],
                  dev["E"], dev["Wout"], D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta, out=out,
                  stream=s, **variant)
    ctx.sync(s)
    return ctx, out


@pytest.mark.parametrize("case", range(len(DEPTHWISE)))
@pytest.mark.parametrize("variant", [dict(head="markov"), dict(candidates="base"),
                                     dict(head="markov", candidates="base")])
def test_depthwise_variant_parity(case, variant):
    w = I.small_workload(800 + case, **DEPTHWISE[case])
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx, out = _build(w, dev, **variant)
    assert ctx.head_calls() == w.D
    P = w.pool_size()
    res = {"pool": {k: v.numpy() for k, v in ctx.get_pool(w.R, P).items()},
           "tree": {k: v.cpu().numpy() for k, v in out.items()}, "rows": [], "states": []}
    F = 1
    for d, fd in enumerate(w.frontier_sizes(), 1):
        res["rows"].append({k: v.numpy() for k, v in ctx.get_rows(d, w.R * F, w.K).items()})
        res["states"].append(ctx.get_states(d, w.R * F))
        F = fd
    ctx.close()
    markov = variant.get("head") == "markov"
    base = variant.get("candidates") == "base"
    for r in range(w.R):
        pool, rows, tree = gu.split_request(res, w, r)
        parity.compare_request(inp, r, w.D, w.W, w.K, w.B, w.beta, w.bf16, pool, rows, tree,
                               gpu_states=gu.request_states(res, w, r), markov=markov,
                               cand_base=base)


BESTFIRST = [
    dict(V=3000, H=128, D=4, W=1, K=4, B=20, beta=-0.2, bf16=True),
    dict(V=1237, H=64, D=3, W=1, K=3, B=30, beta=0.0, bf16=True, R=3),
    dict(V=2000, H=64, D=5, W=1, K=2, B=16, beta=-0.5, bf16=False, R=2),
    dict(V=500, H=64, D=2, W=1, K=3, B=16, beta=-0.1, bf16=True),   # tree smaller than B
]


@pytest.mark.parametrize("case", range(len(BESTFIRST)))
@pytest.mark.parametrize("head", ["recurrent", "markov"])
def test_bestfirst_parity(case, head):
    w = I.small_workload(850 + case, **BESTFIRST[case])
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx, out = _build(w, dev, head=head, expansion="bestfirst")
    assert ctx.head_calls() == w.B
    rows = [{k: v.numpy() for k, v in ctx.get_rows(c + 1, w.R, w.K).items()} for c in range(w.B)]
    states = [ctx.get_states(c + 1, w.R) for c in range(w.B)]
    tree = {k: v.cpu().numpy() for k, v in out.items()}
    ctx.close()
    for r in range(w.R):
        rep = parity.compare_bestfirst(
            inp, r, w.D, w.K, w.B, w.beta, w.bf16, {k: v[r] for k, v in tree.items()},
            [{k: v[r] for k, v in x.items()} for x in rows], [s[r] for s in states],
            markov=head == "markov")
        assert rep["calls"] >= 1


def test_variant_argument_errors():
    w = I.small_workload(870, V=1000, H=64, D=3, W=4, K=3, B=8, bf16=True)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, True)
    ctx = gu.make_ctx(w)
    kw = dict(D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta)
    with pytest.raises(dtl.DartreeError) as e:
        ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], candidates="base",
                  expansion="bestfirst", **kw)
    assert e.value.status == 2                       # UNSUPPORTED
    with pytest.raises(dtl.DartreeError) as e:       # the recurrent head needs A
        ctx.build(dev["z"], dev["state0"], None, dev["E"], dev["Wout"], **kw)
    assert e.value.status == 1
    ctx.build(dev["z"], dev["state0"], None, dev["E"], dev["Wout"], head="markov", **kw)
    ctx.sync()
    ctx.close()
