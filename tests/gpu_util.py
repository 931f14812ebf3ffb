"""Helpers for the GPU tests: run a build through the C ABI and fetch its
pool, per-depth rows and trees as numpy arrays."""
from __future__ import annotations

import numpy as np
import torch

from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300.inputs import Workload


def make_ctx(w: Workload, **over) -> dtl.DARTree:
    kw = dict(max_D=w.D, max_W=w.W, max_K=w.K, max_B=w.B, max_requests=w.R, bf16=w.bf16)
    kw.update(over)
    return dtl.DARTree(w.V, w.H, **kw)


def run_build(ctx: dtl.DARTree, w: Workload, dev: dict) -> dict:
    out = ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W,
                    K=w.K, B=w.B, beta=w.beta)
    ctx.sync()
    P = dtl.pool_size(w.D, w.W, w.K)
    pool = ctx.get_pool(w.R, P)
    rows, states = [], []
    F = 1
    for d, fd in enumerate(dtl.frontier_sizes(w.D, w.W, w.K), start=1):
        rows.append({k: v.numpy() for k, v in ctx.get_rows(d, w.R * F, w.K).items()})
        states.append(ctx.get_states(d, w.R * F))
        F = fd
    tree = {k: v.cpu().numpy() for k, v in out.items()}
    return {"pool": {k: v.numpy() for k, v in pool.items()}, "rows": rows, "tree": tree,
            "states": states, "head_calls": ctx.head_calls()}


def split_request(res: dict, w: Workload, r: int):
    """Per-request views: pool [P], rows per depth [F_{d-1}], tree."""
    pool = {k: v[r] for k, v in res["pool"].items()}
    rows, F = [], 1
    for d, fd in enumerate(dtl.frontier_sizes(w.D, w.W, w.K), start=1):
        x = res["rows"][d - 1]
        rows.append({"lse": x["lse"][r * F:(r + 1) * F], "tok": x["tok"][r * F:(r + 1) * F],
                     "logp": x["logp"][r * F:(r + 1) * F]})
        F = fd
    tree = {k: v[r] for k, v in res["tree"].items()}
    return pool, rows, tree


def request_states(res: dict, w: Workload, r: int) -> list:
    """Per-depth head states of request r ([F_{d-1}, H] each)."""
    out, F = [], 1
    for d, fd in enumerate(dtl.frontier_sizes(w.D, w.W, w.K), start=1):
        out.append(res["states"][d - 1][r * F:(r + 1) * F])
        F = fd
    return out


def cuda_ok() -> bool:
    return torch.cuda.is_available()
