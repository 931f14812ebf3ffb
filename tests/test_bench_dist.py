"""Host logic of the multi-GPU bench path on CPU: world_size 2 over gloo.
The build shards by request (replicas, no data-path collective); the only
exchange is the max of the per-rank step time."""
from __future__ import annotations

import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.aggregate(2.0 + rank, world)          # ranks report 2 ms and 3 ms
    q.put((rank, ms, bench.job_value(ms, world, 32)))
    dist.destroy_process_group()


def test_step_time_is_the_max_over_ranks_and_value_counts_all_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 3.0
        assert abs(value - 2 * 32 * 1e3 / 3.0) < 1e-9


def test_single_rank_value():
    assert bench.aggregate(4.0, 1) == 4.0
    assert bench.job_value(4.0, 1, 1) == 250.0


def test_kernel_source_hash_follows_code_not_comments():
    """The profile captures stay valid across comment edits of the head
    kernels and are voided by any code edit."""
    a = "int f(int x) {  // one\n  /* two\n three */ return x + 1;\n}\n"
    b = "int f(int x) {\n  // a different comment\n  return x + 1;   /* more */\n}\n"
    c = "int f(int x) {  // one\n  return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert len(bench.kernel_source_hash()) == 16


def test_build_bytes_match_the_closed_forms():
    """Per-build algorithmic bytes D*V*H*wb + (D-1)*H*H*wb + gathered
    embedding rows + base logits, at the five workloads (GB)."""
    from speculative_decoding_draft_06_gb300 import inputs as I
    want = {"tiny": 0.2650, "q4b": 12.6535, "q8b": 20.4296, "batch": 20.7605, "wide": 20.4352}
    for name, gb in want.items():
        w = I.CONFIGS[name]
        wb = 2 if w.bf16 else 4
        closed = (w.D * w.V * w.H * wb + (w.D - 1) * w.H * w.H * wb
                  + sum(w.head_rows()[1:]) * w.H * wb + w.R * w.D * w.V * 4)
        assert bench.build_bytes(w) == closed, name
        assert abs(closed / 1e9 - gb) < 1e-3, name
    # launches per build: root, D head calls, D merges, D-1 two-kernel state
    # steps, prune; fp32 head calls of at most 16 rows carry the state step
    # (no launch), wider fp32 calls leave it to one kernel
    assert bench.kernels_per_build(I.CONFIGS["q8b"]) == 1 + 16 + 16 + 2 * 15 + 1
    assert bench.kernels_per_build(I.CONFIGS["tiny"]) == 1 + 8 + 8 + 0 + 1
    wide32 = I.CONFIGS["tiny"].replace(W=20)  # rows 1, 4, 16, 20, ...: depths 1-3 fold
    assert bench.kernels_per_build(wide32) == 1 + 8 + 8 + 4 + 1


def test_wout_layout_choice(monkeypatch):
    """bench.prepare_wout: auto takes the blocked layout except for the
    base-logit candidate variants (their gathered rows are contiguous only
    row-major); fp32 weights and `rows` keep the row-major matrix; the
    conversion runs once per weight set."""
    from speculative_decoding_draft_06_gb300 import dartree as dtl
    calls = []

    class Ctx:
        def set_weight_layout(self, layout):
            calls.append(layout)

    monkeypatch.setattr(dtl, "block_weights", lambda W: ("blocked", W))
    dev = {"Wout": "W"}
    assert bench.prepare_wout(Ctx(), dev, True, "auto", "dartree").startswith("blocks")
    assert dev["Wout"] == ("blocked", "W") and calls == ["blocks"]
    bench.prepare_wout(Ctx(), dev, True, "auto", "markov")
    assert dev["Wout"] == ("blocked", "W")          # not converted twice
    for bf16, layout, variant in ((True, "auto", "base"), (True, "auto", "markov-base"),
                                  (False, "blocks", "dartree"), (True, "rows", "dartree")):
        d = {"Wout": "W"}
        assert bench.prepare_wout(Ctx(), d, bf16, layout, variant) == "rows"
        assert d["Wout"] == "W"
