"""Runs the CPU oracle on many independent depth slices at once -- TEST
INFRASTRUCTURE ONLY.

A full-size build has hundreds to thousands of head rows, each a
full-vocabulary fp64 pass of the single-threaded oracle (about 0.4 s at
V = 151936, H = 4096).  With the GPU's head states and frontier given, every
(request, depth) slice of the comparison is independent, so a process pool
spreads the slices over the host's cores.  Workers are started with
``spawn`` (never forked from a process that has touched CUDA) and map the
workload's arrays read-only from ``.npy`` files in a temporary directory.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

_G: dict = {}


def _init(path: str) -> None:
    for k in ("z", "Wout", "A", "E"):
        f = os.path.join(path, k + ".npy")
        if os.path.exists(f):
            _G[k] = np.load(f, mmap_mode="r")


def _run_slice(t: dict) -> dict:
    import oracle
    o = oracle.depth(_G["z"][t["r"], t["d"] - 1], _G["Wout"], t["states"], t["score"], t["W"],
                     t["K"], t["bf16"], force_slot=t["force_slot"], force_tok=t["force_tok"],
                     cand_base=t["cand_base"])
    if "step_parent" in t:
        A = None if t["markov"] else _G["A"]
        o["step_states"] = np.stack([
            oracle.state_step(A, _G["E"], t["step_parent"][s], int(tk), t["bf16"])
            for s, tk in zip(t["step_slot"].tolist(), t["step_tok"].tolist())])
    return o


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """``with OraclePool(inp) as p: results = p.run(tasks)``; results come
    back in task order."""

    def __init__(self, inp: dict, procs: int | None = None):
        self.tmp = tempfile.mkdtemp(prefix="dartree_oracle_")
        for k in ("z", "Wout", "A", "E"):
            if inp.get(k) is not None:
                np.save(os.path.join(self.tmp, k + ".npy"), np.ascontiguousarray(inp[k]))
        self.procs = procs or host_cores()
        self.pool = mp.get_context("spawn").Pool(self.procs, initializer=_init,
                                                 initargs=(self.tmp,))

    def run(self, tasks: list) -> list:
        # the largest slices first, so that the pool's tail is short
        order = sorted(range(len(tasks)), key=lambda i: -tasks[i]["states"].shape[0])
        done = self.pool.map(_run_slice, [tasks[i] for i in order], chunksize=1)
        out = [None] * len(tasks)
        for i, r in zip(order, done):
            out[i] = r
        return out

    def close(self) -> None:
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
            self.pool = None
        shutil.rmtree(self.tmp, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False
