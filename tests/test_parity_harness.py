"""The GPU-vs-oracle comparison harness itself, on the CPU (no GPU).

The oracle's own build, fed in where a GPU build would be, must pass every
rule with no near-tie, through both the sequential and the sliced (process
pool) paths, and the two paths must see the same oracle values.  Planted
mistakes in the "GPU" side -- a dropped best candidate replaced by a
borderline one, a node kept twice, state steps off in more than 1 % of the
elements -- must be rejected.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import bruteforce as bf
from tests import parity
from tests.oracle_pool import OraclePool


def _oracle_as_gpu(w, inp):
    """One request's oracle build in the layout the GPU helpers return."""
    out = []
    for r in range(w.R):
        o = oracle.build_request(inp, r, w.D, w.W, w.K, w.B, w.beta, w.bf16)
        pool = {"parent": o["pool_parent"], "token": o["pool_token"], "depth": o["pool_depth"],
                "score": o["pool_score"]}
        rows, states, F, off = [], [], 1, 0
        cur = [bf.q(inp["state0"][r], w.bf16)]
        for d, fd in enumerate(w.frontier_sizes(), 1):
            rows.append({"lse": o["row_lse"][d - 1, :F], "tok": o["row_tok"][d - 1, :F],
                         "logp": o["row_logp"][d - 1, :F]})
            states.append(np.stack(cur).astype(np.float32))
            cur = [oracle.state_step(inp["A"], inp["E"], cur[o["own_slot"][off + q]],
                                     int(o["own_tok"][off + q]), w.bf16) for q in range(fd)]
            off += fd
            F = fd
        t = o["tree"]
        tree = {"parent": t["parent"], "token": t["token"], "depth": t["depth"],
                "score": t["score"], "mask": t["mask"], "n_out": t["n_out"]}
        out.append((pool, rows, tree, states))
    return out


W_SMALL = dict(V=300, H=32, D=4, W=6, K=3, B=12, beta=-0.1, bf16=True, R=2)


def test_oracle_build_passes_both_paths_exactly():
    w = I.small_workload(900, **W_SMALL)
    inp = I.make_inputs(w)
    reqs = _oracle_as_gpu(w, inp)
    with OraclePool(inp, procs=2) as pool:
        for r, (gp, rows, tree, states) in enumerate(reqs):
            a = parity.compare_request(inp, r, w.D, w.W, w.K, w.B, w.beta, True, gp, rows, tree,
                                       gpu_states=states)
            res = pool.run(parity.slice_tasks(r, w.D, w.W, w.K, True, gp, states))
            b = parity.compare_request_sliced(res, w.D, w.W, w.K, w.B, w.beta, True, gp, rows,
                                              tree, states)
            for rep in (a, b):
                assert rep["exact_depths"] == w.D and rep["near_ties"] == 0
                assert rep["max_score_err"] == 0 and rep["max_acc_score_err"] == 0
                assert rep["max_lse_err"] == 0 and rep["state_flips"] == 0
            # the slices see exactly what the sequential state-forced build sees
            o = oracle.build_tree(inp, r, w.D, w.W, w.K, True,
                                  force_state=np.stack([np.pad(s, ((0, w.W - len(s)), (0, 0)))
                                                        for s in states]))
            s = parity.assemble(res, w.D, w.W, w.K)
            for k in ("own_slot", "own_tok", "own_score", "pool_score", "pool_logp", "w_cut",
                      "row_tok", "row_logp"):
                assert np.array_equal(s[k], o[k], equal_nan=k.startswith("row")), k


def _fake_o(own, cut, margin, c_o):
    n = len(own)
    return {"own_slot": np.array([x[0] for x in own], np.int32),
            "own_tok": np.array([x[1] for x in own], np.int32),
            "own_score": np.array([x[2] for x in own], np.float32),
            "w_cut": np.array([[cut, cut - 1.0]], np.float32),
            "force_margin": np.full(n, margin, np.float32)}, np.array(c_o, np.float32)


ROWS = {"tok": np.array([[5, 7, 3], [2, 9, 4]], np.int32)}
OWN = [(0, 5, -1.0), (0, 7, -1.5), (1, 2, -2.0)]


def test_frontier_check_accepts_a_near_tie_swap():
    o, c_o = _fake_o(OWN, -2.0, 0.0, [-1.0, -1.5, -2.00005])
    parity._frontier_valid(1, 3, np.array([0, 0, 1]), np.array([5, 7, 9]), ROWS, o,
                           slice(0, 3), c_o)


def test_frontier_check_rejects_a_dropped_best_candidate():
    # keeps two nodes at the cut and drops the best one (score -1.0): margin,
    # cut and order alone would pass this
    o, c_o = _fake_o(OWN, -2.0, 0.0, [-1.5, -2.0, -2.00005])
    with pytest.raises(AssertionError, match="dropped"):
        parity._frontier_valid(1, 3, np.array([0, 1, 1]), np.array([7, 2, 9]), ROWS, o,
                               slice(0, 3), c_o)


def test_frontier_check_rejects_a_node_kept_twice():
    o, c_o = _fake_o(OWN, -2.0, 0.0, [-1.0, -1.0, -1.5])
    with pytest.raises(AssertionError, match="twice"):
        parity._frontier_valid(1, 3, np.array([0, 0, 0]), np.array([5, 5, 7]), ROWS, o,
                               slice(0, 3), c_o)


def test_frontier_check_allows_a_candidate_the_gpu_row_never_offered():
    # (0, 5) is above the cut but a counted top-K near-tie swapped token 5 out
    # of the GPU's row 0, which offers 8 instead
    rows = {"tok": np.array([[8, 7, 3], [2, 9, 4]], np.int32)}
    o, c_o = _fake_o(OWN, -2.0, 0.0, [-1.00002, -1.5, -2.0])
    parity._frontier_valid(1, 3, np.array([0, 0, 1]), np.array([8, 7, 2]), rows, o,
                           slice(0, 3), c_o)


def test_state_steps_off_in_many_elements_are_rejected():
    w = I.small_workload(901, **dict(W_SMALL, R=1))
    inp = I.make_inputs(w)
    gp, rows, tree, states = _oracle_as_gpu(w, inp)[0]
    bad = [s.copy() for s in states]
    for s in bad[1:]:                       # one bf16 step up in 5 % of the elements
        m = np.random.default_rng(0).random(s.shape) < 0.05
        s[m] = (s[m].view(np.uint32) + np.uint32(0x10000)).view(np.float32)
    with pytest.raises(AssertionError):
        parity.compare_request(inp, 0, w.D, w.W, w.K, w.B, w.beta, True, gp, rows, tree,
                               gpu_states=bad)
