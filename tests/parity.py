"""GPU-vs-oracle comparison rules for supertree builds.

Structure (token ids, parents, masks) must match bit for bit, except at
near-ties: where the oracle's own deciding gap is below NEAR_TIE (1e-4) a
different GPU choice is counted and reported, and the comparison continues
from the GPU's choice (teacher forcing), so one flip cannot cascade.  A
differing choice is accepted only when it is a valid one: every candidate the
oracle ranks clearly above the cut is kept, the kept nodes are distinct, and
each kept node is within NEAR_TIE of the cut and of its row's K-th child.
Scores must agree within the dtype's tolerance: 2e-3 absolute with bf16
weights, 1e-5 with fp32 weights.

Two ways to get the oracle's side of one request:
  * ``compare_request``: the oracle's own depth-by-depth build along the
    GPU's frontier (sequential, one process);
  * ``compare_request_sliced``: every depth replayed on its own from the
    GPU's head states and the GPU's previous-frontier scores (independent
    slices that a process pool spreads over the host's cores; see
    ``tests/oracle_pool.py``).  The scores it compares per depth are the
    GPU's parent score plus the oracle's log-prob; the oracle's own
    accumulated scores along the same paths are checked as well.
"""
from __future__ import annotations

import numpy as np

import oracle

NEAR_TIE = 1e-4
TOL = {True: 2e-3, False: 1e-5}
MAX_STATE_FLIP_FRAC = 0.01   # bf16 state elements off by one rounding step


def frontier_sizes(D: int, W: int, K: int) -> list:
    sizes, f = [], 1
    for _ in range(D):
        f = min(W, K * f)
        sizes.append(f)
    return sizes


def forced_frontier(pool: dict, D: int, W: int, K: int):
    """GPU pool of one request -> (parent slot, token) per node, pool layout."""
    sizes = frontier_sizes(D, W, K)
    slot = np.empty(sum(sizes), np.int32)
    off_prev, off = 0, 0
    for d, fd in enumerate(sizes, start=1):
        par = pool["parent"][off:off + fd]
        if d == 1:
            assert np.all(par == -1), "depth-1 parents must be -1"
            slot[off:off + fd] = 0
        else:
            s = par - off_prev
            prev = sizes[d - 2]
            assert np.all((s >= 0) & (s < prev)), "parent outside previous depth"
            slot[off:off + fd] = s
        assert np.all(pool["depth"][off:off + fd] == d)
        off_prev, off = off, off + fd
    return slot, np.ascontiguousarray(pool["token"], np.int32), sizes


def state_diff_ok(got: np.ndarray, ref: np.ndarray, bf16: bool, where) -> int:
    """One state row against the oracle's: equal up to one bf16 rounding step
    (+2e-5 absolute near zero) with bf16 weights, 2e-6 with fp32.  Returns the
    number of differing elements."""
    dif = np.abs(got - ref)
    if bf16:
        ulp = np.spacing(np.abs(ref).astype(np.float32)) * 2 ** 16
        assert np.all(dif <= ulp + 2e-5), (where, float(dif.max()))
    else:
        assert np.all(dif <= 2e-6), (where, float(dif.max()))
    return int(np.count_nonzero(dif))


def check_state_steps(inp: dict, bf16: bool, slot, tok, sizes, gpu_states: list,
                      max_rows: int | None = None, markov: bool = False) -> tuple:
    """Each GPU head state of depth >= 2 against the oracle's state step
    applied to the GPU's own parent state and token.  Returns (differing
    elements, elements checked)."""
    flips, n_el, off = 0, 0, sizes[0]
    for d in range(2, len(gpu_states) + 1):
        fd = sizes[d - 2]                       # rows of call d = nodes of depth d-1
        base = off - fd
        n = fd if max_rows is None else min(fd, max_rows)
        for i in range(n):
            par = gpu_states[d - 2][slot[base + i]]
            ref = oracle.state_step(None if markov else inp["A"], inp["E"], par,
                                    int(tok[base + i]), bf16)
            flips += state_diff_ok(gpu_states[d - 1][i], ref, bf16, (d, i))
            n_el += ref.size
        off += sizes[d - 1] if d - 1 < len(sizes) else 0
    return flips, n_el


def _rows_match(d: int, F: int, rows: dict, o: dict, tol: float, rep: dict) -> None:
    """The GPU's per-row head results of depth d against the oracle's."""
    for i in range(F):
        lse_err = abs(rows["lse"][i] - o["row_lse"][d - 1, i])
        rep["max_lse_err"] = max(rep["max_lse_err"], lse_err)
        assert lse_err <= tol, f"depth {d} row {i}: lse {rows['lse'][i]} vs {o['row_lse'][d-1, i]}"
        gt, ot = rows["tok"][i], o["row_tok"][d - 1, i]
        olp = {int(t): float(v) for t, v in zip(ot, o["row_logp"][d - 1, i])}
        if set(gt.tolist()) != set(olp):
            # only a near-tie at the K-th / (K+1)-th boundary may swap members
            kg = o["row_kgap"][d - 1, i]
            assert kg < NEAR_TIE and len(set(gt.tolist()) - set(olp)) == 1, \
                f"depth {d} row {i}: top-K {gt} vs {ot} (gap {kg})"
            rep["topk_near_ties"] += 1
        common = [(j, int(t)) for j, t in enumerate(gt) if int(t) in olp]
        vals = [olp[t] for _, t in common]
        assert np.all(np.diff(vals) <= NEAR_TIE), f"depth {d} row {i}: order {gt} vs {ot}"
        if not np.array_equal(gt, ot) and set(gt.tolist()) == set(olp):
            rep["topk_near_ties"] += 1
        e = max((abs(float(rows["logp"][i][j]) - olp[t]) for j, t in common), default=0.0)
        rep["max_logp_err"] = max(rep["max_logp_err"], e)
        assert e <= tol, f"depth {d} row {i}: logp err {e}"


def _frontier_valid(d: int, fd: int, g_slot, g_tok, rows: dict, o: dict, sl: slice,
                    c_o: np.ndarray) -> None:
    """A GPU frontier that differs from the oracle's own top-W is accepted
    only as a valid choice among near-ties:
      (i)   every oracle candidate scoring above the W-th cut + NEAR_TIE is
            kept (unless a counted top-K near-tie took its token out of the
            GPU row, which then offered the swapped-in token instead);
      (ii)  the kept (slot, token) pairs are distinct;
      (iii) there are exactly |F_d| of them;
      (iv)  each kept node is within NEAR_TIE of its row's K-th child and of
            the oracle's W-th cut, and the kept scores are in rank order."""
    pairs = list(zip(g_slot.tolist(), g_tok.tolist()))
    assert len(pairs) == fd, f"depth {d}: {len(pairs)} kept nodes, |F_d| = {fd}"
    assert len(set(pairs)) == fd, f"depth {d}: a (slot, token) pair is kept twice"
    kept = set(pairs)
    wth = float(o["w_cut"][d - 1, 0])
    own = zip(o["own_slot"][sl].tolist(), o["own_tok"][sl].tolist(),
              o["own_score"][sl].tolist())
    for s_, t_, c_ in own:
        if c_ > wth + NEAR_TIE and (s_, t_) not in kept:
            offered = int(t_) in set(rows["tok"][s_].tolist())
            assert not offered, (f"depth {d}: candidate (slot {s_}, token {t_}, score {c_}) "
                                 f"above the cut {wth} was dropped")
    ok_topk = np.all(o["force_margin"][sl] >= -NEAR_TIE)
    ok_cut = np.all(c_o >= wth - NEAR_TIE)
    ok_order = np.all(np.diff(c_o) <= NEAR_TIE)
    assert ok_topk and ok_cut and ok_order, (
        f"depth {d}: GPU frontier differs beyond near-ties "
        f"(topk {ok_topk}, cut {ok_cut}, order {ok_order})")


def compare_with(o: dict, D: int, W: int, K: int, B: int, beta: float, bf16: bool,
                 gpu_pool: dict, gpu_rows: list, gpu_tree: dict) -> dict:
    """Compare one request's GPU results with the oracle's results ``o``
    (per-depth rows, own top-W, scores of the GPU's kept nodes, log-probs,
    cuts; laid out as ``oracle.build_tree`` returns them)."""
    tol = TOL[bf16]
    slot, tok, sizes = forced_frontier(gpu_pool, D, W, K)
    rep = {"near_ties": 0, "exact_depths": 0, "max_score_err": 0.0, "max_lse_err": 0.0,
           "max_logp_err": 0.0, "topk_near_ties": 0, "max_acc_score_err": 0.0}
    off, F = 0, 1
    for d in range(1, D + 1):
        fd = sizes[d - 1]
        sl = slice(off, off + fd)
        rows = gpu_rows[d - 1]
        _rows_match(d, F, rows, o, tol, rep)
        # --- kept frontier
        g_slot, g_tok = slot[sl], tok[sl]
        c_o = o["pool_score"][sl]               # oracle's score of the GPU's nodes
        err = float(np.max(np.abs(gpu_pool["score"][sl] - c_o)))
        rep["max_score_err"] = max(rep["max_score_err"], err)
        assert err <= tol, f"depth {d}: score err {err}"
        if np.array_equal(g_slot, o["own_slot"][sl]) and np.array_equal(g_tok, o["own_tok"][sl]):
            rep["exact_depths"] += 1
        else:
            _frontier_valid(d, fd, g_slot, g_tok, rows, o, sl, c_o)
            rep["near_ties"] += 1
        off += fd
        F = fd
    # --- the oracle's accumulated scores along the GPU's paths
    acc = oracle.path_scores(gpu_pool["parent"], o["pool_logp"])
    err = float(np.max(np.abs(gpu_pool["score"] - acc)))
    rep["max_acc_score_err"] = err
    assert err <= tol, f"accumulated score err {err}"
    # --- deferred Top-B: a pure function of the pool -> bit-exact
    ref = oracle.topb(gpu_pool["parent"], gpu_pool["token"], gpu_pool["depth"],
                      gpu_pool["score"], B, beta)
    assert ref["rc"] == 0
    n = ref["n_out"]
    assert int(gpu_tree["n_out"]) == n
    for k in ("parent", "token", "depth"):
        assert np.array_equal(gpu_tree[k], ref[k]), k
    assert np.array_equal(gpu_tree["score"].view(np.uint32), ref["score"].view(np.uint32))
    assert np.array_equal(gpu_tree["mask"].reshape(ref["mask"].shape).view(np.uint32),
                          ref["mask"])
    # Lemma 1 on the GPU's pool
    heap = oracle.heap_prune(gpu_pool["parent"], gpu_pool["depth"], gpu_pool["score"], B, beta)
    assert np.array_equal(ref["order"][:n], heap)
    return rep


def compare_request(inp: dict, r: int, D: int, W: int, K: int, B: int, beta: float,
                    bf16: bool, gpu_pool: dict, gpu_rows: list, gpu_tree: dict,
                    gpu_states: list | None = None, markov: bool = False,
                    cand_base: bool = False) -> dict:
    """Teacher-forced comparison of one request.  Raises AssertionError on a
    mismatch that no near-tie explains; returns counters otherwise.  With
    gpu_states (per depth [F_{d-1}, H] fp32), every head call is compared on
    the GPU's own states and every state step is checked separately (with bf16
    weights at most 1 % of the state elements may differ, each by one rounding
    step; with fp32 every element within 2e-6);
    without, the oracle runs its own states along the GPU's frontier.
    ``markov`` / ``cand_base`` select the build variant."""
    slot, tok, sizes = forced_frontier(gpu_pool, D, W, K)
    fst = None
    if gpu_states is not None:
        H = inp["E"].shape[1]
        fst = np.zeros((D, W, H), np.float32)
        for d, s in enumerate(gpu_states):
            fst[d, :s.shape[0]] = s
    o = oracle.build_tree(inp, r, D, W, K, bf16, force_slot=slot, force_tok=tok,
                          force_state=fst, markov=markov, cand_base=cand_base)
    rep = compare_with(o, D, W, K, B, beta, bf16, gpu_pool, gpu_rows, gpu_tree)
    if gpu_states is not None:
        flips, n_el = check_state_steps(inp, bf16, slot, tok, sizes, gpu_states, markov=markov)
        rep["state_flips"] = flips
        rep["state_elems"] = n_el
        if bf16:       # (fp32 states differ in their last bits almost everywhere)
            assert flips <= MAX_STATE_FLIP_FRAC * max(1, n_el), (flips, n_el)
    return rep


def slice_tasks(r: int, D: int, W: int, K: int, bf16: bool, gpu_pool: dict, gpu_states: list,
                cand_base: bool = False, states=None, markov: bool = False) -> list:
    """Independent oracle tasks, one per depth of request r: the depth's head
    call from the given head states (the GPU's unless ``states`` is given) and
    the GPU's previous-frontier scores, scoring the GPU's kept frontier; and
    for d >= 2 the state step of each row from its GPU parent state."""
    slot, tok, sizes = forced_frontier(gpu_pool, D, W, K)
    st = gpu_states if states is None else states
    tasks, off, F, prev = [], 0, 1, np.zeros(1, np.float32)
    for d in range(1, D + 1):
        fd = sizes[d - 1]
        t = {"r": r, "d": d, "W": W, "K": K, "bf16": bf16, "cand_base": cand_base,
             "states": np.ascontiguousarray(st[d - 1][:F], np.float32), "score": prev,
             "force_slot": slot[off:off + fd].copy(), "force_tok": tok[off:off + fd].copy()}
        if d >= 2 and states is None:
            base = off - F                       # the F nodes of depth d-1
            t["step_parent"] = np.ascontiguousarray(gpu_states[d - 2], np.float32)
            t["step_slot"] = slot[base:base + F].copy()
            t["step_tok"] = tok[base:base + F].copy()
            t["markov"] = markov
        tasks.append(t)
        prev = np.ascontiguousarray(gpu_pool["score"][off:off + fd], np.float32)
        off += fd
        F = fd
    return tasks


def assemble(results: list, D: int, W: int, K: int) -> dict:
    """Per-depth slice results (in depth order) -> the layout of
    ``oracle.build_tree``."""
    sizes = frontier_sizes(D, W, K)
    P = sum(sizes)
    o = {k: np.empty(P, np.int32) for k in ("own_slot", "own_tok")}
    o.update({k: np.empty(P, np.float32) for k in
              ("own_score", "pool_score", "pool_logp", "force_margin")})
    o["row_lse"] = np.full((D, W), np.nan, np.float64)
    o["row_tok"] = np.full((D, W, K), -1, np.int32)
    o["row_logp"] = np.full((D, W, K), np.nan, np.float32)
    o["row_kgap"] = np.full((D, W), np.nan, np.float32)
    o["w_cut"] = np.empty((D, 2), np.float32)
    off, F = 0, 1
    for d in range(1, D + 1):
        x = results[d - 1]
        fd = sizes[d - 1]
        sl = slice(off, off + fd)
        for k in ("own_slot", "own_tok", "own_score", "force_margin"):
            o[k][sl] = x[k]
        o["pool_score"][sl] = x["sel_score"]
        o["pool_logp"][sl] = x["sel_logp"]
        o["row_lse"][d - 1, :F] = x["row_lse"]
        o["row_tok"][d - 1, :F] = x["row_tok"]
        o["row_logp"][d - 1, :F] = x["row_logp"]
        o["row_kgap"][d - 1, :F] = x["row_kgap"]
        o["w_cut"][d - 1] = x["w_cut"]
        off += fd
        F = fd
    return o


def compare_request_sliced(results: list, D: int, W: int, K: int, B: int, beta: float,
                           bf16: bool, gpu_pool: dict, gpu_rows: list, gpu_tree: dict,
                           gpu_states: list) -> dict:
    """Teacher- and state-forced comparison of one request from per-depth
    oracle slices (``slice_tasks`` run by ``tests/oracle_pool.py``).  Same
    rules as ``compare_request`` with gpu_states; the per-depth scores are the
    GPU's parent score plus the oracle's log-prob, and the oracle's own
    accumulated scores along the GPU's paths must also be within tolerance."""
    o = assemble(results, D, W, K)
    rep = compare_with(o, D, W, K, B, beta, bf16, gpu_pool, gpu_rows, gpu_tree)
    flips = n_el = 0
    for d in range(2, D + 1):
        ref = results[d - 1]["step_states"]
        for i in range(ref.shape[0]):
            flips += state_diff_ok(gpu_states[d - 1][i], ref[i], bf16, (d, i))
            n_el += ref[i].size
    rep["state_flips"] = flips
    rep["state_elems"] = n_el
    if bf16:
        assert flips <= MAX_STATE_FLIP_FRAC * max(1, n_el), (flips, n_el)
    return rep


def compare_bestfirst(inp: dict, r: int, D: int, K: int, B: int, beta: float, bf16: bool,
                      gpu_tree: dict, gpu_rows: list, gpu_states: list,
                      markov: bool = False) -> dict:
    """Teacher-forced comparison of a best-first build of request r.

    gpu_rows[c] / gpu_states[c] are head call c's row ({lse, tok, logp}) and
    state ([H] fp32).  The oracle replays the build with the GPU's children
    and states, so the tree (pops, parents, scores, mask) must then match
    bit for bit; each call the oracle makes is compared with the GPU's row
    (near-ties at the K-th child allowed) and each state with the oracle's
    state step from the GPU's parent state."""
    tol = TOL[bf16]
    ft = np.stack([x["tok"] for x in gpu_rows]).astype(np.int32)
    fl = np.stack([x["logp"] for x in gpu_rows]).astype(np.float32)
    fs = np.stack(gpu_states).astype(np.float32)
    o = oracle.bestfirst(inp, r, D, K, B, beta, bf16, markov=markov, force_tok=ft,
                         force_logp=fl, force_state=fs)
    n = int(gpu_tree["n_out"])
    assert n == o["n_out"], (n, o["n_out"])
    for k in ("parent", "token", "depth"):
        assert np.array_equal(gpu_tree[k], o[k]), k
    assert np.array_equal(gpu_tree["score"].view(np.uint32), o["score"].view(np.uint32))
    assert np.array_equal(gpu_tree["mask"].reshape(o["mask"].shape).view(np.uint32), o["mask"])
    rep = {"calls": o["calls"], "topk_near_ties": 0, "max_lse_err": 0.0, "max_logp_err": 0.0}
    for c in range(B):
        if o["call_rank"][c] < -1:
            continue                               # a call whose result is unused
        g = gpu_rows[c]
        err = abs(float(g["lse"]) - o["row_lse"][c])
        rep["max_lse_err"] = max(rep["max_lse_err"], err)
        assert err <= tol, (c, float(g["lse"]), o["row_lse"][c])
        olp = {int(t): float(v) for t, v in zip(o["row_tok"][c], o["row_logp"][c])}
        if set(g["tok"].tolist()) != set(olp):
            assert o["row_kgap"][c] < NEAR_TIE and len(set(g["tok"].tolist()) - set(olp)) == 1, c
            rep["topk_near_ties"] += 1
        e = max((abs(float(lp) - olp[int(t)]) for t, lp in zip(g["tok"], g["logp"])
                 if int(t) in olp), default=0.0)
        rep["max_logp_err"] = max(rep["max_logp_err"], e)
        assert e <= tol, (c, e)
        if c >= 1:                                 # the state of rank c-1
            q = c - 1
            pr = int(o["parent"][q])
            par = gpu_states[0] if pr < 0 else gpu_states[pr + 1]
            ref = oracle.state_step(None if markov else inp["A"], inp["E"], par,
                                    int(o["token"][q]), bf16)
            dif = np.abs(gpu_states[c] - ref)
            lim = (np.spacing(np.abs(ref).astype(np.float32)) * 2 ** 16 + 2e-5) if bf16 else 2e-6
            assert np.all(dif <= lim), (c, float(dif.max()))
    return rep
