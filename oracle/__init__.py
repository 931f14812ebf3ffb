"""CPU oracle for the DARTree supertree build -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library never
does, and the oracle never imports the product library: the two share only
the seeded inputs of ``speculative_decoding_draft_06_gb300.inputs``.

The arithmetic lives in ``dartree_oracle.c`` (plain single-threaded C, built
with ``-ffp-contract=off``); this module compiles it with gcc and marshals
numpy arrays through ctypes.  See the C file for the method and citations.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dartree_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", platform.machine(), "libdartree_oracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_ERR_ARG, ORC_ERR_CLOSURE, ORC_ERR_ORDER, ORC_ERR_MEM = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, portable flags only)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, f32 = ctypes.c_int32, ctypes.c_float
        lib.orc_version.restype = ctypes.c_int
        lib.orc_round_bf16.argtypes = [f32]
        lib.orc_round_bf16.restype = f32
        lib.orc_state_step.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, i32, P]
        lib.orc_state_step.restype = None
        lib.orc_logits_row.argtypes = [ctypes.c_int] * 3 + [P] * 5
        lib.orc_logits_row.restype = None
        lib.orc_topk_row.argtypes = [ctypes.c_int, P, ctypes.c_int, P, P, P]
        lib.orc_topk_row.restype = None
        lib.orc_pool_size.argtypes = [ctypes.c_int] * 3
        lib.orc_pool_size.restype = ctypes.c_int
        lib.orc_build.argtypes = [ctypes.c_int] * 6 + [P] * 21
        lib.orc_build.restype = ctypes.c_int
        lib.orc_build_ex.argtypes = [ctypes.c_int] * 7 + [P] * 22
        lib.orc_build_ex.restype = ctypes.c_int
        lib.orc_depth.argtypes = [ctypes.c_int] * 7 + [P] * 19
        lib.orc_depth.restype = ctypes.c_int
        lib.orc_path_scores.argtypes = [ctypes.c_int, P, P, P]
        lib.orc_path_scores.restype = ctypes.c_int
        lib.orc_cand_row.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int] + [P] * 4
        lib.orc_cand_row.restype = None
        lib.orc_bestfirst.argtypes = [ctypes.c_int] * 6 + [f32] + [P] * 21
        lib.orc_bestfirst.restype = ctypes.c_int
        lib.orc_tree_attention.argtypes = [ctypes.c_int] * 6 + [f32] + [P] * 7
        lib.orc_tree_attention.restype = ctypes.c_int
        lib.orc_accept.argtypes = [ctypes.c_int] * 2 + [P] * 6
        lib.orc_accept.restype = ctypes.c_int
        lib.orc_topb.argtypes = [ctypes.c_int, P, P, P, P, ctypes.c_int, f32] + [P] * 7
        lib.orc_topb.restype = ctypes.c_int
        lib.orc_heap_prune.argtypes = [ctypes.c_int, P, P, P, ctypes.c_int, f32, P]
        lib.orc_heap_prune.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _weights(a: np.ndarray, bf16: bool) -> np.ndarray:
    return _c(a, np.uint16 if bf16 else np.float32)


def round_bf16(x: float) -> float:
    return float(_load().orc_round_bf16(ctypes.c_float(x)))


def pool_size(D: int, W: int, K: int) -> int:
    return int(_load().orc_pool_size(D, W, K))


def state_step(A, E, s_par, tok: int, bf16: bool) -> np.ndarray:
    """One head state update q(tanh(A s_par + E[tok])) -> fp32 [H];
    A=None is the Markov head q(tanh(E[tok]))."""
    H = E.shape[1]
    A = None if A is None else _weights(A, bf16)
    E = _weights(E, bf16)
    s = _c(s_par, np.float32)
    out = np.empty(H, np.float32)
    _load().orc_state_step(H, int(bf16), _ptr(A), _ptr(E), _ptr(s), tok, _ptr(out))
    return out


def logits_row(z_d, Wout, s, bf16: bool):
    """Corrected logits (fp32 [V]) and their log-sum-exp (float, fp64)."""
    V, H = Wout.shape
    z_d, Wout, s = _c(z_d, np.float32), _weights(Wout, bf16), _c(s, np.float32)
    ell = np.empty(V, np.float32)
    lse = np.zeros(1, np.float64)
    _load().orc_logits_row(V, H, int(bf16), _ptr(z_d), _ptr(Wout), _ptr(s),
                           _ptr(ell), _ptr(lse))
    return ell, float(lse[0])


def topk_row(ell, K: int):
    """Top-K (tokens, values) by (value desc, token asc) and the K/K+1 gap."""
    ell = _c(ell, np.float32)
    tok = np.empty(K, np.int32)
    val = np.empty(K, np.float32)
    gap = np.zeros(1, np.float32)
    _load().orc_topk_row(ell.shape[0], _ptr(ell), K, _ptr(tok), _ptr(val), _ptr(gap))
    return tok, val, float(gap[0])


def cand_row(z_d, Wout, s, cand, bf16: bool):
    """Base-candidate head row: the candidates ``cand`` ordered by corrected
    logit (desc, token asc), their fp32 logits and the log-sum-exp over them."""
    V, H = Wout.shape
    z_d, Wout, s = _c(z_d, np.float32), _weights(Wout, bf16), _c(s, np.float32)
    cand = _c(cand, np.int32)
    K = cand.shape[0]
    tok = np.empty(K, np.int32)
    val = np.empty(K, np.float32)
    lse = np.zeros(1, np.float64)
    _load().orc_cand_row(H, int(bf16), _ptr(z_d), _ptr(Wout), _ptr(s), K, _ptr(cand),
                         _ptr(tok), _ptr(val), _ptr(lse))
    return tok, val, float(lse[0])


def build_tree(inp: dict, r: int, D: int, W: int, K: int, bf16: bool,
               force_slot=None, force_tok=None, force_state=None,
               markov: bool = False, cand_base: bool = False) -> dict:
    """Depth-wise supertree construction for request ``r`` of ``inp``.

    ``force_slot`` / ``force_tok`` ([P] each, pool layout) force the kept
    frontier at every depth (teacher forcing); ``force_state`` ([D, W, H]
    fp32) forces the head states of every depth's rows.  ``markov`` uses the
    Markov head (A ignored); ``cand_base`` takes the candidates from the base
    logits.  Returns the kept pool, the oracle's own per-depth selection,
    per-row results and diagnostics.
    """
    z = _c(inp["z"][r, :D], np.float32)
    V = z.shape[1]
    H = inp["E"].shape[1]
    s0 = _c(inp["state0"][r], np.float32)
    A = None if markov else _weights(inp["A"], bf16)
    E, Wo = (_weights(inp[k], bf16) for k in ("E", "Wout"))
    P = pool_size(D, W, K)
    o = {k: np.empty(P, np.int32) for k in
         ("pool_parent", "pool_token", "pool_depth", "own_slot", "own_tok")}
    o.update({k: np.empty(P, np.float32) for k in
              ("pool_score", "pool_logp", "own_score", "force_margin")})
    o["row_lse"] = np.full(D * W, np.nan, np.float64)
    o["row_tok"] = np.full(D * W * K, -1, np.int32)
    o["row_logp"] = np.full(D * W * K, np.nan, np.float32)
    o["row_kgap"] = np.full(D * W, np.nan, np.float32)
    o["w_cut"] = np.empty(2 * D, np.float32)
    calls = np.zeros(1, np.int64)
    fs = ft = None
    if force_slot is not None:
        fs, ft = _c(force_slot, np.int32), _c(force_tok, np.int32)
    fst = None if force_state is None else _c(force_state, np.float32)
    rc = _load().orc_build_ex(
        V, H, D, W, K, int(bf16), int(cand_base), _ptr(z), _ptr(s0), _ptr(A), _ptr(E), _ptr(Wo),
        _ptr(fs), _ptr(ft), _ptr(fst),
        _ptr(o["pool_parent"]), _ptr(o["pool_token"]), _ptr(o["pool_depth"]),
        _ptr(o["pool_score"]), _ptr(o["pool_logp"]), _ptr(o["own_slot"]), _ptr(o["own_tok"]),
        _ptr(o["own_score"]), _ptr(o["force_margin"]), _ptr(o["row_lse"]),
        _ptr(o["row_tok"]), _ptr(o["row_logp"]), _ptr(o["row_kgap"]),
        _ptr(o["w_cut"]), _ptr(calls))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_build_ex failed with code {rc}")
    o["row_lse"] = o["row_lse"].reshape(D, W)
    o["row_tok"] = o["row_tok"].reshape(D, W, K)
    o["row_logp"] = o["row_logp"].reshape(D, W, K)
    o["row_kgap"] = o["row_kgap"].reshape(D, W)
    o["w_cut"] = o["w_cut"].reshape(D, 2)
    o["calls"] = int(calls[0])
    return o


def depth(z_d, Wout, states, score, W: int, K: int, bf16: bool, force_slot=None,
          force_tok=None, cand_base: bool = False) -> dict:
    """One depth of the construction from given frontier rows (see orc_depth):
    ``states`` [fp, H] fp32 and cumulative ``score`` [fp]; optional forced
    kept frontier ``force_slot`` / ``force_tok`` [fd].  Returns the per-row
    head results, the own top-W, the kept frontier's scores and log-probs,
    the forcing margins and the W-th / (W+1)-th candidate scores."""
    Wo = _weights(Wout, bf16)
    V, H = Wo.shape
    z_d = _c(z_d, np.float32)
    st = _c(states, np.float32)
    sc = _c(score, np.float32)
    fp = st.shape[0]
    fd = min(W, K * fp)
    o = {k: np.empty(fd, np.int32) for k in ("own_slot", "own_tok", "sel_slot", "sel_tok")}
    o.update({k: np.empty(fd, np.float32) for k in
              ("own_score", "sel_score", "sel_logp", "force_margin")})
    o["row_lse"] = np.empty(fp, np.float64)
    o["row_tok"] = np.empty((fp, K), np.int32)
    o["row_logp"] = np.empty((fp, K), np.float32)
    o["row_kgap"] = np.empty(fp, np.float32)
    o["w_cut"] = np.empty(2, np.float32)
    fs = ft = None
    if force_slot is not None:
        fs, ft = _c(force_slot, np.int32), _c(force_tok, np.int32)
        assert fs.shape == (fd,) and ft.shape == (fd,)
    rc = _load().orc_depth(
        V, H, fp, W, K, int(bf16), int(cand_base), _ptr(z_d), _ptr(Wo), _ptr(st), _ptr(sc),
        _ptr(fs), _ptr(ft), _ptr(o["own_slot"]), _ptr(o["own_tok"]), _ptr(o["own_score"]),
        _ptr(o["sel_slot"]), _ptr(o["sel_tok"]), _ptr(o["sel_score"]), _ptr(o["sel_logp"]),
        _ptr(o["force_margin"]), _ptr(o["row_lse"]), _ptr(o["row_tok"]), _ptr(o["row_logp"]),
        _ptr(o["row_kgap"]), _ptr(o["w_cut"]))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_depth failed with code {rc}")
    return o


def path_scores(pool_parent, pool_logp) -> np.ndarray:
    """Cumulative scores of a pool from each node's log-prob given its parent."""
    pp, lp = _c(pool_parent, np.int32), _c(pool_logp, np.float32)
    out = np.empty(pp.shape[0], np.float32)
    rc = _load().orc_path_scores(pp.shape[0], _ptr(pp), _ptr(lp), _ptr(out))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_path_scores failed with code {rc}")
    return out


def topb(pool_parent, pool_token, pool_depth, pool_score, B: int, beta: float) -> dict:
    """Deferred Top-B, compaction and ancestor mask over one request's pool."""
    pp, pt, pd = (_c(a, np.int32) for a in (pool_parent, pool_token, pool_depth))
    ps = _c(pool_score, np.float32)
    P = pp.shape[0]
    words = (B + 31) // 32
    o = {"parent": np.empty(B, np.int32), "token": np.empty(B, np.int32),
         "depth": np.empty(B, np.int32), "score": np.empty(B, np.float32),
         "mask": np.empty(B * words, np.uint32), "order": np.full(B, -1, np.int32)}
    n = np.zeros(1, np.int32)
    rc = _load().orc_topb(P, _ptr(pp), _ptr(pt), _ptr(pd), _ptr(ps), B,
                          ctypes.c_float(beta), _ptr(o["parent"]), _ptr(o["token"]),
                          _ptr(o["depth"]), _ptr(o["score"]), _ptr(o["mask"]),
                          _ptr(n), _ptr(o["order"]))
    o["n_out"] = int(n[0])
    o["rc"] = rc
    o["mask"] = o["mask"].reshape(B, words)
    return o


def heap_prune(pool_parent, pool_depth, pool_score, B: int, beta: float) -> np.ndarray:
    """Sequential best-first max-heap pruning; returns the pop order."""
    pp, pd = _c(pool_parent, np.int32), _c(pool_depth, np.int32)
    ps = _c(pool_score, np.float32)
    out = np.full(B, -1, np.int32)
    n = _load().orc_heap_prune(pp.shape[0], _ptr(pp), _ptr(pd), _ptr(ps), B,
                               ctypes.c_float(beta), _ptr(out))
    if n < 0:
        raise MemoryError("orc_heap_prune")
    return out[:n]


def build_request(inp: dict, r: int, D: int, W: int, K: int, B: int,
                  beta: float, bf16: bool) -> dict:
    """Full oracle pipeline for one request: construction then pruning."""
    t = build_tree(inp, r, D, W, K, bf16)
    t["tree"] = topb(t["pool_parent"], t["pool_token"], t["pool_depth"],
                     t["pool_score"], B, beta)
    return t


def bestfirst(inp: dict, r: int, D: int, K: int, B: int, beta: float, bf16: bool,
              markov: bool = False, force_tok=None, force_logp=None,
              force_state=None) -> dict:
    """Sequential best-first build (one head call per expanded node) for
    request ``r``: the tree in pop order plus per-call diagnostics.
    ``force_tok`` / ``force_logp`` ([B, K]) replace each call's children,
    ``force_state`` ([B, H]) each call's state (teacher forcing)."""
    z = _c(inp["z"][r, :D], np.float32)
    V = z.shape[1]
    H = inp["E"].shape[1]
    s0 = _c(inp["state0"][r], np.float32)
    A = None if markov else _weights(inp["A"], bf16)
    E, Wo = (_weights(inp[k], bf16) for k in ("E", "Wout"))
    words = (B + 31) // 32
    o = {"parent": np.empty(B, np.int32), "token": np.empty(B, np.int32),
         "depth": np.empty(B, np.int32), "score": np.empty(B, np.float32),
         "mask": np.empty(B * words, np.uint32), "call_rank": np.empty(B, np.int32),
         "call_state": np.zeros((B, H), np.float32),
         "row_lse": np.full(B, np.nan, np.float64), "row_tok": np.full((B, K), -1, np.int32),
         "row_logp": np.full((B, K), np.nan, np.float32),
         "row_kgap": np.full(B, np.nan, np.float32)}
    n = np.zeros(1, np.int32)
    calls = np.zeros(1, np.int64)
    ft = None if force_tok is None else _c(force_tok, np.int32)
    fl = None if force_logp is None else _c(force_logp, np.float32)
    fs = None if force_state is None else _c(force_state, np.float32)
    rc = _load().orc_bestfirst(
        V, H, D, K, B, int(bf16), ctypes.c_float(beta), _ptr(z), _ptr(s0), _ptr(A), _ptr(E),
        _ptr(Wo), _ptr(ft), _ptr(fl), _ptr(fs), _ptr(o["parent"]), _ptr(o["token"]),
        _ptr(o["depth"]), _ptr(o["score"]), _ptr(o["mask"]), _ptr(n), _ptr(o["call_rank"]),
        _ptr(o["call_state"]), _ptr(o["row_lse"]), _ptr(o["row_tok"]), _ptr(o["row_logp"]),
        _ptr(o["row_kgap"]), _ptr(calls))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_bestfirst failed with code {rc}")
    o["n_out"] = int(n[0])
    o["calls"] = int(calls[0])
    o["mask"] = o["mask"].reshape(B, words)
    return o


def tree_attention(Q, Kp, Vp, Kt, Vt, mask, scale: float, bf16: bool) -> np.ndarray:
    """Tree attention of one request (see orc_tree_attention): Q [B+1, Hq, dh],
    Kp/Vp [Lp, Hkv, dh], Kt/Vt [B, Hkv, dh] (bf16 bits or fp32), mask
    [B, words] -> O [B+1, Hq, dh] fp32."""
    Bp1, Hq, dh = Q.shape
    B = Bp1 - 1
    Lp, Hkv = Kp.shape[0], Kp.shape[1]
    arrs = [_weights(x, bf16) for x in (Q, Kp, Vp, Kt, Vt)]
    m = _c(mask, np.uint32).reshape(-1)
    O = np.empty((Bp1, Hq, dh), np.float32)
    rc = _load().orc_tree_attention(Lp, B, Hq, Hkv, dh, int(bf16), ctypes.c_float(scale),
                                    *[_ptr(a) for a in arrs], _ptr(m), _ptr(O))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_tree_attention failed with code {rc}")
    return O


def accept(parent, token, n_out: int, pred) -> dict:
    """Longest accepted prefix of one request's tree under the target's
    predictions pred [B+1] (root first)."""
    pp, tt = _c(parent, np.int32), _c(token, np.int32)
    pr = _c(pred, np.int32)
    B = pp.shape[0]
    nodes = np.full(max(B, 1), -1, np.int32)
    ln = np.zeros(1, np.int32)
    bonus = np.zeros(1, np.int32)
    rc = _load().orc_accept(B, n_out, _ptr(pp), _ptr(tt), _ptr(pr), _ptr(ln), _ptr(nodes),
                            _ptr(bonus))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_accept failed with code {rc}")
    n = int(ln[0])
    return {"len": n, "nodes": nodes[:n].copy(), "bonus": int(bonus[0])}
