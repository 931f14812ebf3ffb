"""Python binding of the DARTree C ABI (``include/dartree.h``).

Argument marshalling only: every step of a build runs in the CUDA library
``_build/libdartree.so``.  There is no fallback -- if the library has not been
built (``__graft_entry__.build()`` or ``python -m
speculative_decoding_draft_06_gb300.build``), :func:`load` raises.
Tensors are PyTorch CUDA tensors (PyTorch provides device memory and
streams); bf16 weights may be ``torch.bfloat16`` or 16-bit integer tensors
holding bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import platform
import re

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", platform.machine(), "libdartree.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dartree.h")

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "DEVICE_CHECK",
          5: "TIMEOUT", 6: "OOM"}
W_F32, W_BF16 = 0, 1
WEIGHT_LAYOUTS = {"rows": 0, "blocks": 1}
HEAD_KINDS = {"recurrent": 0, "markov": 1}
CAND_KINDS = {"corrected": 0, "base": 1}
EXPANSIONS = {"depthwise": 0, "bestfirst": 1}

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("V", "H", "max_D", "max_W", "max_K", "max_B", "max_requests", "wdtype")]


class HeadWeights(ctypes.Structure):
    _fields_ = [("A", _vp), ("E", _vp), ("Wout", _vp)]


class Options(ctypes.Structure):
    _fields_ = [("head_kind", ctypes.c_int32), ("candidates", ctypes.c_int32),
                ("expansion", ctypes.c_int32)]


class Tree(ctypes.Structure):
    _fields_ = [("parent", _vp), ("token", _vp), ("depth", _vp), ("score", _vp),
                ("mask", _vp), ("n_out", _vp)]


class DartreeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"dartree {STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def declared_symbols() -> list[str]:
    """Function names declared by include/dartree.h."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"\b(dartree_[a-z_]+)\s*\(", txt)))


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"DARTree CUDA library not built ({LIB_PATH} missing); "
                           "run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    st = ctypes.c_int
    sig = {
        "dartree_pool_size": (_i32, [_i32, _i32, _i32]),
        "dartree_create": (st, [ctypes.POINTER(Config), ctypes.POINTER(_vp)]),
        "dartree_destroy": (None, [_vp]),
        "dartree_build": (st, [_vp, _vp, _vp, ctypes.POINTER(HeadWeights), _i32, _i32, _i32,
                               _i32, _i32, ctypes.c_float, ctypes.POINTER(Tree), _vp]),
        "dartree_build_ex": (st, [_vp, _vp, _vp, ctypes.POINTER(HeadWeights), _i32, _i32,
                                  _i32, _i32, _i32, ctypes.c_float, ctypes.POINTER(Options),
                                  ctypes.POINTER(Tree), _vp]),
        "dartree_build_host": (st, [_vp, _vp, _vp, ctypes.POINTER(HeadWeights), _i32, _i32,
                                    _i32, _i32, _i32, ctypes.c_float, ctypes.POINTER(Tree), _vp]),
        "dartree_sync_status": (st, [_vp, _vp]),
        "dartree_head_calls": (ctypes.c_int64, [_vp]),
        "dartree_set_weight_layout": (st, [_vp, _i32]),
        "dartree_blocked_weight_bytes": (ctypes.c_size_t, [_i32, _i32]),
        "dartree_block_weights": (st, [_vp, _i32, _i32, _vp, _vp]),
        "dartree_last_error": (ctypes.c_char_p, [_vp]),
        "dartree_get_pool": (st, [_vp, _vp, _vp, _vp, _vp, _vp]),
        "dartree_get_rows": (st, [_vp, _i32, _vp, _vp, _vp, _vp]),
        "dartree_head_topk": (st, [_vp, _vp, _vp, ctypes.c_int64, _i32, _vp, _i32, _i32, _vp,
                                   _vp, _vp, _vp]),
        "dartree_state_step": (st, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp]),
        "dartree_prune": (st, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_float,
                               ctypes.POINTER(Tree), _vp]),
        "dartree_set_timing": (st, [_vp, _i32]),
        "dartree_get_timing": (st, [_vp, _i32, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_int64)]),
        "dartree_reset_timing": (st, [_vp]),
        "dartree_state_step_noalloc": (st, [_vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp]),
        "dartree_get_states": (st, [_vp, _i32, _vp, _vp]),
        "dartree_tree_attention": (st, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                        ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _vp,
                                        _vp]),
        "dartree_tree_attention_workspace": (ctypes.c_size_t, [_i32, _i32, _i32, _i32, _i32]),
        "dartree_accept": (st, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def pool_size(D: int, W: int, K: int) -> int:
    return int(load().dartree_pool_size(D, W, K))


def frontier_sizes(D: int, W: int, K: int) -> list[int]:
    f, out = 1, []
    for _ in range(D):
        f = min(W, K * f)
        out.append(f)
    return out


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtypes) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


_W16 = (torch.bfloat16, torch.int16, torch.uint16)


class DARTree:
    """One library context: fixed V, H, capacities and weight dtype."""

    def __init__(self, V: int, H: int, *, max_D: int, max_W: int, max_K: int, max_B: int,
                 max_requests: int = 1, bf16: bool = True, device: int | None = None):
        lib = load()
        if device is not None:
            torch.cuda.set_device(device)
        torch.cuda.init()
        self.cfg = Config(V, H, max_D, max_W, max_K, max_B, max_requests,
                          W_BF16 if bf16 else W_F32)
        self.bf16 = bf16
        self.V, self.H = V, H
        h = ctypes.c_void_p()
        s = lib.dartree_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if s != 0:
            raise DartreeError(s, "dartree_create: " + lib.dartree_last_error(None).decode())
        self._h = h
        self._lib = lib

    # ------------------------------------------------------------ plumbing
    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.dartree_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, s: int) -> None:
        if s != 0:
            raise DartreeError(s, self._lib.dartree_last_error(self._h).decode())

    def _wtypes(self):
        return _W16 if self.bf16 else (torch.float32,)

    def _head(self, A, E, Wout) -> HeadWeights:
        """A may be None (Markov head)."""
        wt = self._wtypes()
        _dev(E, "E", wt), _dev(Wout, "Wout", wt)
        if A is not None:
            _dev(A, "A", wt)
        return HeadWeights(None if A is None else A.data_ptr(), E.data_ptr(), Wout.data_ptr())

    def alloc_tree(self, R: int, B: int, *, device="cuda", pin: bool = False) -> dict:
        words = (B + 31) // 32
        kw = {"device": device} if device != "cpu" else {"pin_memory": pin}
        return {"parent": torch.empty(R, B, dtype=torch.int32, **kw),
                "token": torch.empty(R, B, dtype=torch.int32, **kw),
                "depth": torch.empty(R, B, dtype=torch.int32, **kw),
                "score": torch.empty(R, B, dtype=torch.float32, **kw),
                "mask": torch.empty(R, B, words, dtype=torch.int32, **kw),
                "n_out": torch.empty(R, dtype=torch.int32, **kw)}

    @staticmethod
    def _tree(out: dict) -> Tree:
        return Tree(*(out[k].data_ptr() for k in ("parent", "token", "depth", "score", "mask",
                                                  "n_out")))

    # ------------------------------------------------------------ the path
    def build(self, z, state0, A, E, Wout, *, D: int, W: int, K: int, B: int, beta: float,
              out: dict | None = None, stream=None, head: str = "recurrent",
              candidates: str = "corrected", expansion: str = "depthwise") -> dict:
        """Asynchronous supertree build; z [R,D,V] fp32, state0 [R,H] fp32.
        ``head`` / ``candidates`` / ``expansion`` select the build variant
        (dartree_build_ex); the defaults are dartree_build."""
        _dev(z, "z", (torch.float32,)), _dev(state0, "state0", (torch.float32,))
        R = state0.shape[0]
        if z.shape != (R, D, self.V) or state0.shape != (R, self.H):
            raise ValueError(f"z {tuple(z.shape)} / state0 {tuple(state0.shape)} do not match "
                             f"R={R}, D={D}, V={self.V}, H={self.H}")
        if out is None:
            out = self.alloc_tree(R, B, device=z.device)
        hw = self._head(A, E, Wout)
        t = self._tree(out)
        opt = (head, candidates, expansion)
        if opt == ("recurrent", "corrected", "depthwise"):
            self._check(self._lib.dartree_build(self._h, _ptr(z), _ptr(state0), ctypes.byref(hw),
                                                R, D, W, K, B, ctypes.c_float(beta),
                                                ctypes.byref(t), _stream(stream)))
        else:
            o = Options(HEAD_KINDS[head], CAND_KINDS[candidates], EXPANSIONS[expansion])
            self._check(self._lib.dartree_build_ex(
                self._h, _ptr(z), _ptr(state0), ctypes.byref(hw), R, D, W, K, B,
                ctypes.c_float(beta), ctypes.byref(o), ctypes.byref(t), _stream(stream)))
        return out

    def build_host(self, z_host, state0_host, A, E, Wout, *, D: int, W: int, K: int, B: int,
                   beta: float, out_host: dict, stream=None) -> dict:
        """Build from host inputs into host outputs (copies included, synchronous)."""
        for n, t in (("z", z_host), ("state0", state0_host)):
            if t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
                raise TypeError(f"{n} must be a contiguous fp32 host tensor")
        R = state0_host.shape[0]
        head = self._head(A, E, Wout)
        t = self._tree(out_host)
        self._check(self._lib.dartree_build_host(
            self._h, _ptr(z_host), _ptr(state0_host), ctypes.byref(head), R, D, W, K, B,
            ctypes.c_float(beta), ctypes.byref(t), _stream(stream)))
        return out_host

    def sync(self, stream=None) -> None:
        """Synchronise and raise on a device-side check."""
        self._check(self._lib.dartree_sync_status(self._h, _stream(stream)))

    def sync_status(self, stream=None) -> int:
        return int(self._lib.dartree_sync_status(self._h, _stream(stream)))

    KERNEL_KINDS = ("head", "state", "merge", "select", "prune", "root", "candidates",
                    "bestfirst")

    def set_timing(self, on: bool) -> None:
        self._check(self._lib.dartree_set_timing(self._h, 1 if on else 0))

    def reset_timing(self) -> None:
        self._check(self._lib.dartree_reset_timing(self._h))

    def timing(self) -> dict:
        """{kind: (total_ms, launches)} accumulated at each sync()."""
        out = {}
        for i, k in enumerate(self.KERNEL_KINDS):
            ms, n = ctypes.c_double(), ctypes.c_int64()
            self._check(self._lib.dartree_get_timing(self._h, i, ctypes.byref(ms),
                                                     ctypes.byref(n)))
            out[k] = (ms.value, n.value)
        return out

    def set_weight_layout(self, layout: str) -> None:
        """Layout of the Wout passed to later calls: "rows" ([V, H]
        row-major) or "blocks" (128 x 64 blocks, see block_weights;
        dartree_set_weight_layout)."""
        self._check(self._lib.dartree_set_weight_layout(self._h, WEIGHT_LAYOUTS[layout]))

    def head_calls(self) -> int:
        return int(self._lib.dartree_head_calls(self._h))

    def last_error(self) -> str:
        return self._lib.dartree_last_error(self._h).decode()

    def get_pool(self, R: int, P: int, stream=None) -> dict:
        o = {k: torch.empty(R, P, dtype=torch.int32) for k in ("parent", "token", "depth")}
        o["score"] = torch.empty(R, P, dtype=torch.float32)
        self._check(self._lib.dartree_get_pool(self._h, _ptr(o["parent"]), _ptr(o["token"]),
                                               _ptr(o["depth"]), _ptr(o["score"]),
                                               _stream(stream)))
        torch.cuda.synchronize()
        return o

    def get_rows(self, d: int, rows: int, K: int, stream=None) -> dict:
        o = {"lse": torch.empty(rows, dtype=torch.float64),
             "tok": torch.empty(rows, K, dtype=torch.int32),
             "logp": torch.empty(rows, K, dtype=torch.float32)}
        self._check(self._lib.dartree_get_rows(self._h, d, _ptr(o["lse"]), _ptr(o["tok"]),
                                               _ptr(o["logp"]), _stream(stream)))
        torch.cuda.synchronize()
        return o

    def get_states(self, d: int, rows: int, stream=None):
        """Head states of head call d as fp32 [rows, H] (bf16 values widened)."""
        dt = torch.int16 if self.bf16 else torch.float32
        o = torch.empty(rows, self.H, dtype=dt)
        self._check(self._lib.dartree_get_states(self._h, d, _ptr(o), _stream(stream)))
        torch.cuda.synchronize()
        if self.bf16:
            return (o.numpy().view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
        return o.numpy()

    # ------------------------------------------------ single-step entries
    def head_topk(self, S, z, Wout, *, K: int, rows_per_req: int | None = None,
                  z_req_stride: int = 0, stream=None) -> dict:
        """One batched head call: per row lse, top-K tokens and log-probs."""
        _dev(S, "S", self._wtypes()), _dev(z, "z", (torch.float32,))
        _dev(Wout, "Wout", self._wtypes())
        M = S.shape[0]
        dev = S.device
        o = {"lse": torch.empty(M, dtype=torch.float64, device=dev),
             "tok": torch.empty(M, K, dtype=torch.int32, device=dev),
             "logp": torch.empty(M, K, dtype=torch.float32, device=dev)}
        self._check(self._lib.dartree_head_topk(
            self._h, _ptr(S), _ptr(z), int(z_req_stride), rows_per_req or M, _ptr(Wout), M, K,
            _ptr(o["lse"]), _ptr(o["tok"]), _ptr(o["logp"]), _stream(stream)))
        return o

    def state_step(self, S_par, tok, A, E, stream=None):
        """S_out = q(tanh(A S_par + E[tok])) for every row."""
        wt = self._wtypes()
        _dev(S_par, "S_par", wt), _dev(tok, "tok", (torch.int32,))
        _dev(A, "A", wt), _dev(E, "E", wt)
        out = torch.empty_like(S_par)
        self._check(self._lib.dartree_state_step(self._h, _ptr(S_par), _ptr(tok), _ptr(A),
                                                 _ptr(E), S_par.shape[0], _ptr(out),
                                                 _stream(stream)))
        return out

    def prune(self, parent, token, depth, score, *, B: int, beta: float, stream=None) -> dict:
        """Deferred Top-B + compaction + mask over pools [R, P]."""
        for n, t in (("parent", parent), ("token", token), ("depth", depth)):
            _dev(t, n, (torch.int32,))
        _dev(score, "score", (torch.float32,))
        R, P = parent.shape
        out = self.alloc_tree(R, B, device=parent.device)
        t = self._tree(out)
        self._check(self._lib.dartree_prune(self._h, _ptr(parent), _ptr(token), _ptr(depth),
                                            _ptr(score), R, P, B, ctypes.c_float(beta),
                                            ctypes.byref(t), _stream(stream)))
        return out


def state_step_noalloc(S_par, tok, A, E, stream=None):
    """Context-free bf16 state step (dartree_state_step_noalloc): for callers
    that cannot allocate device memory.  The output tensor is allocated here
    by PyTorch only because this is the Python convenience wrapper; the C
    entry point itself allocates nothing.  Raises DartreeError on failure."""
    lib = load()
    for n, t in (("S_par", S_par), ("A", A), ("E", E)):
        _dev(t, n, _W16)
    _dev(tok, "tok", (torch.int32,))
    M, H = S_par.shape
    out = torch.empty_like(S_par)
    s = lib.dartree_state_step_noalloc(_ptr(S_par), _ptr(tok), _ptr(A), _ptr(E), H, M, _ptr(out),
                                       _stream(stream))
    if s != 0:
        raise DartreeError(s, lib.dartree_last_error(None).decode())
    return out


def weights_to_device(inp: dict, bf16: bool, device="cuda") -> dict:
    """Host input arrays (numpy) -> device tensors in the library's layout."""
    def w(a):
        t = torch.from_numpy(a)
        if bf16:
            t = t.view(torch.int16)
        return t.to(device)
    return {"A": w(inp["A"]), "E": w(inp["E"]), "Wout": w(inp["Wout"]),
            "z": torch.from_numpy(inp["z"]).to(device),
            "state0": torch.from_numpy(inp["state0"]).to(device)}


def _check_free(s: int) -> None:
    if s != 0:
        raise DartreeError(s, load().dartree_last_error(None).decode())


def tree_attention(Q, K, Vt, mask, *, Lp: int, scale: float | None = None,
                   want_bf16: bool = True, work=None, split: bool = True, err=None,
                   stream=None) -> dict:
    """Tree attention of the verification forward (dartree_tree_attention):
    Q [R,B+1,Hq,dh], key cache K [R,Hkv,Lp+B,dh] (prefix keys, then the tree
    nodes'), blocked transposed value cache Vt [R,Hkv,ceil(L/64),dh,64] (bf16
    CUDA tensors; see kv_cache),
    mask [R,B,words] int32 -> {"O": fp32, "O16": bf16 bits}.  ``work`` and
    ``split`` are kept for the interface: the key splits need no scratch."""
    for n, t in (("Q", Q), ("K", K), ("Vt", Vt)):
        _dev(t, n, _W16)
    _dev(mask, "mask", (torch.int32,))
    R, Bp1, Hq, dh = Q.shape
    Hkv = K.shape[1]
    O = torch.empty(R, Bp1, Hq, dh, dtype=torch.float32, device=Q.device)
    O16 = torch.empty(R, Bp1, Hq, dh, dtype=torch.int16, device=Q.device) if want_bf16 else None
    sc = float(scale) if scale is not None else dh ** -0.5
    wb = 0 if work is None else work.numel() * work.element_size()
    _check_free(load().dartree_tree_attention(
        _ptr(Q), _ptr(K), _ptr(Vt), _ptr(mask), R, Lp, Bp1 - 1, Hq, Hkv, dh,
        ctypes.c_float(sc), _ptr(O), _ptr(O16), _ptr(work), wb, _ptr(err), _stream(stream)))
    return {"O": O, "O16": O16}


def block_weights(W: torch.Tensor, stream=None) -> torch.Tensor:
    """The blocked layout (blocks of 128 rows x 64 columns, rows past V
    zero; dartree_block_weights) of a row-major bf16 CUDA matrix [V, H],
    as a [ceil(V/128) * 128, H] tensor of the same dtype."""
    _dev(W, "W", _W16)
    V, H = W.shape
    n = int(load().dartree_blocked_weight_bytes(V, H))
    if n == 0:
        raise ValueError("H must be a multiple of 64")
    out = torch.empty(n // (2 * H), H, dtype=W.dtype, device=W.device)
    _check_free(load().dartree_block_weights(_ptr(W), V, H, _ptr(out), _stream(stream)))
    return out


def kv_cache(Kp, Vp, Kt, Vt) -> tuple[torch.Tensor, torch.Tensor]:
    """Key cache [R, Hkv, Lp+B, dh] and blocked transposed value cache
    [R, Hkv, ceil(L/64), dh, 64] from prefix [R, Lp, Hkv, dh] and tree
    [R, B, Hkv, dh] keys / values (CUDA tensors; data movement only)."""
    K = torch.cat([Kp, Kt], dim=1).permute(0, 2, 1, 3).contiguous()   # [R, Hkv, L, dh]
    V = torch.cat([Vp, Vt], dim=1).permute(0, 2, 1, 3)                 # [R, Hkv, L, dh]
    R, Hkv, L, dh = V.shape
    nb = (L + 63) // 64
    Vb = torch.zeros(R, Hkv, nb * 64, dh, dtype=V.dtype, device=V.device)
    Vb[:, :, :L] = V
    VT = Vb.view(R, Hkv, nb, 64, dh).transpose(3, 4).contiguous()      # [R, Hkv, nb, dh, 64]
    return K, VT


def accept(parent, token, n_out, pred, *, max_len: int, stream=None) -> dict:
    """Longest accepted prefix per request (dartree_accept); CUDA int32
    tensors parent/token [R,B], n_out [R], pred [R,B+1]."""
    for n, t in (("parent", parent), ("token", token), ("n_out", n_out), ("pred", pred)):
        _dev(t, n, (torch.int32,))
    R, B = parent.shape
    dev = parent.device
    o = {"len": torch.empty(R, dtype=torch.int32, device=dev),
         "nodes": torch.empty(R, max(max_len, 1), dtype=torch.int32, device=dev),
         "bonus": torch.empty(R, dtype=torch.int32, device=dev)}
    _check_free(load().dartree_accept(_ptr(parent), _ptr(token), _ptr(n_out), _ptr(pred), R, B,
                                      max_len, _ptr(o["len"]), _ptr(o["nodes"]), _ptr(o["bonus"]),
                                      _stream(stream)))
    return o
