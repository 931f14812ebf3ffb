"""The allocation-free state step (dartree_state_step_noalloc).

Some callers cannot create a context because they may not allocate device
memory: their device heap belongs to a server's or framework's allocator, or
they sit on a latency-critical path where cudaMalloc/cudaFree (which
synchronise the device) are not allowed.  For them the library offers one
context-free entry point whose scratch is a static device array.  These tests
check, through the C ABI, that two calls in a row give the rows of the oracle's
state step and of the context-based dartree_state_step, within the state-step
tolerance of the other GPU tests (split-K and unsplit contractions); that a
device wait that runs out is reported by dartree_sync_status(NULL, stream)
instead of being lost; and that sizes beyond the scratch limits and
misaligned weights are refused before any launch.  The file is collected
last and needs no other test to have run first.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I

pytestmark = pytest.mark.gpu

OK, INVALID_ARG, UNSUPPORTED, TIMEOUT = 0, 1, 2, 5


def _bf16_rows(g, M, H):
    S = np.tanh(g.standard_normal((M, H))).astype(np.float32)
    return torch.from_numpy(I.to_bf16_bits(S)).view(torch.int16).cuda()


def _as_f32(t):
    return I.bf16_bits_to_f32(t.cpu().view(torch.int16).numpy().view(np.uint16))


def _noalloc(lib, S, tok, A, E, out, H=None, M=None):
    M0, H0 = S.shape
    return lib.dartree_state_step_noalloc(
        ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(tok.data_ptr()),
        ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(E.data_ptr()), H or H0, M or M0,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _status(lib):
    return lib.dartree_sync_status(None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _within_one_bf16_step(got, want, M, H):
    # the tolerance of the state-step parity test: one bf16 rounding step
    # (fp32 accumulation and tanhf vs fp64 can cross a rounding boundary)
    # plus 2e-5 absolute near zero, in at most 1 % of the elements
    ulp = np.spacing(np.abs(want)) * 2 ** 16
    assert np.all(np.abs(got - want) <= ulp + 2e-5)
    assert np.count_nonzero(got != want) <= 0.01 * M * H


@pytest.mark.parametrize("H,M1,M2", [(256, 37, 200), (4096, 16, 5), (64, 9, 130)])
def test_noalloc_state_step_matches_oracle_and_context_entry_point(H, M1, M2):
    lib = dtl.load()
    w = I.small_workload(77 + H, V=400, H=H, D=1, W=1, K=1, B=1, bf16=True)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, True)
    g = np.random.default_rng(H)
    ctx = dtl.DARTree(w.V, H, max_D=1, max_W=256, max_K=1, max_B=1, bf16=True)
    for M in (M1, M2):                      # two calls in a row, different sizes
        S = _bf16_rows(g, M, H)
        tok_h = g.integers(0, w.V, M).astype(np.int32)
        tok = torch.from_numpy(tok_h).cuda()
        out = torch.empty_like(S)
        assert _noalloc(lib, S, tok, dev["A"], dev["E"], out) == OK, \
            lib.dartree_last_error(None).decode()
        assert _status(lib) == OK, lib.dartree_last_error(None).decode()
        ref = ctx.state_step(S, tok, dev["A"], dev["E"])
        ctx.sync()
        got = _as_f32(out)
        S_h = _as_f32(S)
        want = np.stack([oracle.state_step(inp["A"], inp["E"], S_h[m], int(tok_h[m]), True)
                         for m in range(M)])
        _within_one_bf16_step(got, want, M, H)
        _within_one_bf16_step(got, _as_f32(ref), M, H)
    ctx.close()


def test_noalloc_wait_timeout_is_reported_then_cleared(monkeypatch):
    """A one-cycle limit on the pipeline waits (test knob) makes the
    contraction give up; the next status read reports TIMEOUT and clears the
    word, and a normal call afterwards is correct and reports OK."""
    lib = dtl.load()
    H, M = 256, 16
    w = I.small_workload(79, V=300, H=H, D=1, W=1, K=1, B=1, bf16=True)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, True)
    g = np.random.default_rng(5)
    S = _bf16_rows(g, M, H)
    tok_h = g.integers(0, w.V, M).astype(np.int32)
    tok = torch.from_numpy(tok_h).cuda()
    out = torch.empty_like(S)
    monkeypatch.setenv("DARTREE_WAIT_LIMIT_CYCLES", "1")
    assert _noalloc(lib, S, tok, dev["A"], dev["E"], out) == OK
    monkeypatch.delenv("DARTREE_WAIT_LIMIT_CYCLES")
    assert _status(lib) == TIMEOUT
    assert "timed out" in lib.dartree_last_error(None).decode()
    assert _status(lib) == OK                # read once, then cleared
    assert _noalloc(lib, S, tok, dev["A"], dev["E"], out) == OK
    assert _status(lib) == OK
    S_h = _as_f32(S)
    want = np.stack([oracle.state_step(inp["A"], inp["E"], S_h[m], int(tok_h[m]), True)
                     for m in range(M)])
    _within_one_bf16_step(_as_f32(out), want, M, H)


def test_noalloc_rejects_sizes_beyond_its_scratch_and_misaligned_weights():
    lib = dtl.load()
    one = torch.zeros(4096, dtype=torch.int16, device="cuda")
    p = ctypes.c_void_p(one.data_ptr())
    for H, M in ((4160, 8), (256, 257)):
        s = lib.dartree_state_step_noalloc(p, p, p, p, H, M, p, None)
        assert s == UNSUPPORTED
        assert "4096" in lib.dartree_last_error(None).decode()
    assert lib.dartree_state_step_noalloc(p, p, p, p, 100, 8, p, None) == INVALID_ARG
    odd = ctypes.c_void_p(one.data_ptr() + 8)          # 8-byte but not 16-byte aligned
    assert lib.dartree_state_step_noalloc(p, p, p, odd, 256, 8, p, None) == INVALID_ARG
    assert "aligned" in lib.dartree_last_error(None).decode()
    assert lib.dartree_state_step_noalloc(p, p, odd, p, 256, 8, p, None) == INVALID_ARG
