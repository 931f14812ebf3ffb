"""The allocation-free state step (dartree_state_step_noalloc).

Some callers cannot create a context because they may not allocate device
memory: their device heap belongs to a server's or framework's allocator, or
they sit on a latency-critical path where cudaMalloc/cudaFree (which
synchronise the device) are not allowed.  For them the library offers one
context-free entry point whose scratch is a static device array.  This test
checks, through the C ABI, that two calls in a row give the same rows as the
context-based dartree_state_step within the state-step tolerance of the other
GPU tests, and that sizes beyond the scratch limits are refused before any
launch.  It lives in its own file, collected last, and needs no other test
to have run first.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _bf16_rows(g, M, H):
    S = np.tanh(g.standard_normal((M, H))).astype(np.float32)
    return torch.from_numpy(I.to_bf16_bits(S)).view(torch.int16).cuda()


def _as_f32(t):
    return I.bf16_bits_to_f32(t.cpu().view(torch.int16).numpy().view(np.uint16))


def _noalloc(lib, S, tok, A, E, out):
    M, H = S.shape
    return lib.dartree_state_step_noalloc(
        ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(tok.data_ptr()),
        ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(E.data_ptr()), H, M,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("H,M1,M2", [(256, 37, 200), (4096, 16, 5)])
def test_noalloc_state_step_matches_context_entry_point(H, M1, M2):
    lib = dtl.load()
    w = I.small_workload(77 + H, V=400, H=H, D=1, W=1, K=1, B=1, bf16=True)
    dev = dtl.weights_to_device(I.make_inputs(w), True)
    g = np.random.default_rng(H)
    ctx = dtl.DARTree(w.V, H, max_D=1, max_W=256, max_K=1, max_B=1, bf16=True)
    for M in (M1, M2):                      # two calls in a row, different sizes
        S = _bf16_rows(g, M, H)
        tok = torch.from_numpy(g.integers(0, w.V, M).astype(np.int32)).cuda()
        out = torch.empty_like(S)
        assert _noalloc(lib, S, tok, dev["A"], dev["E"], out) == 0, \
            lib.dartree_last_error(None).decode()
        ref = ctx.state_step(S, tok, dev["A"], dev["E"])
        ctx.sync()
        got, want = _as_f32(out), _as_f32(ref)
        # same tolerance as the state-step parity test: one bf16 rounding
        # step (split-K partial sums may be added in another grouping) plus
        # 2e-5 absolute near zero
        ulp = np.spacing(np.abs(want)) * 2 ** 16
        assert np.all(np.abs(got - want) <= ulp + 2e-5)
        assert np.count_nonzero(got != want) <= 0.01 * M * H
    ctx.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = dtl.load()
    one = torch.zeros(64, dtype=torch.int16, device="cuda")
    p = ctypes.c_void_p(one.data_ptr())
    for H, M in ((4160, 8), (256, 257)):
        s = lib.dartree_state_step_noalloc(p, p, p, p, H, M, p, None)
        assert s == 2                        # DARTREE_ERR_UNSUPPORTED
        assert "4096" in lib.dartree_last_error(None).decode()
    assert lib.dartree_state_step_noalloc(p, p, p, p, 100, 8, p, None) == 1
