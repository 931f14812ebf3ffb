"""The C ABI library builds, loads and exports what include/dartree.h
declares; host-side logic that needs no GPU."""
from __future__ import annotations

import ctypes

import pytest
import torch

from speculative_decoding_draft_06_gb300 import build as cuda_build
from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return dtl.load()


def test_every_declared_symbol_is_exported(lib):
    names = dtl.declared_symbols()
    assert "dartree_build" in names and "dartree_create" in names
    for n in names:
        assert hasattr(lib, n), n


def test_pool_size_host_logic(lib):
    for name, w in I.CONFIGS.items():
        assert dtl.pool_size(w.D, w.W, w.K) == w.pool_size(), name
    assert dtl.pool_size(16, 64, 32) == 992
    assert dtl.pool_size(0, 4, 4) == -1
    assert dtl.frontier_sizes(4, 10, 3) == [3, 9, 10, 10]


def test_workload_closed_forms():
    w = I.CONFIGS["q8b"]
    assert w.head_rows() == [1] + [16] * 15
    assert w.candidates_per_build() == 3856
    assert I.CONFIGS["batch"].candidates_per_build() == 30976
    assert I.CONFIGS["wide"].candidates_per_build() == 29728
    assert I.CONFIGS["tiny"].candidates_per_build() == 116


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_create_fails_cleanly_without_a_gpu(lib):
    cfg = dtl.Config(1000, 64, 4, 4, 4, 8, 1, dtl.W_BF16)
    h = ctypes.c_void_p()
    s = lib.dartree_create(ctypes.byref(cfg), ctypes.byref(h))
    assert s != 0 and not h.value


def test_create_rejects_bad_configs_before_touching_the_device(lib):
    bad = [dtl.Config(1000, 60, 4, 4, 4, 8, 1, dtl.W_BF16),     # H % 64 != 0
           dtl.Config(1000, 64, 4, 4, 33, 8, 1, dtl.W_BF16),    # K > 32
           dtl.Config(1000, 64, 4, 64, 4, 8, 8, dtl.W_BF16),    # R * W > 256
           dtl.Config(1000, 64, 4, 257, 4, 8, 1, dtl.W_BF16),   # W > 256
           dtl.Config(1000, 64, 33, 4, 4, 8, 1, dtl.W_BF16),    # D > 32
           dtl.Config(1000, 64, 4, 4, 4, 1025, 1, dtl.W_BF16),  # B > 1024
           dtl.Config(0, 64, 4, 4, 4, 8, 1, dtl.W_F32),
           dtl.Config(1000, 64, 4, 4, 4, 8, 1, 7)]
    for cfg in bad:
        h = ctypes.c_void_p()
        assert lib.dartree_create(ctypes.byref(cfg), ctypes.byref(h)) in (1, 2)
        assert not h.value


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(dtl, "_lib", None)
    monkeypatch.setattr(dtl, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        dtl.load()


def test_blocked_weight_layout_host_checks(lib):
    """The blocked layout's size (ceil(V/128) 128 H bf16 elements) and the
    argument checks of dartree_block_weights / dartree_set_weight_layout,
    which return before any device call."""
    assert lib.dartree_blocked_weight_bytes(151936, 4096) == 151936 * 4096 * 2
    assert lib.dartree_blocked_weight_bytes(1000, 64) == 1024 * 64 * 2
    assert lib.dartree_blocked_weight_bytes(129, 128) == 256 * 128 * 2
    for V, H in ((0, 64), (100, 0), (100, 100), (-1, 64)):
        assert lib.dartree_blocked_weight_bytes(V, H) == 0
    a, b = ctypes.c_void_p(0x10000000), ctypes.c_void_p(0x20000000)
    bad = [(None, 100, 64, b),                              # null source
           (a, 100, 64, None),                              # null destination
           (a, 100, 100, b),                                # H not a multiple of 64
           (ctypes.c_void_p(0x10000008), 100, 64, b),       # misaligned
           (a, 1000, 64, ctypes.c_void_p(0x10000000 + 4096))]  # overlapping
    for W, V, H, out in bad:
        assert lib.dartree_block_weights(W, V, H, out, None) == 1  # INVALID_ARG
        assert lib.dartree_last_error(None)
    assert lib.dartree_set_weight_layout(None, 1) == 1
