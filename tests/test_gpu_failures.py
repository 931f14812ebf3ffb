"""Failure detection on the GPU without faulting it.

A device-side wait that runs out reports DARTREE_ERR_TIMEOUT through
dartree_sync_status and leaves the CUDA context usable; bad data (a base
logit row with no finite entry) is caught by the kernels' own checks and
reported as DARTREE_ERR_DEVICE_CHECK.  The timeout is provoked by giving the
pipeline waits a limit of one cycle (a test knob read at context creation);
waits for copies and MMAs already in flight keep the full limit, so the
kernels drain before they exit.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

from speculative_decoding_draft_06_gb300 import dartree as dtl
from speculative_decoding_draft_06_gb300 import inputs as I
from tests import gpu_util as gu
from tests import parity

pytestmark = pytest.mark.gpu

TIMEOUT, DEVICE_CHECK = 5, 4


def _small():
    w = I.small_workload(91, V=3000, H=128, D=3, W=8, K=8, B=16, beta=-0.1, bf16=True)
    return w, I.make_inputs(w)


@pytest.mark.parametrize("shape", ["tc", "rows", "pair"])
def test_wait_timeout_is_reported_and_context_stays_usable(monkeypatch, shape):
    """Every head kernel: the vocabulary-on-M kernel (8 rows), the row-major
    kernel (64 rows) and the CTA-pair kernel (160 rows)."""
    w = {"tc": I.small_workload(91, V=3000, H=128, D=3, W=8, K=8, B=16, beta=-0.1, bf16=True),
         "rows": I.small_workload(92, V=3000, H=128, D=3, W=64, K=8, B=40, beta=-0.1, bf16=True),
         "pair": I.small_workload(93, V=3000, H=128, D=3, W=8, K=8, B=16, beta=-0.1, bf16=True,
                                  R=20)}[shape]
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, True)
    monkeypatch.setenv("DARTREE_WAIT_LIMIT_CYCLES", "1")
    ctx = gu.make_ctx(w)
    monkeypatch.delenv("DARTREE_WAIT_LIMIT_CYCLES")
    ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W, K=w.K,
              B=w.B, beta=w.beta)
    assert ctx.sync_status() == TIMEOUT
    ctx.close()
    # same process, same device: a normal context builds correctly
    ctx = gu.make_ctx(w)
    res = gu.run_build(ctx, w, dev)
    for r in range(w.R):
        pool, rows, tree = gu.split_request(res, w, r)
        parity.compare_request(inp, r, w.D, w.W, w.K, w.B, w.beta, True, pool, rows, tree)
    ctx.close()


def test_row_without_finite_logits_is_a_device_check():
    w, inp = _small()
    inp["z"][0, 1, :] = np.nan              # depth 2: every logit of every row NaN
    dev = dtl.weights_to_device(inp, True)
    ctx = gu.make_ctx(w)
    ctx.build(dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W, K=w.K,
              B=w.B, beta=w.beta)
    assert ctx.sync_status() == DEVICE_CHECK
    assert ctx.sync_status() == 0
    ctx.close()
