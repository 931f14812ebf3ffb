"""Pins for the oracle's verification consumer (no GPU): tree attention over
prefix + draft tree with the emitted mask, and the longest accepted prefix.

Tied to closed forms (self-only masks return the node's own value, equal
keys average the visible values), to a torch fp64 causal attention (a chain
tree is an ordinary causal sequence), to plain softmax attention for the
root row, and to brute-force path enumeration for acceptance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle


def _rand(g, shape):
    return g.standard_normal(shape).astype(np.float32)


def _chain_mask(B):
    words = (B + 31) // 32
    m = np.zeros((B, words), np.uint32)
    for i in range(B):
        for j in range(i + 1):
            m[i, j // 32] |= np.uint32(1 << (j % 32))
    return m


def test_self_only_mask_returns_own_value():
    g = np.random.default_rng(1)
    B, Hq, Hkv, dh = 5, 4, 2, 8
    Q, Kt, Vt = _rand(g, (B + 1, Hq, dh)), _rand(g, (B, Hkv, dh)), _rand(g, (B, Hkv, dh))
    empty = np.zeros((0, Hkv, dh), np.float32)
    mask = np.zeros((B, 1), np.uint32)
    for i in range(B):
        mask[i, 0] = 1 << i
    O = oracle.tree_attention(Q, empty, empty, Kt, Vt, mask, 0.3, False)
    assert np.all(O[0] == 0)                       # the root sees no key at all
    for i in range(1, B + 1):
        for h in range(Hq):
            assert np.allclose(O[i, h], Vt[i - 1, h // 2], atol=1e-6, rtol=0)


def test_chain_tree_is_causal_attention():
    g = np.random.default_rng(2)
    Lp, B, Hq, Hkv, dh = 7, 6, 4, 2, 16
    Kp, Vp = _rand(g, (Lp, Hkv, dh)), _rand(g, (Lp, Hkv, dh))
    Kt, Vt = _rand(g, (B, Hkv, dh)), _rand(g, (B, Hkv, dh))
    Q = _rand(g, (B + 1, Hq, dh))
    scale = 1 / np.sqrt(dh)
    O = oracle.tree_attention(Q, Kp, Vp, Kt, Vt, _chain_mask(B), scale, False)
    # the sequence prefix + chain; query row i sits at position Lp - 1 + i
    K = torch.from_numpy(np.concatenate([Kp, Kt])).double().repeat_interleave(Hq // Hkv, 1)
    V = torch.from_numpy(np.concatenate([Vp, Vt])).double().repeat_interleave(Hq // Hkv, 1)
    q = torch.from_numpy(Q).double()
    s = torch.einsum("ihc,jhc->hij", q, K) * scale
    pos = torch.arange(B + 1)[:, None] + Lp - 1
    s = s.masked_fill(torch.arange(Lp + B)[None, :] > pos, float("-inf"))
    ref = torch.einsum("hij,jhc->ihc", torch.softmax(s, -1), V).numpy()
    assert np.allclose(O, ref, atol=1e-5, rtol=0)


def test_root_row_is_plain_attention_over_the_prefix_and_bf16_widening():
    g = np.random.default_rng(3)
    Lp, B, Hq, Hkv, dh = 11, 4, 2, 1, 8
    from speculative_decoding_draft_06_gb300.inputs import to_bf16_bits, bf16_bits_to_f32
    arrs = [to_bf16_bits(_rand(g, s)) for s in [(B + 1, Hq, dh), (Lp, Hkv, dh), (Lp, Hkv, dh),
                                                (B, Hkv, dh), (B, Hkv, dh)]]
    mask = g.integers(0, 2 ** 4, (B, 1)).astype(np.uint32)
    O = oracle.tree_attention(*arrs, mask, 0.5, True)
    Q, Kp, Vp = (torch.from_numpy(bf16_bits_to_f32(a)).double() for a in arrs[:3])
    for h in range(Hq):
        w = torch.softmax(0.5 * (Kp[:, 0] @ Q[0, h]), 0)
        assert np.allclose(O[0, h], (w @ Vp[:, 0]).numpy(), atol=1e-6, rtol=0)


def test_equal_keys_average_the_visible_values():
    g = np.random.default_rng(4)
    Lp, B, Hq, Hkv, dh = 3, 9, 2, 2, 4
    k = _rand(g, dh)
    Kp = np.broadcast_to(k, (Lp, Hkv, dh)).copy()
    Kt = np.broadcast_to(k, (B, Hkv, dh)).copy()
    Vp, Vt, Q = _rand(g, (Lp, Hkv, dh)), _rand(g, (B, Hkv, dh)), _rand(g, (B + 1, Hq, dh))
    mask = g.integers(0, 2 ** 9, (B, 1)).astype(np.uint32)
    O = oracle.tree_attention(Q, Kp, Vp, Kt, Vt, mask, 1.0, False)
    for i in range(1, B + 1):
        vis = [Vp[j] for j in range(Lp)] + [Vt[j] for j in range(B) if mask[i - 1, 0] >> j & 1]
        assert np.allclose(O[i], np.mean(vis, axis=0), atol=1e-6, rtol=0)


# ---------------------------------------------------------------- accept

def test_accept_hand_example():
    # ranks: 0 'a'(root child), 1 'b'(root child), 2 'c'(child of 0), 3 'd'(child of 0),
    #        4 'e'(child of 3); tokens a=10, b=11, c=12, d=13, e=14
    parent = np.array([-1, -1, 0, 0, 3, -1], np.int32)
    token = np.array([10, 11, 12, 13, 14, -1], np.int32)
    pred = np.array([10, 13, 99, 99, 14, 77, 0], np.int32)   # root->a, a->d, d->e, e->77
    r = oracle.accept(parent, token, 5, pred)
    assert r["len"] == 3 and list(r["nodes"]) == [0, 3, 4] and r["bonus"] == 77
    pred[0] = 5                                             # the first token is rejected
    r = oracle.accept(parent, token, 5, pred)
    assert r["len"] == 0 and r["bonus"] == 5
    r = oracle.accept(parent, token, 3, np.array([10, 13, 0, 0, 0, 0, 0], np.int32))
    assert r["len"] == 1 and r["bonus"] == 13               # node 3 is beyond n_out


@pytest.mark.parametrize("seed", range(6))
def test_accept_equals_bruteforce_paths(seed):
    g = np.random.default_rng(100 + seed)
    B = 40
    parent = np.full(B, -1, np.int32)
    token = np.empty(B, np.int32)
    for n in range(B):
        parent[n] = -1 if n < 3 or g.random() < 0.1 else g.integers(0, n)
    for n in range(B):                                      # distinct tokens among siblings
        sib = [m for m in range(n) if parent[m] == parent[n]]
        token[n] = len(sib) + 10 * (parent[n] + 1)
    n_out = int(g.integers(B // 2, B + 1))
    pred = np.empty(B + 1, np.int32)
    for u in range(-1, B):                                  # mostly agree with some child
        kids = [m for m in range(B) if parent[m] == u]
        pred[u + 1] = token[g.choice(kids)] if kids and g.random() < 0.8 else 10 ** 6 + u
    r = oracle.accept(parent, token, n_out, pred)
    best = []
    for n in range(n_out):                                  # every path, checked from scratch
        path, u = [], n
        while u >= 0:
            path.append(u)
            u = parent[u]
        path.reverse()
        ok = all(token[v] == pred[(parent[v] + 1)] for v in path)
        if ok and len(path) > len(best):
            best = path
    assert r["len"] == len(best) and list(r["nodes"]) == best
    last = best[-1] if best else -1
    assert r["bonus"] == pred[last + 1]
