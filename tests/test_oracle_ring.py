"""Pins for the oracle's KV ring append and f16 K/V store.

Pinned against: the ring-wrap walk printed in the Muser book (Ch 15 §15.5,
Figure 15.2), the boundary positions it names (§15.9), the fail-closed
continuity rule, brute-force enumeration of the two index formulas (§15.3), and
numpy's binary16 conversion.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth


def _fill(cap, upto):
    ring = oracle.Ring(cap, 0, 0, 0)
    writes = []
    for pos in range(upto):
        rc, w = oracle.ring_append(ring, pos)
        assert rc == 0
        writes.append(w)
    return ring, writes


def test_ring_wrap_walk_from_book(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "ring_wrap_walk.json")))
    cap = g["capacity"]
    ring, writes = _fill(cap, cap)
    assert writes == list(range(cap))
    assert (ring.len, ring.origin_logical, ring.origin_physical) == (
        g["after_fill"]["len"], g["after_fill"]["origin_logical"], g["after_fill"]["origin_physical"])
    for step in g["steps"]:
        rc, w = oracle.ring_append(ring, step["position"])
        assert rc == 0
        assert (w, ring.origin_logical, ring.origin_physical) == (
            step["write"], step["origin_logical"], step["origin_physical"])


@pytest.mark.parametrize("cap", [32, 2048])
def test_ring_boundary_positions(golden_dir, cap):
    g = json.load(open(os.path.join(golden_dir, "ring_wrap_walk.json")))
    ring = oracle.Ring(cap, 0, 0, 0)
    last = max(g["boundary_positions"])
    seen = {}
    for pos in range(last + 1):
        rc, w = oracle.ring_append(ring, pos)
        assert rc == 0
        seen[pos] = w
        # the live window is always [origin_logical, origin_logical + len)
        assert ring.len == min(pos + 1, cap)
        assert ring.origin_logical == max(0, pos + 1 - cap)
    for pos in g["boundary_positions"]:
        # with a ring started at 0, a position lands at its rotation: pos % cap
        assert seen[pos] == pos % cap


def test_ring_discontinuity_is_rejected_and_changes_nothing():
    ring, _ = _fill(32, 40)
    before = (ring.len, ring.origin_logical, ring.origin_physical)
    for bad in (39, 41, 0, 1000):
        rc, _ = oracle.ring_append(ring, bad)
        assert rc == -4
        assert (ring.len, ring.origin_logical, ring.origin_physical) == before
    rc, w = oracle.ring_append(ring, 40)
    assert rc == 0 and w == 40 % 32


def test_ring_restored_origin_rotation():
    # a plane whose live window starts at logical 100 in physical slot 7
    ring = oracle.Ring(64, 64, 100, 7)
    rc, w = oracle.ring_append(ring, 164)
    assert rc == 0 and w == 7 and ring.origin_physical == 8 and ring.origin_logical == 101
    ring = oracle.Ring(64, 10, 100, 60)
    rc, w = oracle.ring_append(ring, 110)
    assert rc == 0 and w == (60 + 10) % 64 and ring.len == 11


@pytest.mark.parametrize("head_major", [False, True])
def test_kv_write_index_formulas_and_values(head_major):
    cap, kv_dim, head_dim = 8, 6, 3
    key = np.full(cap * kv_dim, 0xDEAD, np.uint16)
    val = np.full(cap * kv_dim, 0xDEAD, np.uint16)
    ring = oracle.Ring(cap, 0, 0, 0)
    k, v = synth.kv_rows(11, kv_dim, seed=2)
    rc, first = oracle.kv_write(ring, key, val, kv_dim, head_dim, head_major, k, v, 0)
    assert rc == 0 and first == 0
    # brute force: the last 8 of the 11 appended tokens are live; token t sits in slot t % 8
    kb = k.astype(np.float16).view(np.uint16)
    vb = v.astype(np.float16).view(np.uint16)
    for t in range(3, 11):
        slot = t % cap
        for e in range(kv_dim):
            dst = ((e // head_dim) * cap + slot) * head_dim + e % head_dim if head_major else slot * kv_dim + e
            assert key[dst] == kb[t, e] and val[dst] == vb[t, e]
    assert not np.any(key == 0xDEAD) and not np.any(val == 0xDEAD)
    assert (ring.len, ring.origin_logical, ring.origin_physical) == (8, 3, 3)


def test_kv_write_discontinuity_leaves_planes_untouched():
    key = np.full(4 * 2, 0xDEAD, np.uint16)
    val = key.copy()
    ring = oracle.Ring(4, 1, 5, 2)
    rc, _ = oracle.kv_write(ring, key, val, 2, 2, False, np.ones((1, 2), np.float32),
                            np.ones((1, 2), np.float32), 7)
    assert rc == -4 and np.all(key == 0xDEAD) and (ring.len, ring.origin_logical) == (1, 5)
