"""Pins for the oracle's KV ring append and f16 K/V store.

Pinned against: the ring-wrap walk printed in the Muser book (Ch 15 §15.5,
Figure 15.2), the boundary positions it names (§15.9), the fail-closed
continuity rule, brute-force enumeration of the two index formulas (§15.3), and
numpy's binary16 conversion.

The snapshot and the rotation-preserving restore (§15.6; Ch 10 §10.7) are
pinned by brute force on the rows they must hold, and by the book's own
criterion: a window restored at origin o and then appended to holds exactly
what a ring built by sequential appends holds (same metadata, same bytes in
every live slot), while the slots outside the window stay untouched.
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


# ------------------------------------------------ snapshot and restore (§15.6)
CASES = [(8, 6, 3, False), (8, 6, 3, True), (5, 4, 2, True), (16, 8, 8, False)]


def _f16(a):
    return np.asarray(a, np.float32).astype(np.float16).view(np.uint16)


def _append_chunks(ring, key, val, kv_dim, head_dim, head_major, k, v, pos0, chunks):
    t = 0
    for c in chunks:
        rc, _ = oracle.kv_write(ring, key, val, kv_dim, head_dim, head_major, k[t:t + c], v[t:t + c],
                                pos0 + t)
        assert rc == 0
        t += c
    assert t == k.shape[0]


def _sequential_plane(cap, kv_dim, head_dim, head_major, ntok, seed=3, fill=0xDEAD):
    key = np.full(cap * kv_dim, fill, np.uint16)
    val = np.full(cap * kv_dim, fill, np.uint16)
    ring = oracle.Ring(cap, 0, 0, 0)
    k, v = synth.kv_rows(ntok, kv_dim, seed=seed)
    chunks = [c for c in (1, 3, 2, 7, 1, 5, 11, 4) * 8]
    out, t = [], 0
    for c in chunks:
        if t >= ntok:
            break
        out.append(min(c, ntok - t))
        t += out[-1]
    _append_chunks(ring, key, val, kv_dim, head_dim, head_major, k, v, 0, out)
    return ring, key, val, k, v


@pytest.mark.parametrize("cap,kv_dim,head_dim,head_major", CASES)
@pytest.mark.parametrize("ntok", [0, 3, 8, 11, 29])
def test_snapshot_rows_brute_force(cap, kv_dim, head_dim, head_major, ntok):
    ntok = ntok * cap // 8
    ring, key, val, k, v = _sequential_plane(cap, kv_dim, head_dim, head_major, ntok)
    live0 = ring.origin_logical
    assert live0 == max(0, ntok - cap) and ring.len == min(ntok, cap)
    # every sub-range of the live window, logical position q holding token q
    for first in range(live0, live0 + ring.len + 1):
        for count in range(0, live0 + ring.len - first + 1):
            rc, kr, vr = oracle.kv_snapshot(ring, key, val, kv_dim, head_dim, head_major, first, count)
            assert rc == 0
            assert np.array_equal(kr, _f16(k[first:first + count]))
            assert np.array_equal(vr, _f16(v[first:first + count]))


@pytest.mark.parametrize("head_major", [False, True])
def test_snapshot_follows_origin_physical_not_position(head_major):
    # a window whose physical origin is not its logical origin modulo capacity
    cap, kv_dim, head_dim = 8, 4, 2
    key = np.zeros(cap * kv_dim, np.uint16)
    val = np.zeros(cap * kv_dim, np.uint16)
    ring = oracle.Ring(cap, 0, 100, 5)
    k, v = synth.kv_rows(6, kv_dim, seed=9)
    _append_chunks(ring, key, val, kv_dim, head_dim, head_major, k, v, 100, [2, 4])
    for j in range(6):
        slot = (5 + j) % cap
        for e in range(kv_dim):
            dst = ((e // head_dim) * cap + slot) * head_dim + e % head_dim if head_major else slot * kv_dim + e
            assert key[dst] == _f16(k[j, e])
    rc, kr, vr = oracle.kv_snapshot(ring, key, val, kv_dim, head_dim, head_major, 100, 6)
    assert rc == 0 and np.array_equal(kr, _f16(k)) and np.array_equal(vr, _f16(v))
    rc, kr, _ = oracle.kv_snapshot(ring, key, val, kv_dim, head_dim, head_major, 102, 3)
    assert rc == 0 and np.array_equal(kr, _f16(k[2:5]))


@pytest.mark.parametrize("cap,kv_dim,head_dim,head_major", CASES)
@pytest.mark.parametrize("ntok,more", [(0, 5), (3, 9), (8, 1), (11, 4), (29, 13), (64, 0)])
def test_restore_then_append_equals_sequential_ring(cap, kv_dim, head_dim, head_major, ntok, more):
    ntok = ntok * cap // 8
    live, lkey, lval, k, v = _sequential_plane(cap, kv_dim, head_dim, head_major, ntok + more)
    # the live ring as it stood after ntok tokens, and its detached window
    a, akey, aval, _, _ = _sequential_plane(cap, kv_dim, head_dim, head_major, ntok)
    rc, kr, vr = oracle.kv_snapshot(a, akey, aval, kv_dim, head_dim, head_major, a.origin_logical, a.len)
    assert rc == 0
    # restore into a fresh plane, then continue appending the same tokens
    bkey = np.full(cap * kv_dim, 0xBEEF, np.uint16)
    bval = np.full(cap * kv_dim, 0xBEEF, np.uint16)
    b = oracle.Ring(cap, 0, 0, 0)
    assert oracle.kv_restore(b, bkey, bval, kv_dim, head_dim, head_major, kr, vr, a.origin_logical) == 0
    assert (b.len, b.origin_logical, b.origin_physical) == (a.len, a.origin_logical, a.origin_physical)
    if more:
        _append_chunks(b, bkey, bval, kv_dim, head_dim, head_major, k[ntok:], v[ntok:], ntok, [more])
    assert (b.len, b.origin_logical, b.origin_physical) == (live.len, live.origin_logical,
                                                             live.origin_physical)
    written = np.zeros(cap, bool)
    for j in range(live.len):
        written[(live.origin_physical + j) % cap] = True
    for slot in range(cap):
        for e in range(kv_dim):
            i = ((e // head_dim) * cap + slot) * head_dim + e % head_dim if head_major else slot * kv_dim + e
            if written[slot]:
                assert bkey[i] == lkey[i] and bval[i] == lval[i]
            else:
                assert bkey[i] == 0xBEEF and bval[i] == 0xBEEF


@pytest.mark.parametrize("head_major", [False, True])
def test_restore_rotation_is_origin_mod_capacity(head_major):
    cap, kv_dim, head_dim = 8, 4, 2
    rows = (np.arange(5 * kv_dim, dtype=np.uint16) + 1).reshape(5, kv_dim)
    for origin, rot in [(0, 0), (3, 3), (8, 0), (100, 4), (101, 5)]:
        key = np.zeros(cap * kv_dim, np.uint16)
        val = np.zeros(cap * kv_dim, np.uint16)
        ring = oracle.Ring(cap, 2, 7, 1)
        assert oracle.kv_restore(ring, key, val, kv_dim, head_dim, head_major, rows, rows + 100, origin) == 0
        assert (ring.len, ring.origin_logical, ring.origin_physical) == (5, origin, rot)
        for j in range(5):
            slot = (rot + j) % cap
            for e in range(kv_dim):
                i = ((e // head_dim) * cap + slot) * head_dim + e % head_dim if head_major else slot * kv_dim + e
                assert key[i] == rows[j, e] and val[i] == rows[j, e] + 100
        # a window packed at slot 0 is a different plane unless the rotation is 0
        rc, kr, _ = oracle.kv_snapshot(ring, key, val, kv_dim, head_dim, head_major, origin, 5)
        assert rc == 0 and np.array_equal(kr, rows)
        packed = np.zeros_like(key)
        for j in range(5):
            for e in range(kv_dim):
                i = ((e // head_dim) * cap + j) * head_dim + e % head_dim if head_major else j * kv_dim + e
                packed[i] = rows[j, e]
        assert np.array_equal(packed, key) == (rot == 0)


def test_snapshot_and_restore_reject_bad_ranges_and_change_nothing():
    cap, kv_dim, head_dim = 8, 4, 2
    ring, key, val, _, _ = _sequential_plane(cap, kv_dim, head_dim, True, 11)
    assert (ring.len, ring.origin_logical) == (8, 3)
    for first, count in [(2, 1), (3, 9), (10, 2), (11, 1), (0, 0), (4, -1)]:
        rc, kr, vr = oracle.kv_snapshot(ring, key, val, kv_dim, head_dim, True, first, max(count, 0))
        if count < 0:
            rc = oracle.lib().orc_kv_snapshot(oracle.ctypes.byref(ring), oracle._p(key), oracle._p(val),
                                              kv_dim, head_dim, 1, first, count, oracle._p(kr),
                                              oracle._p(vr))
        assert rc == -1 and not kr.any() and not vr.any()
    rc, _, _ = oracle.kv_snapshot(ring, key, val, kv_dim, 3, True, 3, 1)
    assert rc == -1
    before = (key.copy(), val.copy(), (ring.len, ring.origin_logical, ring.origin_physical))
    rows = np.ones((9, kv_dim), np.uint16)
    assert oracle.kv_restore(ring, key, val, kv_dim, head_dim, True, rows, rows, 0) == -1
    assert oracle.kv_restore(ring, key, val, kv_dim, head_dim, True, rows[:2], rows[:2], -1) == -1
    assert np.array_equal(key, before[0]) and np.array_equal(val, before[1])
    assert (ring.len, ring.origin_logical, ring.origin_physical) == before[2]
    # an empty window is a valid restore: it only resets the metadata
    assert oracle.kv_restore(ring, key, val, kv_dim, head_dim, True, rows[:0], rows[:0], 20) == 0
    assert (ring.len, ring.origin_logical, ring.origin_physical) == (0, 20, 4)
    assert np.array_equal(key, before[0])
