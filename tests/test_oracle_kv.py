"""Pins of the oracle's KV-block accounting (CPU only): the hand-worked sequence of
kv_hand.json, closed forms, and invariants over random operation sequences."""
import json
import os

import numpy as np
import pytest

from oracle import kv as okv
from oracle import planner as opl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_hand.json")


def replay(alloc, step):
    """Apply one golden step; returns (ids or released count or None, error raised)."""
    op = step["op"]
    try:
        if op == "weights":
            alloc.set_weight_bytes(step["bytes"])
            return None, False
        if op == "announce":
            alloc.announce(step["request"], step["n"])
            return None, False
        if op == "grow":
            return alloc.grow(step["request"], step["n"]), False
        if op == "release":
            return alloc.release(step["request"]), False
    except okv.KVError:
        return None, True
    raise ValueError(op)


def test_hand_worked_sequence():
    g = json.load(open(GOLDEN))
    a = okv.KVAllocator(g["budget_bytes"], g["block_bytes"])
    for k, step in enumerate(g["steps"]):
        out, err = replay(a, step)
        assert err == step.get("error", False), k
        if "ids" in step:
            assert out == step["ids"], k
        if "released" in step:
            assert out == step["released"], k
        st = a.stats()
        for key, val in step["expect"].items():
            assert st[key] == val, (k, key, st[key], val)
        if "D" in step:
            assert opl.target_bytes(g["T_blk"], st["free_blocks"], g["block_bytes"]) == step["D"], k


@pytest.mark.parametrize("S,B", [(10 << 20, 1 << 20), (7_000_001, 65_536), (0, 4096)])
def test_free_blocks_follow_the_released_pages(S, B):
    """With no requests F_blk = floor((S - W) / B) (0 once W >= S): retiring d bytes of pages
    frees exactly floor((S - W + d) / B) - floor((S - W) / B) more blocks."""
    a = okv.KVAllocator(S, B)
    rng = np.random.default_rng(1)
    for _ in range(200):
        W = int(rng.integers(0, S + 3 * B + 1))
        d = int(rng.integers(0, 4 * B))
        a.set_weight_bytes(W)
        f0 = a.free_blocks()
        assert f0 == (max(0, S - W) // B)
        a.set_weight_bytes(max(0, W - d))
        assert a.free_blocks() - f0 == max(0, S - max(0, W - d)) // B - max(0, S - W) // B
        assert a.headroom() == S - max(0, W - d)


def test_random_sequences_keep_the_invariants():
    rng = np.random.default_rng(7)
    S, B = 64 * 4096 + 123, 4096
    a = okv.KVAllocator(S, B)
    for _ in range(3000):
        before = (a.stats(), {r: list(v) for r, v in a.held.items()}, dict(a.announced))
        op = rng.integers(0, 4)
        r = int(rng.integers(0, 6))
        n = int(rng.integers(0, 9))
        if op == 0:
            a.set_weight_bytes(int(rng.integers(0, S + B)))
        elif op == 1:
            a.announce(r, n)
        elif op == 2:
            own = a.announced.get(r, 0)
            ok = n - min(n, own) <= a.free_blocks()
            free_before = sorted(a.free_ids)
            try:
                ids = a.grow(r, n)
                assert ok
                assert ids == free_before[:n]  # the lowest free ids, by brute force
                assert a.used() <= a.capacity()
            except okv.KVError:
                assert not ok
                assert (a.stats(), a.held, a.announced) == before
        else:
            held = list(a.held.get(r, []))
            assert a.release(r) == len(held)
            assert set(held) <= a.free_ids
        st = a.stats()
        assert st["free_blocks"] == st["capacity_blocks"] - st["used_blocks"] - st["pending_blocks"]
        assert st["headroom_bytes"] == S - st["weight_bytes"] - st["used_blocks"] * B
        taken = [i for v in a.held.values() for i in v]
        assert len(taken) == len(set(taken)) == st["used_blocks"]
        assert all(0 <= i < S // B for i in taken)
        assert not (set(taken) & a.free_ids) and len(taken) + len(a.free_ids) == S // B


def test_bad_arguments():
    with pytest.raises(okv.KVError):
        okv.KVAllocator(100, 0)
    a = okv.KVAllocator(100, 10)
    for call in (lambda: a.set_weight_bytes(-1), lambda: a.announce(0, -1), lambda: a.grow(0, -1)):
        with pytest.raises(okv.KVError):
            call()
