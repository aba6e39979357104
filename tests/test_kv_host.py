"""The KV-block allocator of libpw.so (host only, no GPU) against the oracle's accounting:
the hand-worked sequence, random operation streams (every count, id and error equal), bad
arguments, and the planner loop closed through it -- the planner reads F_blk from the
allocator, its plan changes the weight bytes, and the pages an offload retires come back as
free blocks (PagedWeight Sec. 3.2 Eq. 7, Sec. 3.3)."""
import json
import os

import numpy as np
import pytest

from oracle import ap
from oracle import kv as okv
from oracle import planner as opl

pw = pytest.importorskip("any_precision_bit_gb300")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_hand.json")


@pytest.fixture(scope="module", autouse=True)
def built():
    from any_precision_bit_gb300 import _build
    _build.build()


class Lib:
    """The C allocator behind the oracle's method names."""

    def __init__(self, S, B):
        self.h = pw.pw_kv_create(S, B)

    def close(self):
        pw.pw_kv_destroy(self.h)

    def set_weight_bytes(self, w):
        pw.pw_kv_set_weight_bytes(self.h, w)

    def announce(self, r, n):
        pw.pw_kv_announce(self.h, r, n)

    def grow(self, r, n):
        try:
            return [int(i) for i in pw.pw_kv_grow(self.h, r, n)]
        except pw.PwError as e:
            assert e.status == pw.PW_ERR_OOM
            raise okv.KVError("oom")

    def release(self, r):
        return pw.pw_kv_release(self.h, r)

    def request(self, r):
        return pw.pw_kv_request(self.h, r)

    def blocks(self, r):
        return [int(i) for i in pw.pw_kv_blocks(self.h, r)]

    def stats(self):
        return pw.pw_kv_get_stats(self.h)


def apply(a, op, r, n):
    try:
        if op == "weights":
            a.set_weight_bytes(n)
            return None
        if op == "announce":
            a.announce(r, n)
            return None
        if op == "grow":
            return a.grow(r, n)
        return a.release(r)
    except okv.KVError:
        return "error"


def test_hand_worked_sequence_through_the_abi():
    g = json.load(open(GOLDEN))
    a = Lib(g["budget_bytes"], g["block_bytes"])
    try:
        for k, step in enumerate(g["steps"]):
            n = step.get("bytes", step.get("n", 0))
            out = apply(a, step["op"], step.get("request", 0), n)
            assert (out == "error") == step.get("error", False), k
            if "ids" in step:
                assert out == step["ids"], k
            if "released" in step:
                assert out == step["released"], k
            st = a.stats()
            for key, val in step["expect"].items():
                assert st[key] == val, (k, key)
            if "D" in step:
                assert opl.target_bytes(g["T_blk"], st["free_blocks"], g["block_bytes"]) == step["D"]
    finally:
        a.close()


@pytest.mark.parametrize("S,B,seed", [(64 * 4096 + 123, 4096, 0), (1 << 40, 2 << 20, 1), (5000, 7, 2), (0, 64, 3)])
def test_random_streams_match_the_oracle(S, B, seed):
    rng = np.random.default_rng(seed)
    ref, lib = okv.KVAllocator(S, B), Lib(S, B)
    n_ids = S // B
    try:
        for _ in range(4000):
            op = ["weights", "announce", "grow", "grow", "release"][int(rng.integers(0, 5))]
            r = int(rng.integers(-3, 9)) * 1_000_003  # any int64 key
            if op == "weights":
                n = int(rng.integers(0, S + 3 * B + 1))
            else:
                n = int(rng.integers(0, max(2, min(40, n_ids // 4 + 2))))
            assert apply(lib, op, r, n) == apply(ref, op, r, n)
            assert lib.stats() == ref.stats()
            assert lib.request(r) == ref.request(r)
            assert lib.blocks(r) == ref.blocks(r)
    finally:
        lib.close()


def test_bad_arguments_change_nothing():
    for S, B in ((-1, 8), (100, 0), (100, -4), ((1 << 31) * 8, 8)):
        with pytest.raises(pw.PwError) as e:
            pw.pw_kv_create(S, B)
        assert e.value.status == pw.PW_ERR_INVALID
    a = Lib(1000, 10)
    try:
        a.grow(1, 3)
        before = a.stats()
        for call in (lambda: pw.pw_kv_set_weight_bytes(a.h, -1), lambda: pw.pw_kv_announce(a.h, 1, -2),
                     lambda: pw.pw_kv_grow(a.h, 1, -1)):
            with pytest.raises(pw.PwError) as e:
                call()
            assert e.value.status == pw.PW_ERR_INVALID
        assert a.stats() == before and a.blocks(1) == [0, 1, 2]
        with pytest.raises(okv.KVError):
            a.grow(2, 98)  # 97 free
        assert a.stats() == before
        assert a.release(12345) == 0 and a.request(12345) == (0, 0)
    finally:
        a.close()


# ---------------------------------------------------------------- the planner loop
def _problem(rng, E=6, L=2, bits=(3, 4, 5, 6)):
    n = L * E * 2
    q = np.full(n, bits[-1])
    utype = np.arange(n) % 2
    expert = (np.arange(n) // 2) % E
    layer = np.arange(n) // 2 // E
    N = np.where(utype == 0, 256, 128)
    M = np.array([[ap.block_bytes(int(N[i]), 512, bits, b) for b in bits] for i in range(n)], dtype=np.float64)
    return list(bits), q, q.copy(), utype, layer, expert, M, L, E


def _weight_bytes(bits, q, M):
    return int(sum(M[i, bits.index(int(q[i]))] for i in range(len(q))))


def _oracle_plan(bits, q, q_init, utype, layer, expert, M, mass, phi, off, T_blk, F, B_KV, R):
    blocks = opl.Blocks(bits, q, utype, layer, expert, M, off["s"])
    _, chosen, D = opl.plan_step(blocks, mass, phi, off, off["n_stages"], T_blk, F, B_KV)
    if D > 0:
        _, plan, _ = chosen
        return D, [(i, a, b, d) for i, (a, b, d) in plan.items()]
    plan, _ = opl.reload_plan(blocks, q_init, mass, phi, off, T_blk, F, B_KV, R)
    return D, [(i, a, b, d) for i, (a, b, d) in plan.items()]


@pytest.mark.parametrize("seed", range(3))
def test_planner_loop_closed_through_the_allocator(seed):
    """Requests arrive, grow, announce their next growth and finish; every step the planner
    reads F_blk from the allocator, and its plan, applied, sets the weight bytes the
    allocator shares the budget with.  The C path (allocator + pw_plan_host) and the oracle
    (its accounting + its planner) step together.  An offload plan that meets D restores the
    reserve (F_blk >= T_blk + 1 right after it) and a reload plan keeps F_blk >= T_blk + R."""
    from synthetic import gen_planner_offline_np
    rng = np.random.default_rng(seed)
    bits, q, q_init, utype, layer, expert, M, L, E = _problem(rng)
    n = len(q)
    off = gen_planner_offline_np(n, list(range(len(bits))), 4, seed)
    off["n_stages"] = 3
    mass = rng.dirichlet(np.ones(E), size=L)
    phi = np.abs(rng.normal(1.0, 0.5, size=(n, 3)))
    T_blk, R = 4, 2
    B_KV = int(M[0, -1] - M[0, -2])  # one level of a gate_up block per KV block
    full = _weight_bytes(bits, q, M)
    S = full + 12 * B_KV
    lib, ref = Lib(S, B_KV), okv.KVAllocator(S, B_KV)
    q_c, q_o = q.copy(), q.copy()
    live = {}
    kinds = set()
    try:
        for step in range(120):
            # the requests' side: arrivals, growth, announcements, completions
            if rng.random() < 0.35:
                r, n0 = step, int(rng.integers(1, 4))
                out = apply(lib, "grow", r, n0)
                assert out == apply(ref, "grow", r, n0)
                if out != "error":
                    live[r] = n0
            for r in list(live):
                u = rng.random()
                if u < 0.1:
                    assert apply(lib, "release", r, 0) == apply(ref, "release", r, 0)
                    del live[r]
                elif u < 0.5:
                    assert apply(lib, "grow", r, 1) == apply(ref, "grow", r, 1)
                else:
                    k = int(rng.integers(0, 3))
                    apply(lib, "announce", r, k)
                    apply(ref, "announce", r, k)
            assert lib.stats() == ref.stats()
            # the planner reads F_blk, the plan is applied, the weights' bytes go back
            F = lib.stats()["free_blocks"]
            obs = dict(T_blk=T_blk, F_blk=F, B_KV=float(B_KV), R=R, mass=mass, phi=phi)
            got = pw.pw_plan_host(bits, q_c, q_init, utype, layer, expert, M, L, E, obs, off)
            D, want = _oracle_plan(bits, q_o, q_init, utype, layer, expert, M, mass, phi, off, T_blk, F, B_KV, R)
            assert got["D"] == D and got["entries"] == want
            for i, a, b, _ in got["entries"]:
                q_c[i] = b
            for i, a, b, _ in want:
                q_o[i] = b
            lib.set_weight_bytes(_weight_bytes(bits, q_c, M))
            ref.set_weight_bytes(_weight_bytes(bits, q_o, M))
            kinds.add(got["kind"])
            if got["kind"] == 1 and got["total"] >= D:
                assert lib.stats()["free_blocks"] >= T_blk + 1
            if got["kind"] == 2:  # restored bytes fit in (F_blk - T_blk - R) B_KV
                assert lib.stats()["free_blocks"] >= T_blk + R
        assert {1, 2} <= kinds  # pressure met by offloads, and slack returned by reloads
    finally:
        lib.close()


def test_batch_merge_weighted_by_the_allocator():
    """F4 fed by F1: the batch-level table merges each live request's signals with the KV
    blocks the allocator says it holds (Sec. 3.2, batched serving), and equals the oracle's
    merge with its own accounting's counts."""
    rng = np.random.default_rng(11)
    L, E, n, nb = 2, 6, 24, 4
    S, B = 1 << 30, 1 << 20
    lib, ref = Lib(S, B), okv.KVAllocator(S, B)
    try:
        live = list(range(5))
        for r in live:
            k = int(rng.integers(1, 30))
            assert apply(lib, "grow", r, k) == apply(ref, "grow", r, k)
        assert apply(lib, "release", 2, 0) == apply(ref, "release", 2, 0)
        live.remove(2)
        reqs = [dict(mass=rng.dirichlet(np.ones(E), size=L), rho_hat=rng.normal(0, 1, (n, nb - 1)),
                     conf=rng.uniform(0.5, 1.0, (2, nb - 1)), rho_min=float(rng.uniform(-3, -1)),
                     rho_max=float(rng.uniform(1, 3))) for _ in live]
        w_c = [float(lib.request(r)[0]) for r in live]
        w_o = [float(ref.request(r)[0]) for r in live]
        assert w_c == w_o and all(w > 0 for w in w_c)
        got = pw.pw_merge_requests(reqs, w_c, L, E, n, nb)
        want = opl.merge_request_signals(reqs, w_o)
        for key in ("mass", "rho_hat", "conf", "rho_min", "rho_max"):
            assert np.array_equal(np.asarray(got[key]), np.asarray(want[key])), key
    finally:
        lib.close()


def test_request_schedule_is_well_formed():
    """The seeded serving schedule that drives the paging run: each request arrives once (at
    the step that is its id), every growth was announced the step before, nothing follows a
    finish, and the live demand rises from zero, peaks and drains."""
    from synthetic import gen_kv_requests
    steps = 200
    sched = gen_kv_requests(steps, 0)
    seen, done, announced, live, demand = set(), set(), {}, {}, []
    for t, events in enumerate(sched):
        for ev in events:
            kind, r = ev[0], ev[1]
            assert r not in done
            if kind == "arrive":
                assert r == t and r not in seen
                seen.add(r)
                live[r] = ev[2]
            elif kind == "finish":
                assert r in seen
                done.add(r)
                live.pop(r)
            elif kind == "announce":
                assert r in seen
                announced[r] = (t, ev[2])
            else:
                assert kind == "grow" and announced.get(r) == (t - 1, ev[2])
                live[r] += ev[2]
        demand.append(sum(live.values()))
    assert len(seen) > 30 and demand[0] == 0
    peak = int(np.argmax(demand))
    assert 0.3 * steps < peak < 0.7 * steps and demand[-1] < 0.2 * demand[peak]


def test_request_schedule_served_through_the_allocator():
    """The paging run's serving loop on the CPU: the seeded request schedule served by the C
    allocator and by the oracle's accounting in step (a request whose arrival or growth does
    not fit is dropped), the planner reading F_blk from the allocator every step and its
    plan setting the weight bytes (offloads retire one step later, as pages do once their
    copy has landed).  Both planners (pw_plan_host and the oracle's) agree at every step; the
    demand peak drives offloads and the drain reloads."""
    from synthetic import gen_kv_requests, gen_planner_offline_np
    rng = np.random.default_rng(5)
    bits, q, q_init, utype, layer, expert, M, L, E = _problem(rng)
    n = len(q)
    off = gen_planner_offline_np(n, list(range(len(bits))), 4, 5)
    off["n_stages"] = 3
    mass = rng.dirichlet(np.ones(E), size=L)
    phi = np.abs(rng.normal(1.0, 0.5, size=(n, 3)))
    T_blk, R, steps = 4, 2, 200
    schedule = gen_kv_requests(steps, 0)
    live, peak = {}, 0
    for events in schedule:
        for ev in events:
            if ev[0] == "finish":
                live.pop(ev[1])
            elif ev[0] in ("arrive", "grow"):
                live[ev[1]] = live.get(ev[1], 0) + ev[2]
        peak = max(peak, sum(live.values()))
    full = _weight_bytes(bits, q, M)
    B_KV = int(0.3 * full / peak)
    S = full + (T_blk + R) * B_KV
    lib, ref = Lib(S, B_KV), okv.KVAllocator(S, B_KV)
    q_c, pending, dropped, kinds, weights = q.copy(), [], set(), [], []
    try:
        for step in range(steps):
            for i, b in pending:  # offloads retire at the next step's commit
                q_c[i] = b
            pending = []
            w = _weight_bytes(bits, q_c, M)
            lib.set_weight_bytes(w)
            ref.set_weight_bytes(w)
            for ev in schedule[step]:
                kind, r = ev[0], ev[1]
                if r in dropped:
                    continue
                if kind == "finish":
                    assert apply(lib, "release", r, 0) == apply(ref, "release", r, 0)
                elif kind == "announce":
                    apply(lib, "announce", r, ev[2])
                    apply(ref, "announce", r, ev[2])
                else:
                    out = apply(lib, "grow", r, ev[2])
                    assert out == apply(ref, "grow", r, ev[2])
                    if out == "error":
                        dropped.add(r)
                        apply(lib, "release", r, 0)
                        apply(ref, "release", r, 0)
            assert lib.stats() == ref.stats()
            F = lib.stats()["free_blocks"]
            obs = dict(T_blk=T_blk, F_blk=F, B_KV=float(B_KV), R=R, mass=mass, phi=phi)
            got = pw.pw_plan_host(bits, q_c, q_init, utype, layer, expert, M, L, E, obs, off)
            D, want = _oracle_plan(bits, q_c, q_init, utype, layer, expert, M, mass, phi, off, T_blk, F, B_KV, R)
            assert got["D"] == D and got["entries"] == want, step
            kinds.append(got["kind"])
            for i, a, b, _ in got["entries"]:
                if b < a:
                    pending.append((i, b))
                else:
                    q_c[i] = b
            weights.append(_weight_bytes(bits, q_c, M))
        assert 1 in kinds and 2 in kinds
        assert min(weights) < 0.85 * full and weights[-1] > min(weights)
        assert len(dropped) <= 0.25 * len({ev[1] for evs in schedule for ev in evs})
    finally:
        lib.close()
