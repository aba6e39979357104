"""The C-ABI library loads and exports every declared symbol; host-only calls match the
oracle (packer) or its independent restatement (planner).  No GPU is touched."""
import os
import re
import subprocess

import numpy as np
import pytest

from conftest import ROOT, load_golden
from oracle import ap
from oracle import planner as opl

pw = pytest.importorskip("any_precision_bit_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    from any_precision_bit_gb300 import _build
    _build.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "pw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pw_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 25
    out = subprocess.run(["nm", "-D", "--defined-only", pw.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pw_[a-z_]+)\b", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = pw.lib()
    for n in names:
        assert hasattr(lib, n)
    assert "sm_103a" in pw.pw_version()


def test_status_codes_match_the_header():
    """The binding's status constants and names are the header's enum, value for value."""
    src = open(os.path.join(ROOT, "include", "pw.h")).read()
    enum = dict((n, int(v)) for n, v in re.findall(r"\b(PW_(?:OK|ERR_[A-Z]+))\s*=\s*(\d+)", src))
    assert enum["PW_OK"] == 0 and "PW_ERR_RANGE" in enum and "PW_ERR_TIMEOUT" in enum
    for name, value in enum.items():
        assert getattr(pw, name) == value, name
        assert value == 0 or pw.STATUS_NAMES[value] == name


def test_create_rejects_bad_shapes_without_gpu():
    d = pw.pw_desc(L=1, E=8, H=100, I=256, K=2, Is=0, bmax=6, bits_mask=0b1111000, renorm=0, device=0,
                   max_tokens=8, flags=0)
    with pytest.raises(pw.PwError) as ei:
        pw.pw_create(d)
    assert ei.value.status == pw.PW_ERR_INVALID


@pytest.mark.parametrize("N,K,bmax", [(1, 3, 3), (2, 128, 4), (5, 200, 6), (3, 1408, 8), (16, 704, 8)])
def test_plain_packer_matches_oracle(N, K, bmax):
    rng = np.random.default_rng(N * 7 + K)
    idx = rng.integers(0, 1 << bmax, size=(N, K), dtype=np.uint8)
    got = pw.pw_pack_planes_host(idx, bmax)
    want = ap.pack_planes(idx, bmax)
    assert np.array_equal(got, want)


def test_plain_packer_hand_example():
    g = load_golden("planes_hand.json")
    got = pw.pw_pack_planes_host(np.array(g["idx"], dtype=np.uint8), g["bmax"])
    assert [int(got[p, 0, 0]) for p in range(g["bmax"])] == g["plane_word0"]


@pytest.mark.parametrize("N,K,u", [(16, 128, 1), (32, 300, 0), (48, 704, 1), (64, 256, 0)])
def test_tiling_is_a_bijection(N, K, u):
    rng = np.random.default_rng(N + K + u)
    idx = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    planes = ap.pack_planes(idx, 8)
    tiled = pw.pw_tile_planes_host(planes, K, u)
    assert tiled.shape == planes.shape
    assert np.array_equal(pw.pw_untile_planes_host(tiled, K, u), planes)
    # same number of set bits per plane: a permutation of bit positions
    for p in range(8):
        assert int(np.unpackbits(planes[p].view(np.uint8)).sum()) == int(np.unpackbits(tiled[p].view(np.uint8)).sum())
    # one set bit lands exactly once
    one = np.zeros_like(planes[:1])
    one[0, N - 1, 0] = 1 << 5
    t1 = pw.pw_tile_planes_host(one, K, u)
    assert int(np.unpackbits(t1.view(np.uint8)).sum()) == 1


def _random_problem(rng, n_layers=2, E=6, bits=(3, 4, 5, 6)):
    n = n_layers * E * 2
    nb = len(bits)
    q = rng.choice(bits, size=n)
    q_init = np.maximum(q, rng.choice(bits, size=n))
    utype = np.arange(n) % 2
    expert = (np.arange(n) // 2) % E
    layer = np.arange(n) // 2 // E
    N = np.where(utype == 0, 64, 32)
    M = np.array([[ap.block_bytes(int(N[i]), 256, bits, b) for b in bits] for i in range(n)], dtype=np.float64)
    return bits, q, q_init, utype, layer, expert, M, n_layers, E


def _offline(rng, n, nb):
    from synthetic import gen_planner_offline_np
    off = gen_planner_offline_np(n, list(range(nb)), 4, int(rng.integers(1 << 30)))
    off["n_stages"] = 3
    return off


@pytest.mark.parametrize("seed", range(12))
def test_planner_matches_oracle_restatement(seed):
    rng = np.random.default_rng(seed)
    bits, q, q_init, utype, layer, expert, M, L, E = _random_problem(rng)
    n = len(q)
    off = _offline(rng, n, len(bits))
    mass = rng.dirichlet(np.ones(E), size=L)
    phi = np.abs(rng.normal(1.0, 0.5, size=(n, 3)))
    B_KV = float(M[0, 1] - M[0, 0]) * 0.7
    for F in (0, 5, 16, 17, 40):
        obs = dict(T_blk=16, F_blk=F, B_KV=B_KV, R=8, mass=mass, phi=phi)
        got = pw.pw_plan_host(bits, q, q_init, utype, layer, expert, M, L, E, obs, off)
        blocks = opl.Blocks(bits, q, utype, layer, expert, M, off["s"])
        _, chosen, D = opl.plan_step(blocks, mass, phi, off, off["n_stages"], 16, F, B_KV)
        assert got["D"] == D
        if D > 0:
            stage, plan, total = chosen
            assert got["kind"] == 1 and got["stage"] == stage
            assert got["total"] == total
            assert [(i, a, b, d) for i, (a, b, d) in plan.items()] == got["entries"]
        else:
            plan, total = opl.reload_plan(blocks, q_init, mass, phi, off, 16, F, B_KV, 8)
            assert got["kind"] == (2 if total > 0 else 0)
            assert [(i, a, b, d) for i, (a, b, d) in plan.items()] == got["entries"]


def test_planner_hand_example():
    g = load_golden("greedy_hand.json")
    n = len(g["s"])
    off = dict(s=g["s"], head_w=np.zeros((2, 2, 3)), head_a=np.zeros((2, 2)), head_c=np.ones((2, 2)),
               alpha=1.0, rho_min=-2.0, rho_max=2.0, eps=1e-12, mu=[1.0], floors=[3], n_stages=g["n_stages"])
    for case in g["cases"]:
        obs = dict(T_blk=case["D"], F_blk=1, B_KV=1.0, R=1 << 30, mass=np.ones((1, 3)) / 3, phi=np.zeros((n, 3)))
        got = pw.pw_plan_host(g["bits"], [5] * n, [5] * n, [0] * n, [0] * n, list(range(n)), g["M"], 1, 3, obs, off)
        if case["chosen_stage"] is None:
            assert got["kind"] == 0 and got["entries"] == []
        else:
            assert got["stage"] == case["chosen_stage"]
            assert [list(e) for e in got["entries"]] == case["plan"]


def test_planner_rejects_small_capacity():
    rng = np.random.default_rng(1)
    bits, q, q_init, utype, layer, expert, M, L, E = _random_problem(rng)
    off = _offline(rng, len(q), len(bits))
    obs = dict(T_blk=16, F_blk=0, B_KV=1e9, R=8, mass=np.ones((L, E)) / E, phi=np.ones((len(q), 3)))
    with pytest.raises(pw.PwError):
        pw.pw_plan_host(bits, q, q_init, utype, layer, expert, M, L, E, obs, off, capacity=1)


@pytest.mark.parametrize("seed", range(6))
def test_batch_merge_and_residual_table_match_oracle(seed):
    """pw_merge_requests against the oracle's merge, and pw_plan_host planning from the merged
    table against the oracle planner on the same table (Sec. 3.2, batched serving)."""
    rng = np.random.default_rng(100 + seed)
    bits, q, q_init, utype, layer, expert, M, L, E = _random_problem(rng)
    n, nb = len(q), len(bits)
    off = _offline(rng, n, nb)
    reqs = []
    for _ in range(int(rng.integers(1, 5))):
        reqs.append(dict(mass=rng.dirichlet(np.ones(E), size=L), rho_hat=rng.normal(0, 1, (n, nb - 1)),
                         conf=rng.uniform(0.5, 1.0, (2, nb - 1)), rho_min=float(rng.uniform(-3, -1)),
                         rho_max=float(rng.uniform(1, 3))))
    kv = rng.integers(1, 40, size=len(reqs)).astype(float)
    got = pw.pw_merge_requests(reqs, kv, L, E, n, nb)
    want = opl.merge_request_signals(reqs, kv)
    for key in ("mass", "rho_hat", "conf", "rho_min", "rho_max"):
        assert np.array_equal(np.asarray(got[key]), np.asarray(want[key])), key
    off_m = dict(off, head_c=want["conf"], rho_min=want["rho_min"], rho_max=want["rho_max"])
    B_KV = float(M[0, 1] - M[0, 0]) * 0.7
    for F in (0, 5, 40):
        obs = dict(T_blk=16, F_blk=F, B_KV=B_KV, R=8, mass=want["mass"], phi=None, rho_hat=want["rho_hat"])
        plan = pw.pw_plan_host(bits, q, q_init, utype, layer, expert, M, L, E, obs, off_m)
        blocks = opl.Blocks(bits, q, utype, layer, expert, M, off["s"])
        off_t = dict(off_m, rho_hat=want["rho_hat"])
        _, chosen, D = opl.plan_step(blocks, want["mass"], None, off_t, off["n_stages"], 16, F, B_KV)
        assert plan["D"] == D
        if D > 0:
            stage, pl_, total = chosen
            assert plan["kind"] == 1 and plan["stage"] == stage and plan["total"] == total
            assert [(i, a, b, d) for i, (a, b, d) in pl_.items()] == plan["entries"]
        else:
            pl_, total = opl.reload_plan(blocks, q_init, want["mass"], None, off_t, 16, F, B_KV, 8)
            assert [(i, a, b, d) for i, (a, b, d) in pl_.items()] == plan["entries"]


def test_batch_merge_rejects_bad_weights():
    req = dict(mass=np.ones((1, 2)) / 2, rho_hat=np.zeros((2, 1)), conf=np.ones((2, 1)), rho_min=-1.0, rho_max=1.0)
    with pytest.raises(pw.PwError):
        pw.pw_merge_requests([req], [0.0], 1, 2, 2, 2)
    with pytest.raises(pw.PwError):
        pw.pw_merge_requests([req, req], [1.0, -1.0], 1, 2, 2, 2)
