"""Pins of the oracle planner: Eqs. 1, 2, 4, 6, 7, 8 and a hand-sorted greedy example."""
import math

import numpy as np
import pytest

from conftest import load_golden
from oracle import planner as pl


def test_eq1_hand_example():
    g = load_golden("eq1_mass.json")
    m = pl.routing_mass(np.array(g["ids"]), np.array(g["weights"]), g["E"])
    assert np.allclose(m, g["mass"], rtol=0, atol=1e-15)
    assert abs(m.sum() - 1.0) < 1e-15


def test_eq2_hand_example():
    g = load_golden("eq2_sensitivity.json")
    assert pl.sensitivity(g["h"], g["W"], g["Wb"]) == g["s"]
    # no quantisation error -> zero sensitivity; h scales linearly
    assert pl.sensitivity([3.0], [1.0], [1.0]) == 0.0
    assert pl.sensitivity([2.0, 4.0], g["W"], g["Wb"]) == 2 * g["s"]


def test_eq4_eq6_eq8_hand_cases():
    g = load_golden("eq6_eq8.json")
    for lo, hi, want in g["eq4_cases"]:
        assert pl.global_damage(lo, hi) == pytest.approx(want, abs=1e-15)
    for rho, want in g["eta_cases"]:
        got = pl.prompt_factor(g["alpha"], g["c"], rho, g["rho_min"], g["rho_max"])
        assert got == pytest.approx(want, rel=1e-15)
    for gd, eta, want in g["dhat_cases"]:
        assert pl.predicted_damage(g["eps"], g["mu"], gd, eta) == pytest.approx(want, rel=1e-15)
    # Eq. 5 is an affine head
    assert pl.residual_head([1.0, 2.0, 3.0], 0.5, [1.0, 1.0, 1.0]) == 6.5


def test_eq7_hand_cases():
    g = load_golden("eq7_target.json")
    for F, want in g["cases"]:
        assert pl.target_bytes(g["T_blk"], F, g["B_KV"]) == want


def _hand_blocks(g):
    n = len(g["s"])
    return pl.Blocks(g["bits"], [5] * n, [0] * n, [0] * n, list(range(n)), g["M"], g["s"])


def _zero_off():
    return dict(head_w=np.zeros((2, 2, 3)), head_a=np.zeros((2, 2)), head_c=np.ones((2, 2)),
                alpha=1.0, rho_min=-2.0, rho_max=2.0, mu=np.array([1.0]), floors=np.array([3]),
                eps=1e-12)


def test_greedy_hand_sorted():
    g = load_golden("greedy_hand.json")
    blocks = _hand_blocks(g)
    mass = np.ones((1, 3)) / 3
    phi = np.zeros((3, 3))
    for case in g["cases"]:
        D = case["D"]
        queue, chosen, Dgot = pl.plan_step(blocks, mass, phi, _zero_off(), g["n_stages"],
                                           T_blk=D, F_blk=1, B_KV=1.0)
        assert Dgot == D
        assert [e[2] for e in sorted(queue)] == case["stage_totals"]
        if case["chosen_stage"] is None:
            assert chosen is None
            continue
        stage, plan, total = chosen
        assert stage == case["chosen_stage"]
        assert [[i, a, b, d] for i, (a, b, d) in plan.items()] == case["plan"]


def test_buckets_and_floors():
    mass = np.array([[0.1, 0.4, 0.3, 0.2]])
    beta = pl.buckets_from_mass(mass, 2)
    assert beta.tolist() == [[1, 0, 0, 1]]
    beta4 = pl.buckets_from_mass(np.array([[0.25, 0.25, 0.25, 0.25]]), 4)
    assert beta4.tolist() == [[0, 1, 2, 3]]  # ties to the lower expert id
    # a hot expert with floor 5 cannot drop below 5
    blocks = pl.Blocks((3, 4, 5, 6), [6, 6], [0, 0], [0, 0], [0, 1],
                       [[10, 20, 30, 40], [10, 20, 30, 40]], [[4, 3, 2, 1], [4, 3, 2, 1]])
    off = dict(head_w=np.zeros((2, 3, 3)), head_a=np.zeros((2, 3)), head_c=np.ones((2, 3)),
               alpha=1.0, rho_min=-2.0, rho_max=2.0, mu=np.array([1.0, 1.0]),
               floors=np.array([5, 3]), eps=1e-12)
    _, chosen, _ = pl.plan_step(blocks, np.array([[0.9, 0.1]]), np.zeros((2, 3)), off, 3,
                                T_blk=1000, F_blk=0, B_KV=1.0)
    stage, plan, total = chosen
    assert plan[0][1] == 5  # hot expert stops at its floor
    assert plan[1][1] == 3


def test_multiplier_and_residual_reorder_steps():
    """A larger bucket multiplier or a positive residual pushes a step later."""
    bits = (3, 4)
    blocks = pl.Blocks(bits, [4, 4], [0, 1], [0, 0], [0, 1], [[10, 20], [10, 20]], [[2, 1], [2, 1]])
    off = dict(head_w=np.zeros((2, 1, 3)), head_a=np.array([[0.0], [1.0]]), head_c=np.ones((2, 1)),
               alpha=1.0, rho_min=-2.0, rho_max=2.0, mu=np.array([1.0]), floors=np.array([3]),
               eps=1e-12)
    _, chosen, _ = pl.plan_step(blocks, np.array([[0.5, 0.5]]), np.zeros((2, 3)), off, 1,
                                T_blk=10, F_blk=10, B_KV=1.0)  # D = 1 byte -> one step
    assert list(chosen[1].keys()) == [0]  # block 1 (down head a=1 -> eta=e) costs more


def test_reload_restores_most_damaging_first():
    bits = (3, 4, 5)
    blocks = pl.Blocks(bits, [3, 4], [0, 0], [0, 0], [0, 1],
                       [[10, 20, 30], [10, 20, 30]], [[9, 1, 0.5], [3, 2, 1]])
    off = _zero_off()
    off["head_w"] = np.zeros((2, 2, 3))
    plan, total = pl.reload_plan(blocks, [5, 5], np.array([[0.5, 0.5]]), np.zeros((2, 3)), off,
                                 T_blk=16, F_blk=16 + 8 + 20, B_KV=1.0, R=8)
    # keys: b0 3->4 g=8 per 10 B (0.8), b0 4->5 0.05; b1 4->5 0.1. Budget 20 B.
    assert plan == {0: (3, 4, 10.0), 1: (4, 5, 10.0)}
    assert total == 20.0
    none, _ = pl.reload_plan(blocks, [5, 5], np.array([[0.5, 0.5]]), np.zeros((2, 3)), off,
                             T_blk=16, F_blk=20, B_KV=1.0, R=8)
    assert none == {}


def test_eq5_features_hand_example():
    g = load_golden("eq5_features.json")
    phi = pl.routed_input_features(np.array(g["x"]), np.array(g["ids"]), np.array(g["weights"]), g["E"])
    assert np.allclose(phi, np.array(g["phi"]), rtol=1e-14, atol=0)


def test_batch_merge_hand_example():
    g = load_golden("batch_merge.json")
    m = pl.merge_request_signals(g["requests"], g["kv_blocks"])
    for key in ("mass", "rho_hat", "conf"):
        assert np.allclose(m[key], np.array(g["merged"][key]), rtol=1e-15, atol=1e-15), key
    assert m["rho_min"] == pytest.approx(g["merged"]["rho_min"], abs=1e-15)
    assert m["rho_max"] == pytest.approx(g["merged"]["rho_max"], abs=1e-15)


def test_single_request_merge_is_identity_and_residual_table_matches_heads():
    """Merging one request changes nothing, and a residual table equal to the Eq. 5 heads'
    predictions gives the same plan as the heads on phi."""
    rng = np.random.default_rng(4)
    n, bits = 12, [3, 4, 5, 6]
    nb = len(bits)
    q = rng.choice(bits, size=n)
    utype = np.arange(n) % 2
    layer = np.zeros(n, dtype=int)
    expert = np.arange(n) // 2
    M = np.array([[b * 1000.0 + 50.0 * (1 << b) for b in bits] for _ in range(n)])
    s = -np.sort(-rng.lognormal(0.0, 1.0, size=(n, nb)), axis=1)
    off = dict(s=s, head_w=rng.normal(0, 0.5, (2, nb - 1, 3)), head_a=rng.normal(0, 0.5, (2, nb - 1)),
               head_c=rng.uniform(0.5, 1.0, (2, nb - 1)), alpha=1.0, rho_min=-2.0, rho_max=2.0,
               mu=[4.0, 2.0, 1.0, 0.5], floors=[3, 3, 3, 3], eps=1e-12)
    phi = np.abs(rng.normal(1.0, 0.5, (n, 3)))
    mass = rng.dirichlet(np.ones(6))[None, :]
    rho = np.array([[pl.residual_head(off["head_w"][utype[i]][j], off["head_a"][utype[i]][j], phi[i])
                     for j in range(nb - 1)] for i in range(n)])
    req = dict(mass=mass, rho_hat=rho, conf=off["head_c"], rho_min=off["rho_min"], rho_max=off["rho_max"])
    m = pl.merge_request_signals([req], [5.0])
    assert np.array_equal(m["rho_hat"], rho) and np.array_equal(m["mass"], mass)
    blocks = pl.Blocks(bits, q, utype, layer, expert, M, s)
    _, chosen_heads, _ = pl.plan_step(blocks, mass, phi, off, 3, 16, 2, 3000.0)
    off_table = dict(off, rho_hat=m["rho_hat"], head_c=m["conf"], rho_min=m["rho_min"], rho_max=m["rho_max"])
    _, chosen_table, _ = pl.plan_step(blocks, m["mass"], phi, off_table, 3, 16, 2, 3000.0)
    assert chosen_heads == chosen_table
