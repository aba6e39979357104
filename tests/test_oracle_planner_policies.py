"""Invariant pins of the planner oracle's stage/cap and reload policies (CPU only).

Algorithm 1 of PagedWeight Sec. 3.2 gives the stages of bitwidth floors, the greedy
selection and the choice of the best plan but prints no numbers for them, and the pages give
no reload policy at all.  These tests pin the oracle's readings with properties that hold on
any input.  Each would catch a plausible slip: a level cap off by one, a floor compared the
wrong way, a step delta taken with the wrong sign, a stage chosen out of order, or a reload
budget misread.
"""
import numpy as np
import pytest

from oracle import ap
from oracle import planner as opl


def problem(seed, n_layers=2, E=6, bits=(3, 4, 5, 6, 7, 8)):
    rng = np.random.default_rng(seed)
    n = n_layers * E * 2
    q = rng.choice(bits, size=n)
    q_init = np.maximum(q, rng.choice(bits, size=n))
    utype = np.arange(n) % 2
    expert = (np.arange(n) // 2) % E
    layer = np.arange(n) // 2 // E
    N = np.where(utype == 0, 64, 32)
    M = np.array([[ap.block_bytes(int(N[i]), 256, bits, b) for b in bits] for i in range(n)], dtype=np.float64)
    from synthetic import gen_planner_offline_np
    off = gen_planner_offline_np(n, list(range(len(bits))), 4, seed)
    off["n_stages"] = 3
    mass = rng.dirichlet(np.ones(E), size=n_layers)
    phi = np.abs(rng.normal(1.0, 0.5, size=(n, 3)))
    blocks = opl.Blocks(list(bits), q, utype, layer, expert, M, off["s"])
    return rng, list(bits), q, q_init, M, off, mass, phi, blocks


def bucket_of(blocks, mass, off):
    beta = opl.buckets_from_mass(mass, len(off["mu"]))
    return [int(beta[blocks.layer[i], blocks.expert[i]]) for i in range(len(blocks))]


@pytest.mark.parametrize("seed", range(10))
def test_stage_plans_respect_caps_floors_and_eq3(seed):
    rng, bits, q, q_init, M, off, mass, phi, blocks = problem(seed)
    beta = bucket_of(blocks, mass, off)
    B_KV = float(M[0, 1] - M[0, 0])
    for F in (-20, -5, 0, 3, 16):
        queue, chosen, D = opl.plan_step(blocks, mass, phi, off, off["n_stages"], 16, F, B_KV)
        assert D == max(0, 16 + 1 - F) * B_KV  # Eq. 7
        assert sorted(e[0] for e in queue) == list(range(off["n_stages"]))
        meets = []
        for s, plan, total in queue:
            for i, (a, b, d) in plan.items():
                la, lb = bits.index(a), bits.index(b)
                assert a == q[i] and lb < la  # a plan only lowers, from the committed bitwidth
                assert la - lb <= s + 1  # stage s: at most s + 1 levels below q_i
                assert b >= off["floors"][beta[i]]  # never below the bucket's floor
                assert d == M[i, la] - M[i, lb]  # Eq. 3 bytes of the whole reduction
            assert total == sum(d for _, _, d in plan.values())
            if D > 0 and total < D:  # short of D only when no legal step is left
                for i in range(len(blocks)):
                    lv = bits.index(plan[i][1]) if i in plan else bits.index(int(q[i]))
                    lq = bits.index(int(q[i]))
                    if lv > 0:
                        assert bits[lv - 1] < off["floors"][beta[i]] or lq - (lv - 1) > s + 1
            if D == 0:
                assert plan == {} and total == 0
            meets.append(D > 0 and total >= D)
        # more levels allowed never loses the ability to meet D
        for s in range(len(meets) - 1):
            assert not meets[s] or meets[s + 1]
        if D > 0:  # SelectBestPlan: lowest stage meeting D, else the largest release
            s, plan, total = chosen
            if any(meets):
                assert s == meets.index(True)
            else:
                best = max(e[2] for e in queue)
                assert total == best and s == min(e[0] for e in queue if e[2] == best)
        else:
            assert chosen is None


@pytest.mark.parametrize("seed", range(10))
def test_reload_plans_fit_the_budget_and_stop_at_the_first_misfit(seed):
    rng, bits, q, q_init, M, off, mass, phi, blocks = problem(seed)
    B_KV = float(M[0, 1] - M[0, 0])
    T_blk, R = 16, 8
    for F in (0, 16, 23, 24, 25, 30, 60, 500):
        plan, total = opl.reload_plan(blocks, q_init, mass, phi, off, T_blk, F, B_KV, R)
        if opl.target_bytes(T_blk, F, B_KV) > 0 or F < T_blk + R:
            assert plan == {} and total == 0  # reloads only with the reserve and R to spare
            continue
        budget = (F - T_blk - R) * B_KV
        assert total <= budget
        assert total == sum(d for _, _, d in plan.values())
        cur = {i: bits.index(int(q[i])) for i in range(len(blocks))}
        for i, (a, b, d) in plan.items():
            la, lb = bits.index(a), bits.index(b)
            assert a == q[i] and la < lb <= bits.index(int(q_init[i]))  # up to q_init, never past
            assert d == M[i, lb] - M[i, la]
            cur[i] = lb
        # the policy stops at the first step, in its order, that does not fit: the highest
        # priority raise left (largest d_hat / Delta, then larger Delta, then lower block)
        # would overflow the budget
        beta = bucket_of(blocks, mass, off)
        left = []
        for i, j in cur.items():
            if j < bits.index(int(q_init[i])):
                d_hat, delta = opl.score_step(blocks, i, j + 1, beta[i], phi[i], off)
                left.append((-(d_hat / delta), -delta, i, delta))
        if left:
            assert total + min(left)[3] > budget
        if F == 500:  # a budget this large restores every block to its initial bitwidth
            assert all(cur[i] == bits.index(int(q_init[i])) for i in cur)
