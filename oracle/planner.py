"""Quality-aware planner of PagedWeight, Sec. 3.2 (oracle; test infrastructure).

Closed forms: routing mass (Eq. 1), Hessian-weighted sensitivity (Eq. 2), global damage
(Eq. 4), prompt residual head (Eq. 5), prompt factor (Eq. 6), KV-pressure byte target
(Eq. 7) and predicted damage (Eq. 8).  ``plan_step`` follows Algorithm 1 (PlanStep):
target bytes, then for every bitwidth-floor stage ScoreActions -> GreedySelect ->
RefreshPlanQueue, then SelectBestPlan when pressure is triggered.

Readings of what Algorithm 1 leaves open.  The pages print no numbers for them; they are
pinned by the hand-sorted greedy example and by invariants that hold on any input (level
caps, bucket floors, Eq. 3 deltas, stage monotonicity, the choice of SelectBestPlan, the
reload budget and where a reload stops):
* a step is a single-level reduction b -> b' (b' the next lower supported bitwidth);
  taking a block's step unlocks its next lower step;
* buckets: experts of a layer sorted by routing mass (descending, ties to the lower
  expert id), rank r goes to bucket floor(r * n_buckets / E); bucket 0 is the hottest;
* a step is legal at stage s when b' >= floor(bucket) and the block would end at most
  s+1 levels below its committed bitwidth;
* GreedySelect pops the smallest d_hat / Delta (ties: larger Delta, then lower block
  id) until the released bytes reach D;
* the queue keeps the newest plan of every stage; SelectBestPlan returns the lowest
  stage whose plan meets D, else the plan releasing the most bytes (ties: lower stage);
* pressure is triggered when D > 0;
* reload (no printed policy): when D == 0 and F_blk >= T_blk + R, raise blocks that
  sit below their initial bitwidth one level at a time, most damaging reduction first
  (largest d_hat / Delta), while the restored bytes fit in (F_blk - T_blk - R) * B_KV.
"""
from __future__ import annotations

import heapq
import math
from typing import Dict, List, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------- closed forms
def routing_mass(ids: np.ndarray, weights: np.ndarray, E: int) -> np.ndarray:
    """Eq. 1: m_e = sum_{t,k} r_{t,k} [z_{t,k} = e] / sum_{t,k} r_{t,k}."""
    num = np.zeros(E, dtype=np.float64)
    for t in range(ids.shape[0]):
        for k in range(ids.shape[1]):
            num[int(ids[t, k])] += float(weights[t, k])
    return num / float(np.sum(weights, dtype=np.float64))


def routed_input_features(x: np.ndarray, ids: np.ndarray, weights: np.ndarray, E: int) -> np.ndarray:
    """Eq. 5's phi for every expert e (shared by its two linear blocks): over the tokens t
    routed to e with weight r_t, with n_t = ||x_t||_2 the norm of the expert's input row,
    (sum r n / sum r, sqrt(sum r n^2 / sum r), max n); zeros for an expert no token reached.
    x: float [T][H] (the input as the experts read it)."""
    phi = np.zeros((E, 3), dtype=np.float64)
    s0 = np.zeros(E)
    s1 = np.zeros(E)
    s2 = np.zeros(E)
    mx = np.zeros(E)
    for t in range(ids.shape[0]):
        n = math.sqrt(sum(float(v) * float(v) for v in x[t]))
        for k in range(ids.shape[1]):
            e, r = int(ids[t, k]), float(weights[t, k])
            s0[e] += r
            s1[e] += r * n
            s2[e] += r * n * n
            mx[e] = max(mx[e], n)
    for e in range(E):
        if s0[e] > 0:
            phi[e] = (s1[e] / s0[e], math.sqrt(s2[e] / s0[e]), mx[e])
    return phi


def sensitivity(h: np.ndarray, W: np.ndarray, Wb: np.ndarray) -> float:
    """Eq. 2: s^b = sum_j h_j (W_j - W^b_j)^2."""
    h = np.asarray(h, dtype=np.float64)
    d = np.asarray(W, dtype=np.float64) - np.asarray(Wb, dtype=np.float64)
    return float(np.sum(h * d * d))


def global_damage(s_lower: float, s_higher: float) -> float:
    """Eq. 4: g^{b->b'} = max{s^{b'} - s^b, 0}."""
    return max(s_lower - s_higher, 0.0)


def residual_head(w: Sequence[float], a: float, phi: Sequence[float]) -> float:
    """Eq. 5: rho_hat = w^T phi + a."""
    return float(sum(float(wi) * float(pi) for wi, pi in zip(w, phi)) + a)


def prompt_factor(alpha: float, c: float, rho_hat: float, rho_min: float, rho_max: float) -> float:
    """Eq. 6: eta = exp(alpha * c * clip(rho_hat, rho_min, rho_max))."""
    return math.exp(alpha * c * min(max(rho_hat, rho_min), rho_max))


def target_bytes(T_blk: int, F_blk: int, B_KV: float) -> float:
    """Eq. 7: D = max{0, T_blk + 1 - F_blk} * B_KV."""
    return max(0, T_blk + 1 - F_blk) * B_KV


def predicted_damage(eps: float, mu: float, g: float, eta: float) -> float:
    """Eq. 8: d_hat = max{eps, mu * g * eta}."""
    return max(eps, mu * g * eta)


def buckets_from_mass(mass: np.ndarray, n_buckets: int) -> np.ndarray:
    """Bucket of every expert of every layer from its routing mass (0 = hottest)."""
    L, E = mass.shape
    beta = np.zeros((L, E), dtype=np.int32)
    for l in range(L):
        order = sorted(range(E), key=lambda e: (-float(mass[l, e]), e))
        for r, e in enumerate(order):
            beta[l, e] = (r * n_buckets) // E
    return beta


# ---------------------------------------------------------------- Algorithm 1
class Blocks:
    """Planner view of the page table: one entry per linear block."""

    def __init__(self, bits, q, utype, layer, expert, M, s):
        self.bits = list(bits)
        self.q = [int(v) for v in q]
        self.utype = [int(v) for v in utype]
        self.layer = [int(v) for v in layer]
        self.expert = [int(v) for v in expert]
        self.M = np.asarray(M, dtype=np.float64)      # [n][nbits]
        self.s = np.asarray(s, dtype=np.float64)      # [n][nbits]

    def __len__(self):
        return len(self.q)

    def level(self, b: int) -> int:
        return self.bits.index(b)


def merge_request_signals(requests, kv_blocks):
    """Batched serving (Sec. 3.2): the request-level routing masses, prompt residuals,
    confidence scores and clipping bounds merged into one batch-level table, each averaged
    with the requests' KV-block usage as weights (w_r = kv_r / sum kv, summed in request
    order).  requests: dicts with mass [L][E], rho_hat [n_blocks][n_bits-1], conf
    [2][n_bits-1], rho_min, rho_max."""
    tot = 0.0
    for kv in kv_blocks:
        tot += float(kv)
    w = [float(kv) / tot for kv in kv_blocks]
    out = {}
    for key in ("mass", "rho_hat", "conf"):
        acc = np.zeros_like(np.asarray(requests[0][key], dtype=np.float64))
        for wr, r in zip(w, requests):
            acc = acc + wr * np.asarray(r[key], dtype=np.float64)
        out[key] = acc
    for key in ("rho_min", "rho_max"):
        acc = 0.0
        for wr, r in zip(w, requests):
            acc = acc + wr * float(r[key])
        out[key] = acc
    return out


def score_step(blocks: Blocks, i: int, j: int, beta_i: int, phi_i, off) -> tuple:
    """d_hat and Delta of block i stepping from level j to level j-1.  With a batch-level
    table (off["rho_hat"], merged residuals), the residual is read from it instead of the
    Eq. 5 head on phi."""
    u = blocks.utype[i]
    g = global_damage(blocks.s[i, j - 1], blocks.s[i, j])
    if "rho_hat" in off:
        rho = float(off["rho_hat"][i][j - 1])
    else:
        rho = residual_head(off["head_w"][u][j - 1], off["head_a"][u][j - 1], phi_i)
    eta = prompt_factor(off["alpha"], off["head_c"][u][j - 1], rho, off["rho_min"], off["rho_max"])
    d_hat = predicted_damage(off["eps"], off["mu"][beta_i], g, eta)
    delta = blocks.M[i, j] - blocks.M[i, j - 1]
    return d_hat, delta


def greedy_select(blocks: Blocks, beta_blk, phi, off, cap: int, D: float):
    """One stage: take the cheapest legal single-level steps until D bytes are released."""
    if D <= 0:
        return {}, 0.0
    lvl = [blocks.level(b) for b in blocks.q]
    cur = list(lvl)
    heap = []

    def push(i):
        j = cur[i]
        if j == 0:
            return
        if blocks.bits[j - 1] < off["floors"][beta_blk[i]]:
            return
        if lvl[i] - (j - 1) > cap:
            return
        d_hat, delta = score_step(blocks, i, j, beta_blk[i], None if phi is None else phi[i], off)
        heapq.heappush(heap, (d_hat / delta, -delta, i, d_hat, delta))

    for i in range(len(blocks)):
        push(i)
    total = 0.0
    per_block: Dict[int, float] = {}
    while heap and total < D:
        _, _, i, _, delta = heapq.heappop(heap)
        cur[i] -= 1
        total += delta
        per_block[i] = per_block.get(i, 0.0) + delta
        push(i)
    plan = {i: (blocks.q[i], blocks.bits[cur[i]], per_block[i]) for i in sorted(per_block)}
    return plan, total


def plan_step(blocks: Blocks, mass: np.ndarray, phi: np.ndarray, off, n_stages: int,
              T_blk: int, F_blk: int, B_KV: float, queue: Optional[list] = None):
    """PlanStep: returns (queue, chosen plan or None, D).

    The queue holds one (stage, plan, total) entry per stage, refreshed every call.
    """
    D = target_bytes(T_blk, F_blk, B_KV)
    beta = buckets_from_mass(mass, len(off["mu"]))
    beta_blk = [int(beta[blocks.layer[i], blocks.expert[i]]) for i in range(len(blocks))]
    new_queue = list(queue) if queue else []
    for s in range(n_stages):
        plan, total = greedy_select(blocks, beta_blk, phi, off, s + 1, D)
        new_queue = [e for e in new_queue if e[0] != s] + [(s, plan, total)]
    chosen = None
    if D > 0:  # PressureTriggered
        meeting = sorted((e for e in new_queue if e[2] >= D), key=lambda e: e[0])
        if meeting:
            chosen = meeting[0]
        else:
            chosen = sorted(new_queue, key=lambda e: (-e[2], e[0]))[0]
    return new_queue, chosen, D


def reload_plan(blocks: Blocks, q_init, mass, phi, off, T_blk: int, F_blk: int,
                B_KV: float, R: int):
    """Reload policy reading: restore single levels, most damaging reduction first."""
    if target_bytes(T_blk, F_blk, B_KV) > 0 or F_blk < T_blk + R:
        return {}, 0.0
    budget = (F_blk - T_blk - R) * B_KV
    beta = buckets_from_mass(mass, len(off["mu"]))
    cur = [blocks.level(b) for b in blocks.q]
    top = [blocks.level(b) for b in q_init]
    heap = []

    def push(i):
        j = cur[i]
        if j >= top[i]:
            return
        d_hat, delta = score_step(blocks, i, j + 1, int(beta[blocks.layer[i], blocks.expert[i]]),
                                  None if phi is None else phi[i], off)
        heapq.heappush(heap, (-(d_hat / delta), -delta, i, delta))

    for i in range(len(blocks)):
        push(i)
    total = 0.0
    restored: Dict[int, float] = {}
    while heap:
        _, _, i, delta = heap[0]
        if total + delta > budget:
            break
        heapq.heappop(heap)
        cur[i] += 1
        total += delta
        restored[i] = restored.get(i, 0.0) + delta
        push(i)
    plan = {i: (blocks.q[i], blocks.bits[cur[i]], restored[i]) for i in sorted(restored)}
    return plan, total
