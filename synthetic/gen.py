"""Seeded synthetic workloads shaped like the MoE layers the PagedWeight pages evaluate.

Every array here is drawn from numpy's PCG64, keyed by a ``SeedSequence`` built from
(seed, layer, expert, block type, tag), so any single block can be regenerated on its
own.  Nothing in this module performs routing, dequantisation, projection, packing or
planning; it only draws numbers and converts float formats.

Shapes follow the pages' model table (PagedWeight, Table 1) and the synthetic recipe:
bf16 N(0,1) activations, fp32 N(0,1/H) router with a Zipf log-prior bias, uniform
b_max-bit codes, sorted fp16 N(0, sigma) centroid tables per row and per bitwidth, and
bf16 N(0, 0.02) shared-expert weights.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import numpy as np

GATE_UP = 0
DOWN = 1


@dataclass(frozen=True)
class LayerShape:
    name: str
    H: int            # hidden size
    E: int            # routed experts
    I: int            # expert intermediate size
    K: int            # top-K
    Is: int           # shared-expert intermediate (0 = no shared expert)
    L: int            # layers in the stack
    bmax: int         # bit-planes stored per block
    bits: Tuple[int, ...]  # supported bitwidths B_i (ascending)
    sigma_lut: float  # std-dev of the centroid draws
    zipf_a: Optional[float]  # Zipf exponent of the router prior (None = no bias)
    q_rule: str       # "uniform" or "hot_cold"
    decode_T: Tuple[int, ...] = field(default=())
    prefill_T: Optional[int] = None

    def bits_mask(self) -> int:
        m = 0
        for b in self.bits:
            m |= 1 << b
        return m


SHAPES: Dict[str, LayerShape] = {
    # single tiny layer: hidden 128, 8 experts, intermediate 256, top-2, 8 tokens
    "tiny": LayerShape("tiny", H=128, E=8, I=256, K=2, Is=0, L=1, bmax=6,
                       bits=(3, 4, 5, 6), sigma_lut=0.02, zipf_a=None,
                       q_rule="uniform", decode_T=(8,)),
    # Qwen1.5-MoE-A2.7B-shaped stack (60 routed experts + dense shared FFN 5632)
    "qwen": LayerShape("qwen", H=2048, E=60, I=1408, K=4, Is=5632, L=24, bmax=8,
                       bits=(3, 4, 5, 6, 7, 8), sigma_lut=0.02, zipf_a=1.1,
                       q_rule="hot_cold", decode_T=(1, 16, 64, 256)),
    # Mixtral-8x7B-shaped layer
    "mixtral": LayerShape("mixtral", H=4096, E=8, I=14336, K=2, Is=0, L=32, bmax=8,
                          bits=(3, 4, 5, 6, 7, 8), sigma_lut=0.015, zipf_a=None,
                          q_rule="uniform", decode_T=(1, 8, 64, 256), prefill_T=4096),
    # 128-expert top-8 layer with one shared expert (Gemma-4-26B-A4B-like routing width)
    "g128": LayerShape("g128", H=2816, E=128, I=704, K=8, Is=2816, L=30, bmax=8,
                       bits=(3, 4, 5, 6, 7, 8), sigma_lut=0.02, zipf_a=1.0,
                       q_rule="uniform", decode_T=(1, 32, 256), prefill_T=2048),
}


def block_id(layer: int, expert: int, u: int, E: int) -> int:
    """Row of linear block i = (layer, expert, u) in the weight page table."""
    return (layer * E + expert) * 2 + u


def block_shape(shape: LayerShape, u: int) -> Tuple[int, int]:
    """(output rows N, input columns K) of a block; gate_up stacks gate rows over up rows."""
    if u == GATE_UP:
        return 2 * shape.I, shape.H
    return shape.H, shape.I


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in key])))


# ---------------------------------------------------------------- float formats
def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); return the raw uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen raw bfloat16 bits to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- blocks
TAG_IDX, TAG_LUT, TAG_ROUTER, TAG_TOK, TAG_SHARED, TAG_Q, TAG_PLAN, TAG_KV = 1, 2, 3, 4, 5, 6, 7, 8


def gen_block_np(shape: LayerShape, seed: int, layer: int, expert: int, u: int):
    """Codes and centroid tables of one linear block.

    Returns ``idx`` (uint8 [N][K], uniform in [0, 2^bmax)) and ``luts`` (dict b -> uint16
    fp16 bits [N][2^b], each row sorted ascending by value, drawn N(0, sigma_lut)).
    """
    N, Kin = block_shape(shape, u)
    r = _rng(seed, TAG_IDX, layer, expert, u)
    idx = r.integers(0, 1 << shape.bmax, size=(N, Kin), dtype=np.uint8)
    luts = {}
    for b in shape.bits:
        rl = _rng(seed, TAG_LUT, layer, expert, u, b)
        v = (rl.standard_normal(size=(N, 1 << b)) * shape.sigma_lut).astype(np.float16)
        v.sort(axis=1)
        luts[b] = v.view(np.uint16)
    return idx, luts


def zipf_log_prior(E: int, a: float, r: np.random.Generator):
    """Zipf(a) prior over experts with a random rank permutation: returns (log p_e, rank_e)."""
    ranks = r.permutation(E) + 1  # rank 1 = most popular
    p = ranks.astype(np.float64) ** (-a)
    p /= p.sum()
    return np.log(p).astype(np.float32), ranks


def gen_router_np(shape: LayerShape, seed: int, layer: int, attempt: int = 0):
    """Router weights W_r (fp32 [E][H], N(0, 1/H)), bias (fp32 [E] or None) and ranks."""
    r = _rng(seed, TAG_ROUTER, layer, attempt)
    Wr = (r.standard_normal(size=(shape.E, shape.H)) / math.sqrt(shape.H)).astype(np.float32)
    if shape.zipf_a is None:
        return Wr, None, np.arange(1, shape.E + 1)
    rb = _rng(seed, TAG_ROUTER, layer, 1 << 20)
    bias, ranks = zipf_log_prior(shape.E, shape.zipf_a, rb)
    return Wr, bias, ranks


def gen_token_np(shape: LayerShape, seed: int, layer: int, t: int, attempt: int = 0) -> np.ndarray:
    """One bf16 N(0,1) activation row (uint16 bits [H]); ``attempt`` selects a fresh draw."""
    r = _rng(seed, TAG_TOK, layer, t, attempt)
    return bf16_bits_from_f32(r.standard_normal(size=shape.H).astype(np.float32))


def gen_tokens_np(shape: LayerShape, seed: int, layer: int, T: int, attempts=None) -> np.ndarray:
    """Activations x (uint16 bf16 bits [T][H]); attempts[t] picks token t's draw."""
    out = np.empty((T, shape.H), dtype=np.uint16)
    for t in range(T):
        out[t] = gen_token_np(shape, seed, layer, t, 0 if attempts is None else int(attempts[t]))
    return out


def gen_shared_np(shape: LayerShape, seed: int, layer: int):
    """Shared-expert weights, bf16 N(0, 0.02): wgu [2Is][H] (gate rows then up rows), wd [H][Is]."""
    if shape.Is == 0:
        return None, None
    r = _rng(seed, TAG_SHARED, layer)
    wgu = bf16_bits_from_f32((r.standard_normal(size=(2 * shape.Is, shape.H)) * 0.02).astype(np.float32))
    wd = bf16_bits_from_f32((r.standard_normal(size=(shape.H, shape.Is)) * 0.02).astype(np.float32))
    return wgu, wd


def gen_q_assignment(shape: LayerShape, seed: int, layer: int, ranks=None) -> np.ndarray:
    """Initial committed bitwidth per block, int32 [E][2].

    ``uniform``: each block uniform over the supported bits.  ``hot_cold``: experts whose
    Zipf prior rank lies in the top quarter get bits uniform in {5..bmax}; the rest get
    bits uniform in {3, 4}.
    """
    r = _rng(seed, TAG_Q, layer)
    bits = np.array(shape.bits)
    if shape.q_rule == "uniform":
        return r.choice(bits, size=(shape.E, 2)).astype(np.int32)
    if ranks is None:
        raise ValueError("hot_cold assignment needs the router ranks")
    q = np.empty((shape.E, 2), dtype=np.int32)
    hot_cut = max(1, shape.E // 4)
    hot_bits = bits[bits >= 5]
    cold_bits = bits[bits <= 4]
    for e in range(shape.E):
        pool = hot_bits if ranks[e] <= hot_cut else cold_bits
        q[e] = r.choice(pool, size=2)
    return q


# ---------------------------------------------------------------- planner inputs
def gen_planner_offline_np(n_blocks: int, bits, n_buckets: int, seed: int):
    """Synthetic offline calibration: sensitivities decreasing in b with lognormal noise,
    random residual heads, confidences and per-bucket multipliers/floors."""
    r = _rng(seed, TAG_PLAN, 0)
    nb = len(bits)
    base = np.exp(r.normal(0.0, 1.0, size=(n_blocks, 1)))
    lvl = np.arange(nb)[None, :]
    s = base * (4.0 ** (-lvl)) * np.exp(r.normal(0.0, 0.3, size=(n_blocks, nb)))
    s = -np.sort(-s, axis=1)  # decreasing in b
    n_tr = nb - 1
    head_w = r.normal(0.0, 0.5, size=(2, n_tr, 3))
    head_a = r.normal(0.0, 0.5, size=(2, n_tr))
    head_c = r.uniform(0.5, 1.0, size=(2, n_tr))
    mu = np.array([4.0, 2.0, 1.0, 0.5][:n_buckets])
    floors = np.array([5, 4, 3, 3][:n_buckets], dtype=np.int32)
    return dict(s=s, head_w=head_w, head_a=head_a, head_c=head_c, alpha=1.0,
                rho_min=-2.0, rho_max=2.0, mu=mu, floors=floors, eps=1e-12)


def gen_phi_np(n_blocks: int, seed: int, step: int) -> np.ndarray:
    """Random three-dimensional routed-input features phi_i, one row per block."""
    r = _rng(seed, TAG_PLAN, 1, step)
    return np.abs(r.normal(1.0, 0.5, size=(n_blocks, 3)))


def gen_kv_requests(steps: int, seed: int, scale: int = 1, arrive_until: float = 0.7):
    """A decode-serving request schedule, per step a list of events in the order they are
    applied: ("finish", r), ("arrive", r, n) with n blocks of prompt KV, ("grow", r, n) and
    ("announce", r, n) -- n blocks the request expects to need at its next growth.

    Arrivals: one request with probability 0.9 sin^2(pi t / (arrive_until * steps)) at step
    t < arrive_until * steps, none later, so that the live KV demand rises, peaks and drains.
    A request (id = its arrival step) lives 20..50 steps, brings 2..6 prompt blocks and
    grows by one block every 2..4 steps, announcing each growth one step ahead; block
    counts are multiplied by `scale`.  The schedule does not depend on whether an event
    succeeds: a serving loop that cannot grant a request drops that request's later events."""
    r = _rng(seed, TAG_KV, 0)
    events = [[] for _ in range(steps)]
    last = int(arrive_until * steps)
    for t in range(last):
        u, life, prompt, every = r.random(), int(r.integers(20, 51)), int(r.integers(2, 7)), int(r.integers(2, 5))
        if u >= 0.9 * math.sin(math.pi * t / last) ** 2:
            continue
        prompt *= scale
        events[t].append(("arrive", t, prompt))
        end = min(steps - 1, t + life)
        for s in range(t + 1, end):
            if (s - t) % every == 0:
                events[s].append(("grow", t, scale))
            if (s + 1 - t) % every == 0 and s + 1 < end:
                events[s].append(("announce", t, scale))
        if t + life < steps:
            events[end].insert(0, ("finish", t))
    return events
