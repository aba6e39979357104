"""Pins of the oracle's router, top-K, expert FFN and combine (CPU only)."""
import math

import numpy as np
import pytest

import synthetic as syn
from oracle import moe


def test_bf16_exact():
    vals = np.array([1.0, -2.5, 3.140625, 1e-3, 65504.0, -0.0], dtype=np.float32)
    bits = syn.bf16_bits_from_f32(vals)
    back = moe.bf16_to_f64(bits)
    for v, b in zip(vals, back):
        # bf16 keeps 8 mantissa bits: relative rounding error below 2^-8
        assert abs(b - float(v)) <= abs(float(v)) * 2.0 ** -8
    assert moe.bf16_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0


def test_silu_closed_form():
    assert moe.silu(np.array([0.0]))[0] == 0.0
    assert abs(moe.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(moe.silu(np.array([30.0]))[0] - 30.0) < 1e-9
    assert abs(moe.silu(np.array([-30.0]))[0]) < 1e-9
    # silu(x) - silu(-x) = x
    x = np.linspace(-5, 5, 11)
    assert np.allclose(moe.silu(x) - moe.silu(-x), x, atol=1e-14)


def test_softmax_and_topk_against_full_sort():
    rng = np.random.default_rng(0)
    l = rng.normal(size=(50, 16))
    p = moe.softmax(l)
    assert np.allclose(p.sum(axis=1), 1.0)
    ref = np.exp(l) / np.exp(l).sum(axis=1, keepdims=True)
    assert np.allclose(p, ref, rtol=1e-13)
    ids, w = moe.topk(p, 4)
    full = np.argsort(-p, axis=1, kind="stable")
    assert np.array_equal(ids, full[:, :4])
    assert np.array_equal(w, np.take_along_axis(p, full[:, :4], axis=1))


def test_topk_ties_go_to_lower_expert():
    p = np.array([[0.1, 0.3, 0.3, 0.3]])
    ids, _ = moe.topk(p, 2)
    assert ids.tolist() == [[1, 2]]
    ids, _ = moe.topk(np.array([[0.25, 0.25, 0.25, 0.25]]), 3)
    assert ids.tolist() == [[0, 1, 2]]


def test_router_bias_and_renorm():
    x = syn.bf16_bits_from_f32(np.array([[1.0, 0.0], [0.0, 1.0]], dtype=np.float32))
    Wr = np.array([[1.0, 0.0], [0.0, 1.0], [0.5, 0.5]], dtype=np.float32)
    bias = np.array([0.0, 0.0, 10.0], dtype=np.float32)
    l = moe.router_logits(x, Wr, bias)
    assert l.tolist() == [[1.0, 0.0, 10.5], [0.0, 1.0, 10.5]]
    ids, w, p = moe.route(x, Wr, bias, 2, renorm=True)
    assert ids[:, 0].tolist() == [2, 2]
    assert np.allclose(w.sum(axis=1), 1.0)
    ids2, w2, _ = moe.route(x, Wr, bias, 2, renorm=False)
    assert np.array_equal(ids, ids2) and np.all(w2 < w + 1e-15)


def _brute_layer(x_bits, Wr, bias, experts, q, K, bmax, shared, gate=None):
    """Per-output-element loops in a different order from the oracle: each weight is read
    from its code with Python integer bit operations, each dot product summed by hand."""
    T, H = x_bits.shape
    x = moe.bf16_to_f64(x_bits)
    E = Wr.shape[0]
    out = np.zeros((T, H))
    for t in range(T):
        logits = []
        for e in range(E):
            acc = 0.0
            for h in range(H):
                acc += x[t, h] * float(Wr[e, h])
            logits.append(acc + (0.0 if bias is None else float(bias[e])))
        mx = max(logits)
        ex = [math.exp(v - mx) for v in logits]
        tot = sum(ex)
        prob = [v / tot for v in ex]
        chosen = sorted(range(E), key=lambda e: (-prob[e], e))[:K]
        for e in chosen:
            gu_idx, gu_luts, d_idx, d_luts = experts[e]
            qg, qd = int(q[e, 0]), int(q[e, 1])
            I = gu_idx.shape[0] // 2
            lg = gu_luts[qg].view(np.float16)
            ld = d_luts[qd].view(np.float16)
            hvec = []
            for n in range(I):
                g = 0.0
                u = 0.0
                for h in range(H):
                    g += float(lg[n, int(gu_idx[n, h]) >> (bmax - qg)]) * x[t, h]
                    u += float(lg[I + n, int(gu_idx[I + n, h]) >> (bmax - qg)]) * x[t, h]
                hvec.append(g / (1.0 + math.exp(-g)) * u)
            for m in range(H):
                acc = 0.0
                for n in range(I):
                    acc += float(ld[m, int(d_idx[m, n]) >> (bmax - qd)]) * hvec[n]
                out[t, m] += prob[e] * acc
        if shared is not None:
            wgu = moe.bf16_to_f64(shared[0])
            wd = moe.bf16_to_f64(shared[1])
            Is = wgu.shape[0] // 2
            hs = []
            for n in range(Is):
                g = sum(wgu[n, h] * x[t, h] for h in range(H))
                u = sum(wgu[Is + n, h] * x[t, h] for h in range(H))
                hs.append(g / (1.0 + math.exp(-g)) * u)
            scale = 1.0
            if gate is not None:
                z = sum(x[t, h] * float(gate[h]) for h in range(H))
                scale = 1.0 / (1.0 + math.exp(-z))
            for m in range(H):
                out[t, m] += scale * sum(wd[m, n] * hs[n] for n in range(Is))
    return out


@pytest.mark.parametrize("with_shared", [False, True])
def test_layer_matches_brute_force(with_shared):
    shape = syn.LayerShape("brute", H=16, E=4, I=8, K=2, Is=8 if with_shared else 0, L=1, bmax=6,
                           bits=(3, 4, 5, 6), sigma_lut=0.2, zipf_a=1.0, q_rule="uniform")
    seed = 11
    Wr, bias, _ = syn.gen_router_np(shape, seed, 0)
    x = syn.gen_tokens_np(shape, seed, 0, 3)
    experts = {}
    for e in range(shape.E):
        gi, gl = syn.gen_block_np(shape, seed, 0, e, 0)
        di, dl = syn.gen_block_np(shape, seed, 0, e, 1)
        experts[e] = (gi, gl, di, dl)
    q = syn.gen_q_assignment(shape, seed, 0)
    shared = syn.gen_shared_np(shape, seed, 0) if with_shared else None
    y, ids, w = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared)
    ref = _brute_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    # token subsets give the same rows
    y2, _, _ = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared, tokens=[2, 0])
    assert np.allclose(y2, y[[2, 0]], rtol=1e-13, atol=1e-15)


def test_layer_uses_committed_bits():
    """Changing one block's committed bitwidth changes only tokens routed to that expert."""
    shape = syn.SHAPES["tiny"]
    seed = 5
    Wr, bias, _ = syn.gen_router_np(shape, seed, 0)
    x = syn.gen_tokens_np(shape, seed, 0, shape.decode_T[0])
    experts = {e: syn.gen_block_np(shape, seed, 0, e, 0) + syn.gen_block_np(shape, seed, 0, e, 1)
               for e in range(shape.E)}
    q = syn.gen_q_assignment(shape, seed, 0)
    y, ids, _ = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax)
    e0 = int(ids[0, 0])
    q2 = q.copy()
    q2[e0, 1] = 3 if q[e0, 1] != 3 else 6
    y2, _, _ = moe.moe_layer(x, Wr, bias, experts, q2, shape.K, shape.bmax)
    for t in range(x.shape[0]):
        changed = not np.allclose(y[t], y2[t])
        assert changed == (e0 in ids[t])


def test_rmsnorm_and_prenorm_layer():
    x = np.array([[3.0, 4.0], [1.0, -1.0]])
    n = moe.rmsnorm(x, eps=0.0)
    assert np.allclose(n, [[3 / np.sqrt(12.5), 4 / np.sqrt(12.5)], [1.0, -1.0]])
    # a pre-normalised layer is invariant to scaling its input (up to eps)
    shape = syn.SHAPES["tiny"]
    Wr, bias, _ = syn.gen_router_np(shape, 3, 0)
    xb = syn.gen_tokens_np(shape, 3, 0, 4)
    experts = {e: syn.gen_block_np(shape, 3, 0, e, 0) + syn.gen_block_np(shape, 3, 0, e, 1) for e in range(shape.E)}
    q = syn.gen_q_assignment(shape, 3, 0)
    y1, ids1, _ = moe.moe_layer(xb, Wr, bias, experts, q, shape.K, shape.bmax, prenorm=True)
    x2 = syn.bf16_bits_from_f32((moe.bf16_to_f64(xb) * 4.0).astype(np.float32))  # exact power of two
    y2, ids2, _ = moe.moe_layer(x2, Wr, bias, experts, q, shape.K, shape.bmax, prenorm=True)
    assert np.array_equal(ids1, ids2)
    # eps = 1e-6 against mean(x^2) ~ 1 perturbs the scale by ~eps/2
    assert np.allclose(y1, y2, rtol=1e-5, atol=1e-9)


def test_gated_shared_expert():
    """Sigmoid-gated shared expert: brute force with a random gate, and the closed forms
    sigmoid(0) = 1/2 (the shared output exactly halved) and a saturated gate (ungated)."""
    shape = syn.LayerShape("gate", H=16, E=4, I=8, K=2, Is=8, L=1, bmax=6, bits=(3, 4, 5, 6), sigma_lut=0.2,
                           zipf_a=1.0, q_rule="uniform")
    seed = 12
    Wr, bias, _ = syn.gen_router_np(shape, seed, 0)
    x = syn.gen_tokens_np(shape, seed, 0, 3)
    experts = {}
    for e in range(shape.E):
        gi, gl = syn.gen_block_np(shape, seed, 0, e, 0)
        di, dl = syn.gen_block_np(shape, seed, 0, e, 1)
        experts[e] = (gi, gl, di, dl)
    q = syn.gen_q_assignment(shape, seed, 0)
    shared = syn.gen_shared_np(shape, seed, 0)
    gate = np.random.default_rng(3).normal(0.0, 0.5, size=shape.H)
    y, _, _ = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared, shared_gate=gate)
    ref = _brute_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared, gate)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    y_none, _, _ = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax)
    y_full, _, _ = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared)
    y_half, _, _ = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared,
                                 shared_gate=np.zeros(shape.H))
    assert np.allclose(y_half - y_none, 0.5 * (y_full - y_none), rtol=1e-12, atol=1e-15)
    xf = moe.bf16_to_f64(x)
    sat = 60.0 * np.linalg.lstsq(xf, np.ones(xf.shape[0]), rcond=None)[0]  # x . sat = 60 for every token
    assert np.allclose(xf @ sat, 60.0)
    y_sat, _, _ = moe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared, shared_gate=sat)
    assert np.allclose(y_sat, y_full, rtol=1e-12, atol=1e-14)
