"""MoE layer forward in float64 (oracle; test infrastructure).

PagedWeight, Sec. 2.1: the router gives routing weights to E experts and picks the top
K per token.  Sec. 3.3: the fused kernel does the routing, the expert activation, the
down projection and the routing-weighted output accumulation, each linear block read
at its own committed bitwidth.  Table 1 counts shared experts alongside routed ones.

Readings where the pages are silent:
* router logits l = x W_r^T + bias; routing weights are the softmax over all E experts
  (r = p, not renormalised over the chosen K unless ``renorm``);
* top-K keeps the K largest p, ties to the lower expert id, listed by descending p;
* expert activation is SiLU(gate) * up with gate rows [0, I) and up rows [I, 2I) of the
  gate_up block; silu(g) = g / (1 + exp(-g));
* the shared expert is a dense FFN of the same form added to every token, ungated by
  default; with ``shared_gate`` (a vector w_g of length H) its output is scaled per token by
  sigmoid(x . w_g), the gated shared expert of the Qwen1.5-MoE model in the pages' Table 1;
* with ``prenorm`` the layer reads RMSNorm(x) = x / sqrt(mean(x^2) + 1e-6) with unit
  gain, as the pre-norm transformers of the pages' model table (Table 1) feed their MoE
  blocks; the caller adds the output to the un-normalised x.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

from . import ap


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of raw bfloat16 bits."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Unit-gain RMSNorm over the hidden dimension."""
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)


def router_logits(x_bits: np.ndarray, Wr: np.ndarray, bias: Optional[np.ndarray], prenorm: bool = False) -> np.ndarray:
    x = bf16_to_f64(x_bits)
    if prenorm:
        x = rmsnorm(x)
    l = x @ np.asarray(Wr, dtype=np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    return l


def softmax(l: np.ndarray) -> np.ndarray:
    z = np.exp(l - l.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def topk(p: np.ndarray, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-K experts per token by probability; ties go to the lower expert id."""
    T, E = p.shape
    ids = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -p[t]))  # primary: -p, secondary: expert id
        ids[t] = order[:K]
    w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    return ids, w


def route(x_bits, Wr, bias, K: int, renorm: bool = False, prenorm: bool = False):
    p = softmax(router_logits(x_bits, Wr, bias, prenorm))
    ids, w = topk(p, K)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return ids, w, p


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def block_weight(idx: np.ndarray, luts: Dict[int, np.ndarray], bmax: int, q: int) -> np.ndarray:
    """Dense float64 weight of a block at bitwidth q: split the codes into planes, read the
    top q planes back into q-bit codes, and look them up in LUT_q."""
    N, K = idx.shape
    planes = ap.pack_planes(idx, bmax)
    idx_q = ap.unpack_indices(planes, q, K)
    return ap.dequant(idx_q, luts[q])


def expert_ffn(xe: np.ndarray, Wgu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """o = W_d (silu(W_g x) * (W_u x)) for every row of xe (float64 [n][H])."""
    I = Wgu.shape[0] // 2
    gu = xe @ Wgu.T
    h = silu(gu[:, :I]) * gu[:, I:]
    return h @ Wd.T


def sigmoid(g: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-g))


def moe_layer(x_bits: np.ndarray, Wr, bias, experts, q: np.ndarray, K: int, bmax: int,
              shared=None, renorm: bool = False, tokens=None, prenorm: bool = False, shared_gate=None):
    """Forward of one MoE layer in float64.

    experts: dict e -> (gu_idx, gu_luts, d_idx, d_luts); only routed experts are needed.
    q: int [E][2] committed bitwidths (gate_up, down).
    shared: None or (wgu_bits [2Is][H], wd_bits [H][Is]) bf16.
    shared_gate: None or float [H]: the shared output is scaled by sigmoid(x . shared_gate).
    tokens: optional subset of token rows to evaluate (rows are independent).
    Returns (y float64 [T'][H], ids [T'][K], weights [T'][K]).
    """
    xb = np.asarray(x_bits)
    if tokens is not None:
        xb = xb[np.asarray(tokens)]
    ids, w, _ = route(xb, Wr, bias, K, renorm, prenorm)
    x = bf16_to_f64(xb)
    if prenorm:
        x = rmsnorm(x)
    T, H = x.shape
    y = np.zeros((T, H), dtype=np.float64)
    o = np.zeros((T, K, H), dtype=np.float64)
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        gu_idx, gu_luts, d_idx, d_luts = experts[int(e)]
        Wgu = block_weight(gu_idx, gu_luts, bmax, int(q[e, 0]))
        Wd = block_weight(d_idx, d_luts, bmax, int(q[e, 1]))
        o[rows, slots] = expert_ffn(x[rows], Wgu, Wd)
    for k in range(K):  # routing-weighted accumulation in k order
        y += w[:, k:k + 1] * o[:, k, :]
    if shared is not None:
        ys = expert_ffn(x, bf16_to_f64(shared[0]), bf16_to_f64(shared[1]))
        if shared_gate is not None:
            ys = sigmoid(x @ np.asarray(shared_gate, dtype=np.float64))[:, None] * ys
        y += ys
    return y, ids, w
