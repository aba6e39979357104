"""Shared set-up of the GPU parity tests: seeded inputs from ``synthetic``, expected values
from ``oracle``, the product through its C ABI binding."""
from __future__ import annotations

import numpy as np

import synthetic as syn
from oracle import moe as omoe

TOL_REL_FRO = 5e-3   # relative Frobenius error of layer outputs
TOL_ABS_RMS = 2e-2   # per-element |err| <= TOL_ABS_RMS * rms(y_ref)


def gapped_router_and_tokens(shape, seed, layer, T, gap=1e-3, resample_router=False, prenorm=False):
    """Router weights and tokens whose sorted logits differ by >= gap among ranks 1..K+1.

    The tiny layer resamples W_r; the others resample individual tokens.  The logits are
    the oracle's (float64)."""
    def ok(l):
        s = np.sort(l)[::-1][: shape.K + 1]
        return np.all(-np.diff(s) >= gap)

    if resample_router:
        for attempt in range(1000):
            Wr, bias, ranks = syn.gen_router_np(shape, seed, layer, attempt)
            x = syn.gen_tokens_np(shape, seed, layer, T)
            l = omoe.router_logits(x, Wr, bias, prenorm)
            if all(ok(l[t]) for t in range(T)):
                return Wr, bias, ranks, x
        raise RuntimeError("no router draw met the logit gap")
    Wr, bias, ranks = syn.gen_router_np(shape, seed, layer)
    x = syn.gen_tokens_np(shape, seed, layer, T)
    for t in range(T):
        attempt = 0
        while not ok(omoe.router_logits(x[t:t + 1], Wr, bias, prenorm)[0]):
            attempt += 1
            x[t] = syn.gen_token_np(shape, seed, layer, t, attempt)
    return Wr, bias, ranks, x


def lut_concat(luts, bits):
    return np.ascontiguousarray(np.concatenate([luts[b].ravel() for b in bits]))


def filler_block(shape, u):
    N, K = syn.block_shape(shape, u)
    idx = np.zeros((N, K), dtype=np.uint8)
    lut = np.zeros(sum(N * (1 << b) for b in shape.bits), dtype=np.uint16)
    return idx, lut


def make_ctx(pw, shape, L=1, max_tokens=64, flags=0, renorm=0):
    d = pw.pw_desc(L=L, E=shape.E, H=shape.H, I=shape.I, K=shape.K, Is=shape.Is, bmax=shape.bmax,
                   bits_mask=shape.bits_mask(), renorm=renorm, device=0, max_tokens=max_tokens, flags=flags)
    return pw.pw_create(d)


class LayerData:
    """One layer's inputs; experts listed in ``real`` get generated weights, the rest zeros."""

    def __init__(self, shape, seed, layer, T, real=None, q=None, gap=1e-3, tiny=False, prenorm=False):
        self.shape, self.seed, self.layer, self.T = shape, seed, layer, T
        self.prenorm = prenorm
        self.Wr, self.bias, self.ranks, self.x = gapped_router_and_tokens(shape, seed, layer, T, gap,
                                                                          resample_router=tiny, prenorm=prenorm)
        ids, _, _ = omoe.route(self.x, self.Wr, self.bias, shape.K, prenorm=prenorm)
        self.routed = sorted(set(int(e) for e in np.unique(ids)))
        self.real = self.routed if real is None else sorted(real)
        self.experts = {}
        for e in self.real:
            gi, gl = syn.gen_block_np(shape, seed, layer, e, 0)
            di, dl = syn.gen_block_np(shape, seed, layer, e, 1)
            self.experts[e] = (gi, gl, di, dl)
        self.q = syn.gen_q_assignment(shape, seed, layer, self.ranks) if q is None else np.array(q, dtype=np.int32)
        self.shared = syn.gen_shared_np(shape, seed, layer) if shape.Is else None

    def load(self, pw, ctx, layer_slot=0, q_init=None):
        sh = self.shape
        for e in range(sh.E):
            for u in (0, 1):
                qi = int(self.q[e, u]) if q_init is None else int(q_init)
                if e in self.experts:
                    idx = self.experts[e][2 * u]
                    lut = lut_concat(self.experts[e][2 * u + 1], sh.bits)
                else:
                    idx, lut = filler_block(sh, u)
                pw.pw_pack(ctx, layer_slot, e, u, idx, lut, qi)
        pw.pw_set_router(ctx, layer_slot, self.Wr, self.bias)
        if self.shared is not None:
            pw.pw_set_shared(ctx, layer_slot, self.shared[0], self.shared[1])

    def oracle(self, q=None, tokens=None, renorm=False, shared_gate=None):
        return omoe.moe_layer(self.x, self.Wr, self.bias, self.experts, self.q if q is None else q,
                              self.shape.K, self.shape.bmax, shared=self.shared, renorm=renorm, tokens=tokens,
                              prenorm=self.prenorm, shared_gate=shared_gate)


def bf16_to_f64(a):
    return omoe.bf16_to_f64(np.asarray(a))


def assert_close(y_gpu, y_ref, what=""):
    err = y_gpu - y_ref
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-30))
    mx = float(np.max(np.abs(err)))
    assert rel <= TOL_REL_FRO, f"{what} rel-Frobenius {rel:.3e} > {TOL_REL_FRO}"
    assert mx <= TOL_ABS_RMS * rms, f"{what} max|err| {mx:.3e} > {TOL_ABS_RMS} * rms {rms:.3e}"
    return rel, mx / rms
