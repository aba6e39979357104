"""fp16 activation range: the experts read x and write h in fp16 (PagedWeight Sec. 3.3, the
fused kernel's operands; the pages leave the activation type open), so a value past 65504
must not pass silently.  Activations near the limit keep parity and leave no flag; an h or
an x that rounds past it makes pw_check report PW_ERR_RANGE once, and the next launch on the
same context is clean and correct again.  The scales are chosen with the oracle's own
h = silu(W_g x) * (W_u x), so each case is known to sit on its side of the limit."""
import numpy as np
import pytest

import synthetic as syn
from oracle import moe as omoe

from gpu_helpers import LayerData, assert_close, bf16_to_f64, make_ctx

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pw = pytest.importorskip("any_precision_bit_gb300")

FP16_MAX = 65504.0


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from any_precision_bit_gb300 import _build
    _build.build()


def to_bf16_bits(v):
    """Round-to-nearest-even float64 -> bf16 bit patterns (through float32)."""
    f = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def h_max(data, xb):
    """Largest |h| the oracle computes for the routed (token, expert) pairs of bf16 rows xb."""
    sh = data.shape
    ids, _, _ = omoe.route(xb, data.Wr, data.bias, sh.K)
    x = bf16_to_f64(xb)
    cache = data.__dict__.setdefault("_wgu", {})
    m = 0.0
    for e in np.unique(ids):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        if int(e) not in cache:
            gi, gl, _, _ = data.experts[int(e)]
            cache[int(e)] = omoe.block_weight(gi, gl, sh.bmax, int(data.q[e, 0]))
        Wgu = cache[int(e)]
        gu = x[rows] @ Wgu.T
        I = Wgu.shape[0] // 2
        with np.errstate(over="ignore"):  # exp(-g) overflows to inf for large negative g: silu -> 0
            h = omoe.silu(gu[:, :I]) * gu[:, I:]
        m = max(m, float(np.max(np.abs(h))))
    return m


def scale_for(data, target):
    """A scale s (bisection on the oracle) with h_max(bf16(s x)) close to target."""
    x = bf16_to_f64(data.x)
    lo, hi = 1.0, 1.0
    while h_max(data, to_bf16_bits(x * hi)) < target:
        hi *= 2.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if h_max(data, to_bf16_bits(x * mid)) < target:
            lo = mid
        else:
            hi = mid
    return lo


def run(ctx, xb, T):
    x = torch.from_numpy(xb.view(np.int16)).cuda()
    y = torch.zeros_like(x)
    torch.cuda.synchronize()
    pw.pw_moe_forward(ctx, 0, x, T, y, None, None, 0, pw.pw_get_stream(ctx))
    torch.cuda.synchronize()
    return bf16_to_f64(y.cpu().numpy().view(np.uint16))


def oracle_y(data, xb):
    y, _, _ = omoe.moe_layer(xb, data.Wr, data.bias, data.experts, data.q, data.shape.K, data.shape.bmax)
    return y


def expect_range_error(ctx):
    with pytest.raises(pw.PwError) as ei:
        pw.pw_check(ctx)
    assert ei.value.status == pw.PW_ERR_RANGE
    pw.pw_check(ctx)  # reported once


@pytest.fixture(scope="module")
def layer():
    shape = syn.SHAPES["tiny"]
    T = 8
    data = LayerData(shape, 21, 0, T, real=range(shape.E), tiny=True)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    data.load(pw, ctx)
    yield data, ctx, T
    pw.pw_destroy(ctx)


def test_near_limit_activations_keep_parity_and_raise_no_flag(layer):
    data, ctx, T = layer
    s = scale_for(data, 0.6 * FP16_MAX)
    xb = to_bf16_bits(bf16_to_f64(data.x) * s)
    hm = h_max(data, xb)
    assert 0.3 * FP16_MAX < hm < 0.9 * FP16_MAX and np.max(np.abs(bf16_to_f64(xb))) < FP16_MAX
    pw.pw_check(ctx)
    assert_close(run(ctx, xb, T), oracle_y(data, xb), f"h up to {hm:.0f}")
    pw.pw_check(ctx)


def test_h_past_the_limit_is_reported_and_the_context_recovers(layer):
    data, ctx, T = layer
    s = scale_for(data, 3.0 * FP16_MAX)
    xb = to_bf16_bits(bf16_to_f64(data.x) * s)
    assert h_max(data, xb) > 1.5 * FP16_MAX and np.max(np.abs(bf16_to_f64(xb))) < FP16_MAX
    pw.pw_check(ctx)
    run(ctx, xb, T)
    expect_range_error(ctx)
    assert_close(run(ctx, data.x, T), oracle_y(data, data.x), "after")
    pw.pw_check(ctx)


def test_x_past_the_limit_is_reported(layer):
    data, ctx, T = layer
    xb = data.x.copy()
    xb[3, 5] = to_bf16_bits(np.array([7.0e4]))[0]   # above the largest fp16
    pw.pw_check(ctx)
    run(ctx, xb, T)
    expect_range_error(ctx)
    xb = data.x.copy()
    xb[0, 1] = np.uint16(0x7FC0)                     # a bf16 NaN
    run(ctx, xb, T)
    expect_range_error(ctx)
    assert_close(run(ctx, data.x, T), oracle_y(data, data.x), "after")
    pw.pw_check(ctx)
