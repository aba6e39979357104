"""Device-side failure detection without a GPU fault: a bounded barrier wait inside the
gate_up expert kernel is made to expire by withholding one arrival (nothing asynchronous is
held back), with the wait limit cut short; the launch is reported through pw_check as
PW_ERR_TIMEOUT and the next launch on the same context is correct again."""
import numpy as np
import pytest

import synthetic as syn

from gpu_helpers import LayerData, assert_close, bf16_to_f64, make_ctx

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pw = pytest.importorskip("any_precision_bit_gb300")


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from any_precision_bit_gb300 import _build
    _build.build()


def forward(ctx, data, T):
    x = torch.from_numpy(data.x.view(np.int16)).cuda()
    y = torch.zeros_like(x)
    torch.cuda.synchronize()
    pw.pw_moe_forward(ctx, 0, x, T, y, None, None, 0, pw.pw_get_stream(ctx))
    torch.cuda.synchronize()
    return bf16_to_f64(y.cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("name,T", [("tiny", 8), ("qwen", 16)])
def test_expired_device_wait_is_reported_and_the_context_recovers(name, T):
    shape = syn.SHAPES[name]
    data = LayerData(shape, 11, 0, T, real=range(shape.E) if name == "tiny" else None, tiny=(name == "tiny"))
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        y_ref, _, _ = data.oracle()
        assert_close(forward(ctx, data, T), y_ref, "before")
        pw.pw_check(ctx)
        pw.pw_set_fault(ctx, 5, 500)  # waits give up after about 0.5 ms
        pw.pw_set_fault(ctx, 4, 1)    # the next gate_up launch withholds one arrival
        forward(ctx, data, T)         # its outputs are invalid
        with pytest.raises(pw.PwError) as ei:
            pw.pw_check(ctx)
        assert ei.value.status == pw.PW_ERR_TIMEOUT
        pw.pw_check(ctx)              # reported once
        assert_close(forward(ctx, data, T), y_ref, "with the short limit, nothing withheld")
        pw.pw_set_fault(ctx, 5, 0)
        again = forward(ctx, data, T)
        assert_close(again, y_ref, "after")
        assert np.array_equal(again, forward(ctx, data, T))
        pw.pw_check(ctx)
    finally:
        pw.pw_destroy(ctx)


def test_fault_kinds_are_checked():
    shape = syn.SHAPES["tiny"]
    ctx = make_ctx(pw, shape, L=1, max_tokens=8)
    try:
        for kind, n in ((5, -1), (9, 1)):
            with pytest.raises(pw.PwError) as ei:
                pw.pw_set_fault(ctx, kind, n)
            assert ei.value.status == pw.PW_ERR_INVALID
    finally:
        pw.pw_destroy(ctx)
