"""pw_route_noalloc: routing for callers that cannot allocate device memory where they route
(its scratch is a static array inside the library).  Collected last on purpose.

Checks, through the C ABI, that two calls in a row give the same expert ids and routing
weights as pw_moe_forward's router (the entry point that uses the context's allocated
scratch) and as the float64 oracle, within the tolerance the other GPU tests use for
routing weights, on the second layer of a two-layer context whose layers have different
routers."""
import numpy as np
import pytest

import synthetic as syn
from oracle import moe as omoe

from gpu_helpers import LayerData, make_ctx

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pw = pytest.importorskip("any_precision_bit_gb300")


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from any_precision_bit_gb300 import _build
    _build.build()


@pytest.mark.parametrize("name,T,flags", [("tiny", 8, 0), ("qwen", 16, 0), ("qwen", 64, 2)])
def test_route_noalloc_matches_forward_router_and_oracle(name, T, flags):
    shape = syn.SHAPES[name]
    tiny, prenorm = name == "tiny", bool(flags & 2)
    other = LayerData(shape, 3, 0, T, tiny=tiny, prenorm=prenorm)  # layer 0: another router
    data = LayerData(shape, 7, 1, T, tiny=tiny, prenorm=prenorm)   # layer 1: the one routed
    ctx = make_ctx(pw, shape, L=2, max_tokens=T)
    try:
        other.load(pw, ctx, layer_slot=0)
        data.load(pw, ctx, layer_slot=1)
        ids_o, w_o, _ = omoe.route(data.x, data.Wr, data.bias, shape.K, prenorm=prenorm)
        ids_l0, _, _ = omoe.route(data.x, other.Wr, other.bias, shape.K, prenorm=prenorm)
        assert not np.array_equal(ids_o, ids_l0)  # the layers route these tokens differently
        stream = pw.pw_get_stream(ctx)
        x = torch.from_numpy(data.x.view(np.int16)).cuda()
        y = torch.zeros_like(x)
        ids_ref = torch.zeros((T, shape.K), dtype=torch.int32, device="cuda")
        w_ref = torch.zeros((T, shape.K), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        pw.pw_moe_forward(ctx, 1, x, T, y, ids_ref, w_ref, flags, stream)
        torch.cuda.synchronize()
        for _ in range(2):  # two calls in a row: the static scratch keeps the last call's contents
            ids = torch.full((T, shape.K), -1, dtype=torch.int32, device="cuda")
            w = torch.full((T, shape.K), -1.0, dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            pw.pw_route_noalloc(ctx, 1, x, T, ids, w, flags, stream)
            torch.cuda.synchronize()
            got_ids, got_w = ids.cpu().numpy(), w.cpu().numpy()
            assert np.array_equal(got_ids, ids_o)
            assert np.allclose(got_w, w_o, rtol=1e-5, atol=1e-7)
            assert np.array_equal(got_ids, ids_ref.cpu().numpy())
            assert np.allclose(got_w, w_ref.cpu().numpy(), rtol=1e-5, atol=1e-7)
        pw.pw_check(ctx)  # no bounded wait gave up
    finally:
        pw.pw_destroy(ctx)


def test_route_noalloc_rejects_oversized_batches():
    shape = syn.SHAPES["qwen"]
    ctx = make_ctx(pw, shape, L=1, max_tokens=65536)
    try:
        LayerData(shape, 7, 0, 1).load(pw, ctx)
        x = torch.zeros((1, shape.H), dtype=torch.int16, device="cuda")
        ids = torch.zeros((1, shape.K), dtype=torch.int32, device="cuda")
        w = torch.zeros((1, shape.K), dtype=torch.float32, device="cuda")
        with pytest.raises(pw.PwError) as ei:
            pw.pw_route_noalloc(ctx, 0, x, 65536, ids, w, 0, pw.pw_get_stream(ctx))
        assert ei.value.status == pw.PW_ERR_INVALID  # 65536 x 60 fp32 logits alone exceed 8 MiB
        assert "static array" in str(ei.value)
    finally:
        pw.pw_destroy(ctx)
