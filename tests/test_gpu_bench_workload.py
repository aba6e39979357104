"""Teacher-forced parity of the benchmark's own workload: the Qwen-shaped 24-layer stack of
bench.py (seed 0, weights drawn on the device by the same generator keys), decoding its
64-token batch with pre-norm and the residual accumulate of pw_stack_forward.  The first and
the last layer are checked against the float64 oracle on the inputs the GPU stack gave them,
on every token whose router logits are separated by at least 1e-3 (ties may route
differently in fp32 and fp64)."""
import numpy as np
import pytest

import synthetic as syn
from oracle import moe as omoe

from gpu_helpers import assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pw = pytest.importorskip("any_precision_bit_gb300")


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from any_precision_bit_gb300 import _build
    _build.build()


def layer_reference(shape, seed, layer, x_bits, tokens):
    """The oracle's layer on the given input rows, with the weights bench.py draws."""
    from synthetic.gen_torch import gen_block_torch, gen_shared_torch, split_luts
    Wr, bias, ranks = syn.gen_router_np(shape, seed, layer)
    q = syn.gen_q_assignment(shape, seed, layer, ranks)
    xs = x_bits[tokens]
    ids, _, _ = omoe.route(xs, Wr, bias, shape.K, prenorm=True)
    experts = {}
    for e in np.unique(ids):
        blk = []
        for u in (0, 1):
            idx, lut = gen_block_torch(shape, seed, layer, int(e), u)
            N, _ = syn.block_shape(shape, u)
            blk += [idx.cpu().numpy(), split_luts(lut.cpu().numpy(), N, shape.bits)]
        experts[int(e)] = tuple(blk)
    wgu, wd = gen_shared_torch(shape, seed, layer)
    shared = (wgu.cpu().numpy().view(np.uint16), wd.cpu().numpy().view(np.uint16))
    y, ids, w = omoe.moe_layer(xs, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared, prenorm=True)
    return y, ids, w


def gapped(x_bits, shape, seed, layer, gap=1e-3):
    Wr, bias, _ = syn.gen_router_np(shape, seed, layer)
    l = omoe.router_logits(x_bits, Wr, bias, True)
    s = -np.sort(-l, axis=1)[:, : shape.K + 1]
    return np.nonzero(np.all(-np.diff(s, axis=1) >= gap, axis=1))[0]


def test_bench_workload_first_and_last_layer_teacher_forced():
    import bench
    shape = syn.SHAPES["qwen"]
    L, T, seed = shape.L, 64, 0
    ctx, _ = bench.load_stack(pw, torch, shape, L, T, seed, 0)
    try:
        stream = torch.cuda.Stream()
        pw.pw_set_stream(ctx, stream)
        x = torch.from_numpy(syn.gen_tokens_np(shape, seed, 0, T).view(np.int16)).cuda()
        ids = torch.zeros((T, shape.K), dtype=torch.int32, device="cuda")
        seen = {}
        torch.cuda.synchronize()
        for l in range(L):
            if l in (0, L - 1):
                x_in = x.cpu().numpy().view(np.uint16).copy()
            pw.pw_moe_forward(ctx, l, x, T, x, ids, None, pw.PW_ACCUMULATE | pw.PW_PRENORM, stream)
            stream.synchronize()
            if l in (0, L - 1):
                seen[l] = (x_in, x.cpu().numpy().view(np.uint16).copy(), ids.cpu().numpy().copy())
        pw.pw_check(ctx)
        for l, (x_in, x_out, ids_gpu) in seen.items():
            tok = gapped(x_in, shape, seed, l)
            assert len(tok) >= T // 2
            y_ref, ids_ref, _ = layer_reference(shape, seed, l, x_in, tok)
            assert np.array_equal(ids_gpu[tok], ids_ref), f"layer {l}"
            assert_close(bf16_to_f64(x_out[tok]), bf16_to_f64(x_in[tok]) + y_ref, f"layer {l}")
    finally:
        pw.pw_destroy(ctx)
