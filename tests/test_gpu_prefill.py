"""GPU parity of the prefill tiling (batches of >= 512 tokens: 128-token work items, two
accumulators of 128 tensor-memory columns, activation stages split along K) against the
float64 oracle.

Small layers are checked on every token; the model-shaped prefill batches (a 4096-token
Mixtral-shaped layer, a 2048-token 128-expert layer with a shared expert) on a sample of
tokens, since every output row depends only on its own token."""
import numpy as np
import pytest

import synthetic as syn
from oracle import moe as omoe

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
    ids = torch.zeros((T, data.shape.K), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, data.shape.K), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    pw.pw_moe_forward(ctx, 0, x, T, y, ids, w, 0, pw.pw_get_stream(ctx))
    torch.cuda.synchronize()
    return bf16_to_f64(y.cpu().numpy().view(np.uint16)), ids.cpu().numpy(), w.cpu().numpy()


# ragged everywhere: K of both blocks not a multiple of 128, N not a multiple of 128, a
# shared expert whose down projection is split along K, token chunks with short tails
RAGGED = syn.LayerShape("ragged_prefill", H=400, E=6, I=176, K=2, Is=240, L=1, bmax=8,
                        bits=(3, 4, 5, 6, 7, 8), sigma_lut=0.02, zipf_a=1.0, q_rule="uniform")


@pytest.mark.parametrize("name,T", [("tiny", 512), ("tiny", 1000), ("ragged", 700)])
def test_small_prefill_layer_every_token(name, T):
    shape = RAGGED if name == "ragged" else syn.SHAPES[name]
    data = LayerData(shape, 3, 0, T, real=range(shape.E))
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        y, ids, w = forward(ctx, data, T)
        y_ref, ids_ref, w_ref = data.oracle()
        assert np.array_equal(ids, ids_ref)
        assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)
        assert_close(y, y_ref, f"{name} T={T}")
        # the per-expert token counts include 128-token chunks and ragged tails
        counts = np.bincount(ids_ref.ravel(), minlength=shape.E)
        assert counts.max() > 128
    finally:
        pw.pw_destroy(ctx)


def test_prefill_output_is_bitwise_repeatable():
    shape = RAGGED
    T = 900
    q = np.where(np.arange(shape.E)[:, None] % 2 == 0, 3, 8) * np.ones((1, 2), dtype=np.int32)
    data = LayerData(shape, 5, 0, T, real=range(shape.E), q=q)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        first, _, _ = forward(ctx, data, T)
        for _ in range(4):
            again, _, _ = forward(ctx, data, T)
            assert np.array_equal(first, again)
        y_ref, _, _ = data.oracle()
        assert_close(first, y_ref, "repeatable prefill")
    finally:
        pw.pw_destroy(ctx)


def test_prefill_and_decode_tilings_agree():
    """The same tokens through a decode-sized launch (64-token items) and inside a prefill-
    sized launch give the same rows up to accumulation order."""
    shape = RAGGED
    T = 640
    data = LayerData(shape, 6, 0, T, real=range(shape.E))
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        y_big, _, _ = forward(ctx, data, T)
        x = torch.from_numpy(data.x[:200].view(np.int16)).cuda()
        y = torch.zeros_like(x)
        torch.cuda.synchronize()
        pw.pw_moe_forward(ctx, 0, x, 200, y, None, None, 0, pw.pw_get_stream(ctx))
        torch.cuda.synchronize()
        y_small = bf16_to_f64(y.cpu().numpy().view(np.uint16))
        y_ref, _, _ = data.oracle(tokens=range(200))
        assert_close(y_small, y_ref, "decode tiling")
        assert_close(y_big[:200], y_ref, "prefill tiling")
    finally:
        pw.pw_destroy(ctx)


def sample_tokens(ids, n=12, seed=0):
    """Token rows to check: the first, the last and a seeded random sample of the batch."""
    T = ids.shape[0]
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], r.choice(T, n - 2, replace=False)]))


def cover_tokens(ids, E):
    """Token rows to check on a layer with few experts: for every expert the first and the
    last token routed to it, so that every expert's prefill work items (and the first and
    last chunk of the largest and smallest token groups) are checked."""
    tok = set()
    for e in range(E):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        if len(rows):
            tok.update((int(rows[0]), int(rows[-1])))
    return np.array(sorted(tok))


@pytest.mark.parametrize("name", ["mixtral", "g128"])
def test_model_shaped_prefill_sampled_tokens(name):
    shape = syn.SHAPES[name]
    T = shape.prefill_T
    data = LayerData(shape, 1, 0, T)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        y, ids, w = forward(ctx, data, T)
        ids_all, _, _ = omoe.route(data.x, data.Wr, data.bias, shape.K)
        assert np.array_equal(ids, ids_all)  # top-K of every token, bit-exact
        tok = cover_tokens(ids_all, shape.E) if name == "mixtral" else sample_tokens(ids_all)
        if name == "mixtral":  # every expert, two tokens each at least
            assert all((ids_all[tok] == e).any(axis=1).sum() >= 2 for e in range(shape.E))
        y_ref, ids_ref, w_ref = data.oracle(tokens=tok)
        assert np.array_equal(ids[tok], ids_ref)
        assert np.allclose(w[tok], w_ref, rtol=1e-5, atol=1e-7)
        assert_close(y[tok], y_ref, f"{name} prefill T={T}")
    finally:
        pw.pw_destroy(ctx)
