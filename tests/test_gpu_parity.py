"""GPU parity: codes, dequantised weights, routing and layer outputs of libpw.so against
the float64 oracle on the same seeded inputs."""
import numpy as np
import pytest

import synthetic as syn
from oracle import ap
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


def run_layer(ctx, data, T, flags=0, y_init=None):
    x = torch.from_numpy(data.x.view(np.int16)).cuda()
    y = torch.zeros_like(x) if y_init is None else torch.from_numpy(y_init.view(np.int16)).cuda()
    ids = torch.zeros((T, data.shape.K), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, data.shape.K), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()  # inputs made on torch's stream; the layer runs on the ctx stream
    pw.pw_moe_forward(ctx, 0, x, T, y, ids, w, flags, pw.pw_get_stream(ctx))
    torch.cuda.synchronize()
    return bf16_to_f64(y.cpu().numpy().view(np.uint16)), ids.cpu().numpy(), w.cpu().numpy()


# ---------------------------------------------------------------- codes and weights
ODD = syn.LayerShape("odd", H=144, E=4, I=200, K=2, Is=0, L=1, bmax=8, bits=(3, 4, 5, 6, 7, 8),
                     sigma_lut=0.02, zipf_a=None, q_rule="uniform")


@pytest.mark.parametrize("shape_name", ["tiny", "odd"])
def test_unpack_and_dequant_bit_exact(shape_name):
    shape = syn.SHAPES["tiny"] if shape_name == "tiny" else ODD
    ctx = make_ctx(pw, shape, L=1, max_tokens=8)
    try:
        data = {}
        for e in range(shape.E):
            for u in (0, 1):
                idx, luts = syn.gen_block_np(shape, 21, 0, e, u)
                data[(e, u)] = (idx, luts)
                pw.pw_pack(ctx, 0, e, u, idx, np.concatenate([luts[b].ravel() for b in shape.bits]), shape.bmax)
        for (e, u), (idx, luts) in data.items():
            block = syn.block_id(0, e, u, shape.E)
            N, K = idx.shape
            planes = ap.pack_planes(idx, shape.bmax)
            for b in range(1, shape.bmax + 1):
                got = pw.pw_unpack_indices(ctx, block, b, N, K)
                assert np.array_equal(got, ap.unpack_indices(planes, b, K)), (e, u, b)
            for b in shape.bits:
                got = pw.pw_dequant(ctx, block, b, N, K)
                want = ap.dequant_fp16_bits(ap.unpack_indices(planes, b, K), luts[b])
                assert np.array_equal(got, want), (e, u, b)
    finally:
        pw.pw_destroy(ctx)


def test_pack_from_device_memory_matches_host_pack():
    shape = ODD
    ctx = make_ctx(pw, shape, L=1, max_tokens=8)
    try:
        idx, luts = syn.gen_block_np(shape, 5, 0, 1, 0)
        lut = np.concatenate([luts[b].ravel() for b in shape.bits])
        pw.pw_pack(ctx, 0, 0, 0, idx, lut, 5)
        pw.pw_pack(ctx, 0, 1, 0, torch.from_numpy(idx).cuda(), torch.from_numpy(lut.view(np.int16)).cuda(), 5)
        N, K = idx.shape
        for b in (1, 3, 5):
            a = pw.pw_unpack_indices(ctx, syn.block_id(0, 0, 0, shape.E), b, N, K)
            c = pw.pw_unpack_indices(ctx, syn.block_id(0, 1, 0, shape.E), b, N, K)
            assert np.array_equal(a, c) and np.array_equal(a, idx >> (8 - b))
        # pages above q_init are CPU-resident and cannot be read back
        with pytest.raises(pw.PwError) as ei:
            pw.pw_unpack_indices(ctx, syn.block_id(0, 1, 0, shape.E), 6, N, K)
        assert ei.value.status == pw.PW_ERR_STATE
    finally:
        pw.pw_destroy(ctx)


# ---------------------------------------------------------------- tiny layer, every kind of q mix
def test_tiny_layer_all_uniform_and_mixed_q():
    shape = syn.SHAPES["tiny"]
    T = shape.decode_T[0]
    data = LayerData(shape, 0, 0, T, real=range(shape.E), tiny=True)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx, q_init=shape.bmax)
        rng = np.random.default_rng(123)
        assignments = [np.full((shape.E, 2), b, dtype=np.int32) for b in shape.bits]
        assignments.append(data.q)
        assignments += [rng.choice(shape.bits, size=(shape.E, 2)).astype(np.int32) for _ in range(16)]
        for q in assignments:
            for e in range(shape.E):
                for u in (0, 1):
                    pw.pw_set_bits(ctx, syn.block_id(0, e, u, shape.E), int(q[e, u]))
            y, ids, w = run_layer(ctx, data, T)
            y_ref, ids_ref, w_ref = data.oracle(q=q)
            assert np.array_equal(ids, ids_ref)
            assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)
            assert_close(y, y_ref, f"q={q.tolist()}")
    finally:
        pw.pw_destroy(ctx)


def test_tiny_layer_accumulate_in_place_and_renorm():
    shape = syn.SHAPES["tiny"]
    T = shape.decode_T[0]
    data = LayerData(shape, 0, 0, T, real=range(shape.E), tiny=True)
    for renorm in (0, 1):
        ctx = make_ctx(pw, shape, L=1, max_tokens=T, renorm=renorm)
        try:
            data.load(pw, ctx)
            x = torch.from_numpy(data.x.view(np.int16)).cuda()
            torch.cuda.synchronize()
            pw.pw_moe_forward(ctx, 0, x, T, x, None, None, pw.PW_ACCUMULATE, pw.pw_get_stream(ctx))
            torch.cuda.synchronize()
            got = bf16_to_f64(x.cpu().numpy().view(np.uint16))
            y_ref, _, _ = data.oracle(renorm=bool(renorm))
            assert_close(got, bf16_to_f64(data.x) + y_ref, f"accumulate renorm={renorm}")
        finally:
            pw.pw_destroy(ctx)


# Split K parts.  NARROW: a routed down projection of one 128-column stage (I <= 128) beside
# a long shared down projection (Is = 1200: ten stages), whose K parts hit the cap of 8 and
# come out five parts of two stages.  LONGDOWN: a routed down projection of 40 stages
# (I = 5008, not a multiple of 128), split at decode sizes into parts of 14, 14 and 12.
NARROW = syn.LayerShape("narrow", H=256, E=8, I=112, K=2, Is=1200, L=1, bmax=8, bits=(3, 4, 5, 6, 7, 8),
                        sigma_lut=0.02, zipf_a=None, q_rule="uniform")
LONGDOWN = syn.LayerShape("longdown", H=256, E=6, I=5008, K=2, Is=0, L=1, bmax=8, bits=(3, 4, 5, 6, 7, 8),
                          sigma_lut=0.02, zipf_a=None, q_rule="uniform")


@pytest.mark.parametrize("name,T", [("narrow", 8), ("narrow", 40), ("longdown", 24), ("longdown", 200)])
def test_split_k_parts(name, T):
    shape = NARROW if name == "narrow" else LONGDOWN
    data = LayerData(shape, 4, 0, T, real=range(shape.E))
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        y, ids, w = run_layer(ctx, data, T)
        y_ref, ids_ref, w_ref = data.oracle()
        assert np.array_equal(ids, ids_ref)
        assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)
        assert_close(y, y_ref, f"{name} T={T}")
        again, _, _ = run_layer(ctx, data, T)  # the parts are added in a fixed order
        assert np.array_equal(y, again)
    finally:
        pw.pw_destroy(ctx)


# ---------------------------------------------------------------- model-shaped layers
# every decode batch the benchmarks time: Qwen-shaped T = 1, 16, 64, 256; 128-expert T = 1, 32,
# 256; Mixtral-shaped T = 1, 8, 64, 256
CASES = [("qwen", 1), ("qwen", 16), ("qwen", 64), ("qwen", 256), ("g128", 1), ("g128", 32), ("g128", 256),
         ("mixtral", 1), ("mixtral", 8), ("mixtral", 64), ("mixtral", 256)]


def expert_cover(ids, E):
    """The first and the last token routed to each expert (every expert's work items)."""
    tok = set()
    for e in range(E):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        if len(rows):
            tok.update((int(rows[0]), int(rows[-1])))
    return np.array(sorted(tok))


@pytest.mark.parametrize("name,T", CASES)
def test_model_shaped_layer(name, T):
    shape = syn.SHAPES[name]
    data = LayerData(shape, 1, 0, T)
    ctx = make_ctx(pw, shape, L=1, max_tokens=max(T, 8))
    try:
        data.load(pw, ctx)
        y, ids, w = run_layer(ctx, data, T)
        # the Mixtral shape's dense float64 experts are large: check its bigger batches on the
        # first and last token of every expert (rows are independent); routing on every token
        tok = expert_cover(ids, shape.E) if (name == "mixtral" and T > 8) else None
        ids_all, w_all, _ = omoe.route(data.x, data.Wr, data.bias, shape.K)
        assert np.array_equal(ids, ids_all)
        assert np.allclose(w, w_all, rtol=1e-5, atol=1e-7)
        y_ref, _, _ = data.oracle(tokens=tok)
        assert_close(y if tok is None else y[tok], y_ref, f"{name} T={T}")
    finally:
        pw.pw_destroy(ctx)


@pytest.mark.parametrize("name,T,qmode", [("qwen", 16, "mixed"), ("qwen", 64, "mixed"), ("g128", 32, "default")])
def test_layer_output_is_bitwise_repeatable(name, T, qmode):
    """The expert kernels overlap many asynchronous producers and consumers; a missed
    synchronisation shows up first as run-to-run differences, so the same inputs must give
    bit-identical outputs on every launch."""
    shape = syn.SHAPES[name]
    q = None
    if qmode == "mixed":  # alternate a register-LUT width with the two-slot q = 8 tables
        q = np.where(np.arange(shape.E)[:, None] % 2 == 0, 4, 8) * np.ones((1, 2), dtype=np.int32)
    data = LayerData(shape, 1, 0, T, q=q)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        first, _, _ = run_layer(ctx, data, T)
        for _ in range(5):
            again, _, _ = run_layer(ctx, data, T)
            assert np.array_equal(first, again)
        y_ref, _, _ = data.oracle()
        assert_close(first, y_ref, f"{name} T={T} q={qmode}")
    finally:
        pw.pw_destroy(ctx)


@pytest.mark.parametrize("name,T", [("tiny", 8), ("qwen", 16)])
def test_prenorm_layer(name, T):
    shape = syn.SHAPES[name]
    data = LayerData(shape, 4, 0, T, prenorm=True, tiny=(name == "tiny"))
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        y, ids, w = run_layer(ctx, data, T, flags=pw.PW_PRENORM)
        y_ref, ids_ref, w_ref = data.oracle()
        assert np.array_equal(ids, ids_ref)
        assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)
        assert_close(y, y_ref, f"{name} T={T}")
    finally:
        pw.pw_destroy(ctx)


@pytest.mark.parametrize("name,T,prenorm", [("qwen", 16, False), ("qwen", 64, True)])
def test_gated_shared_expert(name, T, prenorm):
    """The shared expert scaled per token by sigmoid(x . w_sg); removing the gate restores the
    ungated layer."""
    shape = syn.SHAPES[name]
    data = LayerData(shape, 8, 0, T, prenorm=prenorm)
    wsg = np.random.default_rng(8).normal(0.0, 2.0 / np.sqrt(shape.H), size=shape.H)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        flags = pw.PW_PRENORM if prenorm else 0
        pw.pw_set_shared_gate(ctx, 0, wsg.astype(np.float32))
        y, _, _ = run_layer(ctx, data, T, flags=flags)
        y_ref, _, _ = data.oracle(shared_gate=wsg.astype(np.float32).astype(np.float64))
        assert_close(y, y_ref, f"gated {name} T={T}")
        y_plain_ref, _, _ = data.oracle()
        assert not np.allclose(y_ref, y_plain_ref, rtol=1e-2)  # the gate matters at this scale
        pw.pw_set_shared_gate(ctx, 0, None)
        y2, _, _ = run_layer(ctx, data, T, flags=flags)
        assert_close(y2, y_plain_ref, f"ungated again {name} T={T}")
    finally:
        pw.pw_destroy(ctx)


# decode batches, one token to sixteen (four lanes per expert), and prefill batches (a warp
# per expert)
@pytest.mark.parametrize("name,T,prenorm", [("qwen", 1, True), ("qwen", 16, False), ("qwen", 16, True),
                                            ("qwen", 600, True), ("g128", 1100, False)])
def test_routed_input_features_match_eq5(name, T, prenorm):
    """Eq. 5's phi per expert from the device sums, against the oracle's definition on the
    oracle's routing of the same tokens; the planner reads them when obs->phi is NULL."""
    from oracle import planner as opl
    shape = syn.SHAPES[name]
    data = LayerData(shape, 9, 0, T, prenorm=prenorm)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        flags = pw.PW_PRENORM if prenorm else 0
        for _ in range(2):  # the same tokens twice: the ratios and the maximum are unchanged
            run_layer(ctx, data, T, flags=flags)
        phi = pw.pw_routing_features(ctx, 0, shape.E)
        ids, w, _ = omoe.route(data.x, data.Wr, data.bias, shape.K, prenorm=prenorm)
        xin = bf16_to_f64(data.x)
        if prenorm:
            xin = omoe.rmsnorm(xin)
        ref = opl.routed_input_features(xin, ids, w, shape.E)
        assert np.allclose(phi, ref, rtol=1e-4, atol=1e-6)
        assert (phi[:, 0] > 0).sum() == len(set(ids.ravel().tolist()))
        # the planner's default features are these, expanded to both blocks of each expert
        n = shape.E * 2
        off = syn.gen_planner_offline_np(n, list(shape.bits), 4, 3)
        off["n_stages"] = 3
        obs = dict(T_blk=16, F_blk=2, B_KV=1.0e6, R=8, mass=None, phi=None)
        p_dev = pw.pw_plan_step(ctx, n, obs, off)
        obs["phi"] = np.repeat(phi, 2, axis=0)
        p_exp = pw.pw_plan_step(ctx, n, obs, off)
        assert p_dev == p_exp and p_dev["entries"]
        pw.pw_routing_features(ctx, 0, shape.E, reset=True)
        assert not pw.pw_routing_features(ctx, 0, shape.E).any()
    finally:
        pw.pw_destroy(ctx)


def test_routing_statistics_match_eq1_inputs():
    shape = syn.SHAPES["tiny"]
    T = shape.decode_T[0]
    data = LayerData(shape, 0, 0, T, real=range(shape.E), tiny=True)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        for _ in range(3):
            run_layer(ctx, data, T)
        cnt, ws = pw.pw_routing_stats(ctx, 0, shape.E, reset=True)
        _, ids_ref, w_ref = data.oracle()
        want_cnt = np.bincount(ids_ref.ravel(), minlength=shape.E) * 3
        want_ws = np.zeros(shape.E)
        for t in range(T):
            for k in range(shape.K):
                want_ws[ids_ref[t, k]] += 3 * w_ref[t, k]
        assert np.array_equal(cnt, want_cnt)
        assert np.allclose(ws, want_ws, rtol=1e-5)
        cnt2, _ = pw.pw_routing_stats(ctx, 0, shape.E)
        assert not cnt2.any()
    finally:
        pw.pw_destroy(ctx)


def test_stack_graph_replay_equals_layer_by_layer():
    shape = syn.LayerShape("stack", H=256, E=8, I=128, K=2, Is=64, L=3, bmax=8, bits=(3, 4, 5, 6, 7, 8),
                           sigma_lut=0.02, zipf_a=1.0, q_rule="uniform")
    T = 12
    ctx = make_ctx(pw, shape, L=3, max_tokens=T)
    try:
        for layer in range(3):
            d = LayerData(shape, 2, layer, T, real=range(shape.E))
            d.load(pw, ctx, layer_slot=layer)
        x0 = syn.gen_tokens_np(shape, 9, 0, T)
        xa = torch.from_numpy(x0.view(np.int16)).cuda()
        xb = xa.clone()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for layer in range(3):
                pw.pw_moe_forward(ctx, layer, xa, T, xa, None, None, pw.PW_ACCUMULATE | pw.PW_PRENORM, s)
            pw.pw_stack_forward(ctx, xb, T, s)  # first call captures and replays
        s.synchronize()
        assert torch.equal(xa, xb)
        xc = torch.from_numpy(x0.view(np.int16)).cuda()
        x0_dev = torch.from_numpy(x0.view(np.int16)).cuda()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            pw.pw_stack_forward(ctx, xc, T, s)  # new buffer: new graph
            xd = xc.clone()
            xc.copy_(x0_dev)
            pw.pw_stack_forward(ctx, xc, T, s)  # replay of the cached graph
        s.synchronize()
        assert torch.equal(xc, xd) and torch.equal(xc, xa)
        yh = np.zeros_like(x0)
        pw.pw_stack_forward_host(ctx, x0, T, yh)
        assert np.array_equal(yh.view(np.int16), xa.cpu().numpy())
    finally:
        pw.pw_destroy(ctx)


# ---------------------------------------------------------------- the two decode kernels
@pytest.mark.parametrize("gemv", [0, 8])
@pytest.mark.parametrize("name,T", [("tiny", 8), ("odd", 6), ("qwen", 16), ("qwen", 64), ("g128", 32),
                                    ("mixtral", 8), ("longdown", 24)])
def test_decode_item_paths(name, T, gemv):
    """Routed items on the tensor cores only (threshold 0) and, with threshold 8, every item of
    up to 8 tokens on the CUDA cores: both against the oracle and bit-for-bit repeatable."""
    shape = {"odd": ODD, "longdown": LONGDOWN}.get(name) or syn.SHAPES[name]
    small = name in ("tiny", "odd", "longdown")
    data = LayerData(shape, 6, 0, T, real=range(shape.E) if small else None, tiny=(name == "tiny"))
    ctx = make_ctx(pw, shape, L=1, max_tokens=T)
    try:
        data.load(pw, ctx)
        pw.pw_set_gemv_tokens(ctx, gemv)
        y, ids, w = run_layer(ctx, data, T)
        y_ref, ids_ref, w_ref = data.oracle()
        assert np.array_equal(ids, ids_ref)
        assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)
        assert_close(y, y_ref, f"{name} T={T} gemv<={gemv}")
        again, _, _ = run_layer(ctx, data, T)
        assert np.array_equal(y, again)
    finally:
        pw.pw_destroy(ctx)


def test_gemv_threshold_is_checked():
    shape = syn.SHAPES["tiny"]
    ctx = make_ctx(pw, shape, L=1, max_tokens=8)
    try:
        for bad in (-1, 9):
            with pytest.raises(pw.PwError) as ei:
                pw.pw_set_gemv_tokens(ctx, bad)
            assert ei.value.status == pw.PW_ERR_INVALID
        pw.pw_set_gemv_tokens(ctx, 0)
        pw.pw_set_gemv_tokens(ctx, 8)
    finally:
        pw.pw_destroy(ctx)
