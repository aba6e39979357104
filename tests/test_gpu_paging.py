"""Weight-page movement on the device: the Fig. 4 walk-through, ordering rules, poisoned
retired pages, host-injected copy/allocation faults and resident-bytes accounting.
Every failure here is made on the host; no GPU fault is ever provoked."""
import numpy as np
import pytest

import synthetic as syn
from conftest import load_golden
from oracle import ap, pages

from gpu_helpers import LayerData, assert_close, bf16_to_f64, make_ctx

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pw = pytest.importorskip("any_precision_bit_gb300")

STATE = {pw.PW_PAGE_GPU: "gpu", pw.PW_PAGE_CPU: "cpu", pw.PW_PAGE_TO_CPU: "to_cpu", pw.PW_PAGE_TO_GPU: "to_gpu"}


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from any_precision_bit_gb300 import _build
    _build.build()


@pytest.fixture()
def tiny():
    shape = syn.SHAPES["tiny"]
    T = shape.decode_T[0]
    data = LayerData(shape, 0, 0, T, real=range(shape.E), tiny=True)
    ctx = make_ctx(pw, shape, L=1, max_tokens=T, flags=pw.PW_FLAG_POISON)
    data.load(pw, ctx, q_init=shape.bmax)
    yield shape, T, data, ctx
    pw.pw_destroy(ctx)


def committed_q(ctx, shape):
    q = np.zeros((shape.E, 2), dtype=np.int32)
    for e in range(shape.E):
        for u in (0, 1):
            q[e, u] = pw.pw_query(ctx, syn.block_id(0, e, u, shape.E)).q
    return q


def forward_matches_oracle(ctx, shape, data, T):
    x = torch.from_numpy(data.x.view(np.int16)).cuda()
    y = torch.zeros_like(x)
    torch.cuda.synchronize()
    pw.pw_moe_forward(ctx, 0, x, T, y, None, None, 0, pw.pw_get_stream(ctx))
    torch.cuda.synchronize()
    y_ref, _, _ = data.oracle(q=committed_q(ctx, shape))
    assert_close(bf16_to_f64(y.cpu().numpy().view(np.uint16)), y_ref)


def test_fig4_walkthrough_on_device(tiny):
    """Replays the Fig. 4 sequence exactly: transfers are held in flight (host-side) until
    the walk-through says they landed."""
    shape, T, data, ctx = tiny
    g = load_golden("fig4_scenario.json")
    e = data.routed[0]
    block = syn.block_id(0, e, 1, shape.E)  # the down block of a routed expert
    model = pages.BlockPages(g["bits"], g["bmax"], g["q0"])
    for ev in g["events"]:
        op = ev["op"]
        if op == "offload":
            pw.pw_set_fault(ctx, 3, 1)
            pw.pw_offload(ctx, block, ev["arg"])
            model.offload(ev["arg"])
        elif op == "reload":
            pw.pw_set_fault(ctx, 3, 1)
            pw.pw_reload(ctx, block, ev["arg"])
            model.reload(ev["arg"])
        elif op == "landed":
            pw.pw_sync_io(ctx)
            pw.pw_set_fault(ctx, 3, 0)  # pw_query now observes the landed copies
            model.copies_landed()
        elif op == "commit":
            assert pw.pw_commit(ctx) == model.commit() == ev["applied"]
        info = pw.pw_query(ctx, block)
        assert info.q == ev["q"], ev
        assert [STATE[s] for s in info.state[:shape.bmax]] == ev["state"], ev
        # inference reads exactly the committed bitwidth at every point of the sequence
        forward_matches_oracle(ctx, shape, data, T)


def test_illegal_orders_are_refused(tiny):
    shape, T, data, ctx = tiny
    block = syn.block_id(0, data.routed[0], 0, shape.E)
    pw.pw_set_fault(ctx, 3, 1)  # keep the offload in flight
    pw.pw_offload(ctx, block, 4)
    with pytest.raises(pw.PwError) as ei:
        pw.pw_reload(ctx, block, 6)  # pages 4, 5 still in transfer to the CPU
    assert ei.value.status == pw.PW_ERR_BUSY
    with pytest.raises(pw.PwError) as ei:
        pw.pw_set_bits(ctx, block, 5)
    assert ei.value.status == pw.PW_ERR_BUSY
    pw.pw_sync_io(ctx)
    pw.pw_set_fault(ctx, 3, 0)
    pw.pw_commit(ctx)
    with pytest.raises(pw.PwError) as ei:
        pw.pw_set_bits(ctx, block, 6)  # planes 4, 5 are CPU-resident
    assert ei.value.status == pw.PW_ERR_STATE
    with pytest.raises(pw.PwError) as ei:
        pw.pw_offload(ctx, block, 5)  # offload must lower
    assert ei.value.status == pw.PW_ERR_STATE
    pw.pw_set_bits(ctx, block, 3)  # lowering without moving pages is always allowed
    forward_matches_oracle(ctx, shape, data, T)


def test_injected_copy_and_allocation_faults_roll_back(tiny):
    shape, T, data, ctx = tiny
    block = syn.block_id(0, data.routed[0], 1, shape.E)
    # a failed offload copy keeps the pages on the GPU (q stays lowered)
    pw.pw_set_fault(ctx, 1, 1)
    pw.pw_offload(ctx, block, 4)
    pw.pw_sync_io(ctx)
    with pytest.raises(pw.PwError) as ei:
        pw.pw_commit(ctx)
    assert ei.value.status == pw.PW_ERR_CUDA
    info = pw.pw_query(ctx, block)
    assert info.q == 4 and [info.state[p] for p in range(6)] == [pw.PW_PAGE_GPU] * 6
    pw.pw_set_bits(ctx, block, 6)
    forward_matches_oracle(ctx, shape, data, T)
    # clean offload, then an allocation fault on reload changes nothing
    pw.pw_offload(ctx, block, 3)
    pw.pw_sync_io(ctx)
    pw.pw_commit(ctx)
    pw.pw_set_fault(ctx, 2, 1)
    with pytest.raises(pw.PwError) as ei:
        pw.pw_reload(ctx, block, 6)
    assert ei.value.status == pw.PW_ERR_OOM
    info = pw.pw_query(ctx, block)
    assert info.q == 3 and info.pending_q == 0
    assert [info.state[p] for p in range(3, 6)] == [pw.PW_PAGE_CPU] * 3
    # a failed reload copy leaves the pages CPU-resident and q un-raised
    pw.pw_set_fault(ctx, 1, 2)
    pw.pw_reload(ctx, block, 5)
    pw.pw_sync_io(ctx)
    with pytest.raises(pw.PwError):
        pw.pw_commit(ctx)
    info = pw.pw_query(ctx, block)
    assert info.q == 3 and [info.state[p] for p in range(3, 6)] == [pw.PW_PAGE_CPU] * 3
    forward_matches_oracle(ctx, shape, data, T)
    # and a clean reload works afterwards
    pw.pw_set_fault(ctx, 1, 0)
    pw.pw_reload(ctx, block, 6)
    pw.pw_sync_io(ctx)
    assert pw.pw_commit(ctx) == 1
    assert pw.pw_query(ctx, block).q == 6
    forward_matches_oracle(ctx, shape, data, T)


def test_resident_bytes_follow_eq3(tiny):
    shape, T, data, ctx = tiny
    def expected():
        tot = 0
        for e in range(shape.E):
            for u in (0, 1):
                N, K = syn.block_shape(shape, u)
                tot += ap.block_bytes(N, K, shape.bits, pw.pw_query(ctx, syn.block_id(0, e, u, shape.E)).q)
        return tot
    assert pw.pw_memory(ctx).resident_bytes == expected()
    block = syn.block_id(0, 2, 0, shape.E)
    before = pw.pw_memory(ctx).resident_bytes
    pw.pw_offload(ctx, block, 3)
    N, K = syn.block_shape(shape, 0)
    assert before - pw.pw_memory(ctx).resident_bytes == ap.delta_bytes(N, K, shape.bits, 6, 3)
    info = pw.pw_query(ctx, block)
    for b in shape.bits:
        assert info.M[b] == ap.block_bytes(N, K, shape.bits, b)
    pw.pw_sync_io(ctx)
    pw.pw_commit(ctx)
    assert pw.pw_memory(ctx).resident_bytes == expected()


def test_kv_allocator_follows_the_held_pages(tiny):
    """The KV-block allocator attached to a context: its weight bytes are the device pages
    the context holds, so an offload frees KV blocks only once pw_commit retires its pages,
    and a reload takes them back when it allocates its pages (Sec. 3.3)."""
    shape, T, data, ctx = tiny
    B = 4096
    mem = pw.pw_memory(ctx)
    W0 = mem.held_bytes
    assert W0 == mem.resident_bytes  # every page resident, LUT rows a multiple of 128
    S = W0 + 40 * B + 123
    kv = pw.pw_kv_create(S, B)
    try:
        pw.pw_kv_attach(kv, ctx)
        pw.pw_kv_grow(kv, 7, 5)
        st = pw.pw_kv_get_stats(kv)
        assert st["weight_bytes"] == W0 and st["free_blocks"] == (S - W0) // B - 5
        block = syn.block_id(0, data.routed[0], 0, shape.E)
        N, K = syn.block_shape(shape, 0)
        delta = ap.delta_bytes(N, K, shape.bits, 6, 3)
        pw.pw_set_fault(ctx, 3, 1)  # hold the copy in flight
        pw.pw_offload(ctx, block, 3)
        assert pw.pw_memory(ctx).resident_bytes == W0 - delta
        assert pw.pw_kv_get_stats(kv) == st  # the pages are still held
        pw.pw_sync_io(ctx)
        pw.pw_set_fault(ctx, 3, 0)
        pw.pw_commit(ctx)
        st = pw.pw_kv_get_stats(kv)
        assert st["weight_bytes"] == W0 - delta
        assert st["free_blocks"] == (S - W0 + delta) // B - 5
        assert st["headroom_bytes"] == S - (W0 - delta) - 5 * B
        pw.pw_reload(ctx, block, 6)  # allocates the pages at once
        assert pw.pw_kv_get_stats(kv)["weight_bytes"] == W0
        pw.pw_sync_io(ctx)
        assert pw.pw_commit(ctx) == 1
        assert pw.pw_kv_get_stats(kv)["free_blocks"] == (S - W0) // B - 5
        pw.pw_kv_set_weight_bytes(kv, 0)  # detached
        assert pw.pw_kv_get_stats(kv)["weight_bytes"] == 0
    finally:
        pw.pw_kv_destroy(kv)
