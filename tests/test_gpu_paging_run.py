"""The dynamic paging run (PagedWeight Sec. 3.2 and Sec. 3.3, Fig. 4) on the device, its KV
pressure coming from a running KV-block allocator: a seeded request schedule (arrivals with
prompt blocks, growth one block at a time, each growth announced a step ahead, completions)
is served by ``pw_kv`` attached to the context, so the weight pages the GPU holds and the KV
blocks share one budget.  Every step the greedy planner (Eqs. 3-8, Algorithm 1) reads F_blk
from the allocator, the plan is applied with pw_offload / pw_reload on the side stream and
pw_commit between steps (retired pages become KV headroom), retired device pages are
poisoned with 0xFF, and at EVERY step every layer's output is compared with the float64
oracle at that step's committed bitwidths; the allocator's accounting is checked against the
oracle's (oracle/kv.py) at every step too.

The layers have the structure of the Qwen1.5-MoE-shaped stack (60 routed experts, top-4,
hot/cold bitwidths under a Zipf(1.1) router prior, a dense shared expert, bits 3..8) at
reduced widths, so that the oracle can check all 200 steps; the KV block size is scaled with
the weight bytes so that the demand peak pushes blocks toward their floors and the drain
restores them.  A second test serves the schedule on full-size Qwen-shaped layers and checks
the oracle at a handful of steps."""
import numpy as np
import pytest

import synthetic as syn
from oracle import ap
from oracle import kv as okv
from oracle import moe as omoe
from oracle import planner as opl

from gpu_helpers import assert_close, bf16_to_f64, make_ctx, lut_concat

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pw = pytest.importorskip("any_precision_bit_gb300")

MINI = syn.LayerShape("qwen_mini", H=256, E=60, I=128, K=4, Is=512, L=2, bmax=8, bits=(3, 4, 5, 6, 7, 8),
                      sigma_lut=0.02, zipf_a=1.1, q_rule="hot_cold")
STEPS, T, T_BLK, R = 200, 64, 16, 8


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from any_precision_bit_gb300 import _build
    _build.build()


class Stack:
    """Seeded layers of `shape`, packed into a context with poisoned retired pages."""

    def __init__(self, shape, L, seed=0):
        self.shape, self.L, self.seed = shape, L, seed
        self.ctx = make_ctx(pw, shape, L=L, max_tokens=T, flags=pw.PW_FLAG_POISON)
        self.layers = []
        for l in range(L):
            Wr, bias, ranks = syn.gen_router_np(shape, seed, l)
            q = syn.gen_q_assignment(shape, seed, l, ranks)
            experts = {}
            for e in range(shape.E):
                gi, gl = syn.gen_block_np(shape, seed, l, e, 0)
                di, dl = syn.gen_block_np(shape, seed, l, e, 1)
                experts[e] = (gi, gl, di, dl)
                pw.pw_pack(self.ctx, l, e, 0, gi, lut_concat(gl, shape.bits), int(q[e, 0]))
                pw.pw_pack(self.ctx, l, e, 1, di, lut_concat(dl, shape.bits), int(q[e, 1]))
            shared = syn.gen_shared_np(shape, seed, l)
            pw.pw_set_router(self.ctx, l, Wr, bias)
            pw.pw_set_shared(self.ctx, l, shared[0], shared[1])
            self.layers.append(dict(Wr=Wr, bias=bias, q0=q, experts=experts, shared=shared))
        self.n_blocks = L * shape.E * 2
        self._w = {}

    def committed_q(self, l):
        E = self.shape.E
        return np.array([[pw.pw_query(self.ctx, syn.block_id(l, e, u, E)).q for u in (0, 1)] for e in range(E)],
                        dtype=np.int32)

    def tokens(self, step, l):
        """Step-dependent tokens whose sorted logits are separated by >= 1e-3 among ranks
        1..K+1, so that the top-K decision does not depend on the rounding of fp32 logits."""
        sh, lay = self.shape, self.layers[l]
        seed = self.seed * 100003 + 7 + step
        x = syn.gen_tokens_np(sh, seed, l, T)

        def ok(row):
            s = np.sort(omoe.router_logits(row[None], lay["Wr"], lay["bias"], True)[0])[::-1][: sh.K + 1]
            return np.all(-np.diff(s) >= 1e-3)
        for t in range(T):
            a = 0
            while not ok(x[t]):
                a += 1
                x[t] = syn.gen_token_np(sh, seed, l, t, a)
        return x

    def oracle(self, l, x, q):
        """The float64 layer at bitwidths q on the rows of x; the dense weight of each
        (block, q) is the oracle's own block_weight, memoised across steps."""
        lay, sh = self.layers[l], self.shape
        n = x.shape[0]
        ids, w, _ = omoe.route(x, lay["Wr"], lay["bias"], sh.K, prenorm=True)
        xf = omoe.rmsnorm(bf16_to_f64(x))
        y = np.zeros((n, sh.H))
        o = np.zeros((n, sh.K, sh.H))
        for e in np.unique(ids):
            e = int(e)
            W = []
            for u in (0, 1):
                key = (l, e, u, int(q[e, u]))
                if key not in self._w:
                    self._w[key] = omoe.block_weight(lay["experts"][e][2 * u], lay["experts"][e][2 * u + 1], sh.bmax,
                                                     int(q[e, u]))
                W.append(self._w[key])
            rows, slots = np.nonzero(ids == e)
            o[rows, slots] = omoe.expert_ffn(xf[rows], W[0], W[1])
        for k in range(sh.K):
            y += w[:, k:k + 1] * o[:, k, :]
        if ("shared", l) not in self._w:
            self._w[("shared", l)] = (bf16_to_f64(lay["shared"][0]), bf16_to_f64(lay["shared"][1]))
        y += omoe.expert_ffn(xf, *self._w[("shared", l)])
        return y

    def forward(self, l, x):
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        yd = torch.zeros_like(xd)
        torch.cuda.synchronize()
        pw.pw_moe_forward(self.ctx, l, xd, T, yd, None, None, pw.PW_PRENORM, pw.pw_get_stream(self.ctx))
        torch.cuda.synchronize()
        return bf16_to_f64(yd.cpu().numpy().view(np.uint16))

    def resident_bytes_eq3(self):
        tot = 0
        for l in range(self.L):
            q = self.committed_q(l)
            for e in range(self.shape.E):
                for u in (0, 1):
                    N, K = syn.block_shape(self.shape, u)
                    tot += ap.block_bytes(N, K, self.shape.bits, int(q[e, u]))
        return tot


def oracle_plan(st, off, obs):
    """The oracle planner (Algorithm 1 restated) on the blocks that can take a step now: no
    page in transfer and no landed reload awaiting its commit.  Routing mass (Eq. 1) from the
    context's accumulated routing-weight sums."""
    sh, E = st.shape, st.shape.E
    idle, q, q0, ut, ly, ex, M = [], [], [], [], [], [], []
    for l in range(st.L):
        for e in range(E):
            for u in (0, 1):
                b = syn.block_id(l, e, u, E)
                info = pw.pw_query(st.ctx, b)
                busy = info.pending_q != 0 or any(info.state[p] in (pw.PW_PAGE_TO_CPU, pw.PW_PAGE_TO_GPU)
                                                  for p in range(sh.bmax))
                if busy:
                    continue
                N, K = syn.block_shape(sh, u)
                idle.append(b)
                q.append(info.q)
                q0.append(int(st.layers[l]["q0"][e, u]))
                ut.append(u)
                ly.append(l)
                ex.append(e)
                M.append([ap.block_bytes(N, K, sh.bits, bb) for bb in sh.bits])
    mass = np.array([pw.pw_routing_stats(st.ctx, l, E)[1] for l in range(st.L)], dtype=np.float64)
    for l in range(st.L):  # normalised per layer, summed in expert order
        tot = 0.0
        for e in range(E):
            tot += float(mass[l, e])
        mass[l] = mass[l] / tot if tot > 0 else 1.0 / E
    idx = np.array(idle, dtype=np.int64)
    sub = dict(off, s=np.asarray(off["s"])[idx])
    if obs.get("rho_hat") is not None:  # a batch-level residual table, re-indexed like the blocks
        sub["rho_hat"] = np.asarray(obs["rho_hat"])[idx]
    blocks = opl.Blocks(list(sh.bits), q, ut, ly, ex, np.array(M, dtype=np.float64), sub["s"])
    phi = None if obs.get("phi") is None else np.asarray(obs["phi"])[idx]
    _, chosen, D = opl.plan_step(blocks, mass, phi, sub, off["n_stages"], obs["T_blk"], obs["F_blk"], obs["B_KV"])
    if D > 0:
        stage, plan, total = chosen
        return 1, stage, D, [(idle[i], a, b, d) for i, (a, b, d) in plan.items()]
    plan, total = opl.reload_plan(blocks, q0, mass, phi, sub, obs["T_blk"], obs["F_blk"], obs["B_KV"], obs["R"])
    return (2 if total > 0 else 0), -1, D, [(idle[i], a, b, d) for i, (a, b, d) in plan.items()]


class Serving:
    """The request side of a serving loop on two allocators in step: the library's (attached
    to the context, so its weight bytes are the pages the context holds) and the oracle's
    accounting, given the same held bytes.  A request whose arrival or growth does not fit
    is dropped (its blocks are released and its later events skipped)."""

    def __init__(self, st, S, B):
        self.ctx = st.ctx
        self.kv = pw.pw_kv_create(S, B)
        pw.pw_kv_attach(self.kv, st.ctx)
        self.ref = okv.KVAllocator(S, B)
        self.dropped = set()

    def close(self):
        pw.pw_kv_destroy(self.kv)

    def sync_weights(self):
        self.ref.set_weight_bytes(pw.pw_memory(self.ctx).held_bytes)

    def apply(self, events):
        self.sync_weights()
        for ev in events:
            kind, r = ev[0], ev[1]
            if r in self.dropped:
                continue
            if kind == "finish":
                assert pw.pw_kv_release(self.kv, r) == self.ref.release(r)
            elif kind == "announce":
                pw.pw_kv_announce(self.kv, r, ev[2])
                self.ref.announce(r, ev[2])
            else:  # arrive / grow
                try:
                    want = self.ref.grow(r, ev[2])
                except okv.KVError:
                    want = None
                try:
                    got = [int(i) for i in pw.pw_kv_grow(self.kv, r, ev[2])]
                except pw.PwError as e:
                    assert e.status == pw.PW_ERR_OOM
                    got = None
                assert got == want, (kind, r)
                if got is None:
                    self.dropped.add(r)
                    pw.pw_kv_release(self.kv, r)
                    self.ref.release(r)
        return self.stats()

    def stats(self):
        self.sync_weights()
        got = pw.pw_kv_get_stats(self.kv)
        assert got == self.ref.stats()
        return got


def run_requests(st, off, S, B, check_steps, check_layers, check_tokens=None, check_plans=False):
    schedule = syn.gen_kv_requests(STEPS, st.seed)
    srv = Serving(st, S, B)
    log = []
    try:
        for step in range(STEPS):
            F = srv.apply(schedule[step])["free_blocks"]
            obs = dict(T_blk=T_BLK, F_blk=int(F), B_KV=float(B), R=R, mass=None,
                       phi=syn.gen_phi_np(st.n_blocks, st.seed, step))
            if check_plans:
                pw.pw_set_fault(st.ctx, 3, 1)  # hold: no transfer is observed landing until the plan is compared
                want = oracle_plan(st, off, obs)
            plan = pw.pw_plan_step(st.ctx, st.n_blocks, obs, off)
            if check_plans:
                pw.pw_set_fault(st.ctx, 3, 0)
                assert (plan["kind"], plan["stage"], plan["D"]) == want[:3], f"step {step}"
                assert plan["entries"] == want[3], f"step {step}"
            for block, fb, tb, _ in plan["entries"]:
                if tb < fb:
                    pw.pw_offload(st.ctx, block, tb)
                else:
                    pw.pw_reload(st.ctx, block, tb)
            pw.pw_commit(st.ctx)  # landed offloads retire their pages (KV headroom), landed reloads raise q
            for l in range(st.L):
                x = st.tokens(step, l)
                y = st.forward(l, x)
                if step in check_steps and l in check_layers:
                    q = st.committed_q(l)
                    rows = np.arange(T) if check_tokens is None else (np.arange(check_tokens) + 5 * step) % T
                    assert_close(y[rows], st.oracle(l, x[rows], q), f"step {step} layer {l}")
            kv = srv.stats()
            log.append(dict(step=step, kind=plan["kind"], n=len(plan["entries"]), F_blk=int(F),
                            resident=pw.pw_memory(st.ctx).resident_bytes, used=kv["used_blocks"],
                            free_after=kv["free_blocks"]))
    finally:
        srv.close()
    return log, srv.dropped


def offline_inputs(st):
    off = syn.gen_planner_offline_np(st.n_blocks, list(st.shape.bits), 4, st.seed)
    off["n_stages"] = 3
    return off


def budget(st, peak_frac):
    """Block size and budget: the schedule's demand peak asks for peak_frac of the resident
    weight bytes, and the budget leaves T_blk + R free blocks over the packed weights."""
    start = pw.pw_memory(st.ctx).held_bytes
    live, peak = {}, 0
    for events in syn.gen_kv_requests(STEPS, st.seed):
        for ev in events:
            if ev[0] == "finish":
                live.pop(ev[1])
            elif ev[0] in ("arrive", "grow"):
                live[ev[1]] = live.get(ev[1], 0) + ev[2]
        peak = max(peak, sum(live.values()))
    B = int(peak_frac * start / peak)
    return start + (T_BLK + R) * B, B


def test_paging_run_every_step_matches_oracle():
    st = Stack(MINI, L=MINI.L)
    try:
        start = st.resident_bytes_eq3()
        assert pw.pw_memory(st.ctx).resident_bytes == start
        S, B = budget(st, 0.3)
        log, dropped = run_requests(st, offline_inputs(st), S, B, check_steps=set(range(STEPS)),
                                    check_layers=range(st.L), check_plans=True)
        pw.pw_sync_io(st.ctx)
        pw.pw_commit(st.ctx)
        kinds = [r["kind"] for r in log]
        resident = [r["resident"] for r in log]
        assert 1 in kinds and 2 in kinds          # both offload and reload plans were applied
        assert min(resident) < 0.8 * start        # the demand peak freed weight pages
        assert resident[-1] > min(resident)       # and the drain brought some back
        assert max(r["used"] for r in log) > 2 * (T_BLK + R)  # the KV blocks took the freed bytes
        assert len(dropped) < 0.25 * len({ev[1] for evs in syn.gen_kv_requests(STEPS, st.seed) for ev in evs})
        assert pw.pw_memory(st.ctx).resident_bytes == st.resident_bytes_eq3()
        for l in range(st.L):                     # never above the packed bitwidths
            assert np.all(st.committed_q(l) <= st.layers[l]["q0"])
    finally:
        pw.pw_destroy(st.ctx)


def test_paging_run_full_size_spot_checks():
    shape = syn.SHAPES["qwen"]
    st = Stack(shape, L=2)
    try:
        S, B = budget(st, 0.3)
        log, _ = run_requests(st, offline_inputs(st), S, B, check_steps={0, 100, 199}, check_layers={0},
                              check_tokens=3)
        assert any(r["kind"] == 1 for r in log)
        pw.pw_sync_io(st.ctx)
        pw.pw_commit(st.ctx)
        assert pw.pw_memory(st.ctx).resident_bytes == st.resident_bytes_eq3()
    finally:
        pw.pw_destroy(st.ctx)


def test_planner_leaves_blocks_in_transit_out():
    """Blocks whose pages are in transfer take no planner step, and the other blocks keep
    their own offline sensitivities (the problem is re-indexed over the idle blocks)."""
    st = Stack(MINI, L=1)
    try:
        off = offline_inputs(st)
        for step in range(3):  # routing statistics for Eq. 1
            st.forward(0, st.tokens(step, 0))
        pw.pw_set_fault(st.ctx, 3, 1)  # transfers stay in flight while held
        E = MINI.E
        moved = [syn.block_id(0, e, 0, E) for e in (0, 5, 11, 17)]
        for b in moved:
            pw.pw_offload(st.ctx, b, 3)
        start = pw.pw_memory(st.ctx).resident_bytes
        obs = dict(T_blk=T_BLK, F_blk=0, B_KV=0.25 * start, R=R, mass=None, phi=syn.gen_phi_np(st.n_blocks, 0, 7))
        want = oracle_plan(st, off, obs)
        plan = pw.pw_plan_step(st.ctx, st.n_blocks, obs, off)
        assert (plan["kind"], plan["stage"], plan["D"]) == want[:3]
        assert plan["entries"] == want[3]
        assert plan["kind"] == 1 and plan["entries"]
        assert not set(moved) & {blk for blk, _, _, _ in plan["entries"]}
        # the same with a batch-level residual table in place of the Eq. 5 heads
        obs_t = dict(obs, phi=None, rho_hat=np.random.default_rng(2).normal(0, 1, (st.n_blocks, len(MINI.bits) - 1)))
        want = oracle_plan(st, off, obs_t)
        plan = pw.pw_plan_step(st.ctx, st.n_blocks, obs_t, off)
        assert (plan["kind"], plan["stage"], plan["D"]) == want[:3]
        assert plan["entries"] == want[3] and plan["entries"]
        pw.pw_set_fault(st.ctx, 3, 0)
        pw.pw_sync_io(st.ctx)
        pw.pw_commit(st.ctx)
    finally:
        pw.pw_destroy(st.ctx)
