#!/usr/bin/env python3
"""Throughput of the fused mixed-precision Any-Precision MoE layer stack on GB300.

Workload (default): the Qwen1.5-MoE-A2.7B-shaped stack -- hidden 2048, 60 routed experts
of intermediate 1408, top-4, a dense bf16 shared FFN of intermediate 5632, 24 layers,
8 bit-planes per block with bitwidths 3..8 (experts in the top quarter of the Zipf(1.1)
router prior at 5..8 bits, the rest at 3..4) -- decoding a batch of T tokens.  A step is
one pass of the whole stack over one batch: in every layer the router, top-K, bucketing,
gate_up (SiLU*up), down and combine kernels, x <- x + layer(x).  Inputs are synthetic and
seeded; the step's weights (~6 GB) are far larger than L2.

Prints one JSON line.  ``--impl reference`` times the float64 CPU oracle instead, on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402

METRIC = "MoE-layer tokens/s (T*L / stack time); weight-read HBM GB/s vs GB300 peak at mixed per-block bits"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen", choices=["qwen", "mixtral", "g128"])
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--layers", type=int, default=0, help="0 = the configuration's layer count")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-also", action="store_true",
                    help="skip the largest single-GPU configurations timed after the main workload")
    ap.add_argument("--gemv-tokens", type=int, default=None,
                    help="routed work items of at most this many tokens run on the CUDA cores (default: the library's)")
    ap.add_argument("--paging", action="store_true",
                    help="dynamic paging run: a request schedule served by the KV-block allocator drives the planner, "
                         "offload and reload every step")
    return ap.parse_args()


PREFILL_MIN_T = 512  # batches of at least this many tokens run the prefill tiling (tensor-bound)

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum, one ncu capture of each launch) per
# algorithmic byte of that launch, for the expert kernels: (phase, prefill tiling) -> ratio.
# Taken on the two-layer Qwen-shaped decode run (T = 64) and the one-layer Mixtral-shaped
# prefill run (T = 4096) of the current kernels (profiles/ names the commands); to be measured
# again whenever the expert kernels change.
TRAFFIC_PER_ALGORITHMIC_BYTE = {(1, False): 1.025, (2, False): 1.027, (1, True): 1.321, (2, True): 2.469}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense fp16/bf16 tensor throughput in TFLOP/s (kind::f16 runs fp16 and bf16 at one
    rate): the sustained cuBLAS figure, as the expert kernels run inside a long step."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        return 1700.0, "fallback (sustained)"


def workload_config(shape, T, L):
    kind = "prefill" if T >= PREFILL_MIN_T else "decode"
    return {
        "workload": f"{shape.name}-shaped MoE stack {kind}: {L} layers, T={T} tokens",
        "model_shape": {"H": shape.H, "E": shape.E, "I": shape.I, "K": shape.K, "Is": shape.Is,
                        "bmax": shape.bmax, "bits": list(shape.bits), "q_rule": shape.q_rule},
        "T": T, "layers": L,
        "l2": "inputs larger than L2 (every step streams the whole stack's resident planes)",
    }


# ---------------------------------------------------------------- clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=5):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # the first sample is taken before the timed region starts: wait for it (so that the
        # sampler is running), and leave it out of the record
        t_end = time.time() + 3.0
        while time.time() < t_end and self.proc.poll() is None:
            with open(self.path) as f:
                if f.readline():
                    break
            time.sleep(0.01)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        if len(lines) > 1:
            lines = lines[1:]  # the sample from before the timed region
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- ranks
def reduce_max_over_ranks(dist, values, device):
    """The job's time is its slowest rank's: each value replaced by its maximum over the
    ranks (a no-op without a process group)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


# ---------------------------------------------------------------- workload set-up
def load_stack(pw, torch, shape, L, T, seed, device):
    from synthetic.gen_torch import gen_block_torch, gen_shared_torch
    d = pw.pw_desc(L=L, E=shape.E, H=shape.H, I=shape.I, K=shape.K, Is=shape.Is, bmax=shape.bmax,
                   bits_mask=shape.bits_mask(), renorm=0, device=device, max_tokens=T, flags=0)
    ctx = pw.pw_create(d)
    qs = []
    for l in range(L):
        Wr, bias, ranks = syn.gen_router_np(shape, seed, l)
        pw.pw_set_router(ctx, l, Wr, bias)
        q = syn.gen_q_assignment(shape, seed, l, ranks)
        qs.append(q)
        if shape.Is:
            wgu, wd = gen_shared_torch(shape, seed, l)
            torch.cuda.synchronize()
            pw.pw_set_shared(ctx, l, wgu, wd)
            del wgu, wd
        for e in range(shape.E):
            for u in (0, 1):
                idx, lut = gen_block_torch(shape, seed, l, e, u)
                torch.cuda.synchronize()
                pw.pw_pack(ctx, l, e, u, idx, lut, int(q[e, u]))
                del idx, lut
    return ctx, qs


def layer_bytes(shape, q, counts, T):
    """Algorithmic bytes of one layer: the active blocks' q planes + LUT_q, the shared FFN,
    the router and the activations in and out."""
    def read_bytes(N, K, b):  # b planes of N rows x ceil(K/128)*128 bits, plus LUT_b (2^b fp16 per row)
        return b * N * ((K + 127) // 128 * 128) // 8 + N * (1 << b) * 2
    gu = dn = 0
    for e in np.nonzero(counts)[0]:
        N, K = syn.block_shape(shape, 0)
        gu += read_bytes(N, K, int(q[e, 0]))
        N, K = syn.block_shape(shape, 1)
        dn += read_bytes(N, K, int(q[e, 1]))
    sh_gu = 2 * shape.Is * shape.H * 2
    sh_dn = shape.H * shape.Is * 2
    router = shape.E * shape.H * 4
    act = 2 * T * shape.H * 2
    return dict(gu=gu, dn=dn, sh_gu=sh_gu, sh_dn=sh_dn, router=router, act=act,
                total=gu + dn + sh_gu + sh_dn + router + act, weights=gu + dn + sh_gu + sh_dn)


# ---------------------------------------------------------------- oracle timing
def oracle_sample(shape, seed, T_sample, device_gen=True):
    """Layer 0 of the workload on the host: router, shared weights and the routed experts of
    the first T_sample tokens, drawn with the same generator keys as the GPU run."""
    from oracle import moe as omoe
    from synthetic.gen_torch import gen_block_torch, gen_shared_torch, split_luts
    Wr, bias, ranks = syn.gen_router_np(shape, seed, 0)
    q = syn.gen_q_assignment(shape, seed, 0, ranks)
    x = syn.gen_tokens_np(shape, seed, 0, T_sample)
    ids, _, _ = omoe.route(x, Wr, bias, shape.K)
    experts = {}
    for e in np.unique(ids):
        blk = []
        for u in (0, 1):
            idx, lut = gen_block_torch(shape, seed, 0, int(e), u)
            N, _ = syn.block_shape(shape, u)
            blk += [idx.cpu().numpy(), split_luts(lut.cpu().numpy(), N, shape.bits)]
        experts[int(e)] = tuple(blk)
    shared = None
    if shape.Is:
        wgu, wd = gen_shared_torch(shape, seed, 0)
        shared = (wgu.cpu().numpy().view(np.uint16), wd.cpu().numpy().view(np.uint16))
    return x, Wr, bias, experts, q, shared


def time_oracle(shape, sample, reps=1):
    from oracle import moe as omoe
    x, Wr, bias, experts, q, shared = sample
    t0 = time.perf_counter()
    for _ in range(reps):
        omoe.moe_layer(x, Wr, bias, experts, q, shape.K, shape.bmax, shared=shared)
    return (time.perf_counter() - t0) / reps


# ---------------------------------------------------------------- arms
def run_reference(args, shape, L, T):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    T_sample = min(T, 4)
    sample = oracle_sample(shape, args.seed, T_sample)
    for _ in range(args.warmup):
        time_oracle(shape, sample)
    t = sum(time_oracle(shape, sample) for _ in range(args.steps)) / args.steps
    value = T_sample * 1 / t
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, T, L),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"layer 0 of {L}, first {T_sample} of {T} tokens per step (float64 numpy oracle)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def serve_requests(pw, kv, events, dropped):
    """Apply one step of the request schedule to the KV-block allocator; a request whose
    arrival or growth does not fit is dropped (its blocks released, its later events
    skipped)."""
    for ev in events:
        kind, r = ev[0], ev[1]
        if r in dropped:
            continue
        if kind == "finish":
            pw.pw_kv_release(kv, r)
        elif kind == "announce":
            pw.pw_kv_announce(kv, r, ev[2])
        else:
            try:
                pw.pw_kv_grow(kv, r, ev[2])
            except pw.PwError as e:
                if e.status != pw.PW_ERR_OOM:
                    raise
                dropped.add(r)
                pw.pw_kv_release(kv, r)


def run_paging(args, pw, torch, ctx, shape, L, T, stream, x0, xw, clocks_cls):
    """PagedWeight Sec. 3.2-3.3 in the loop: per decode step a seeded request schedule
    (arrivals, growth announced a step ahead, completions) is served by the KV-block
    allocator attached to the context, which shares one device budget with the weight
    pages; the planner (Eqs. 3-8) reads the allocator's free KV blocks, its plan is applied
    with offload / reload on the side stream, landed transfers are committed (retired pages
    become KV headroom), then the stack runs.  Timed end to end on the host (the serving
    loop, the planner and the page I/O calls are part of the step) and on the device."""
    steps = 200
    schedule = syn.gen_kv_requests(steps, args.seed)
    n_blocks = L * shape.E * 2
    off = syn.gen_planner_offline_np(n_blocks, list(shape.bits), 4, args.seed)
    off["n_stages"] = 3
    T_blk, R = 16, 8
    start = pw.pw_memory(ctx).resident_bytes
    held0 = pw.pw_memory(ctx).held_bytes
    live, peak = {}, 0  # the schedule's demand peak in blocks
    for events in schedule:
        for ev in events:
            if ev[0] == "finish":
                live.pop(ev[1])
            elif ev[0] in ("arrive", "grow"):
                live[ev[1]] = live.get(ev[1], 0) + ev[2]
        peak = max(peak, sum(live.values()))
    B_KV = int(0.3 * held0 / peak)            # the peak asks for 30% of the weight bytes
    S = held0 + (T_blk + R) * B_KV            # and the budget starts with T_blk + R free blocks
    kv = pw.pw_kv_create(S, B_KV)
    pw.pw_kv_attach(kv, ctx)
    dropped = set()
    moved = {"offload": 0.0, "reload": 0.0}
    applied = 0
    kinds = {0: 0, 1: 0, 2: 0}
    resident, free_blk, used = [], [], []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clocks = clocks_cls(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    t0 = time.perf_counter()
    try:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for step in range(steps):
                serve_requests(pw, kv, schedule[step], dropped)
                st = pw.pw_kv_get_stats(kv)
                obs = dict(T_blk=T_blk, F_blk=int(st["free_blocks"]), B_KV=float(B_KV), R=R, mass=None,
                           phi=syn.gen_phi_np(n_blocks, args.seed, step))
                plan = pw.pw_plan_step(ctx, n_blocks, obs, off)
                kinds[plan["kind"]] += 1
                applied += len(plan["entries"])
                for block, fb, tb, delta in plan["entries"]:
                    if tb < fb:
                        pw.pw_offload(ctx, block, tb)
                        moved["offload"] += delta
                    else:
                        pw.pw_reload(ctx, block, tb)
                        moved["reload"] += delta
                pw.pw_commit(ctx)
                xw.copy_(x0)
                pw.pw_stack_forward(ctx, xw, T, stream)
                resident.append(pw.pw_memory(ctx).resident_bytes)
                free_blk.append(int(st["free_blocks"]))
                used.append(int(st["used_blocks"]))
            ev1.record(stream)
        stream.synchronize()
        wall = time.perf_counter() - t0
        clk = clocks.stop()
        dev_ms = ev0.elapsed_time(ev1)
        pw.pw_sync_io(ctx)
    finally:
        pw.pw_kv_destroy(kv)
    n_req = len({ev[1] for events in schedule for ev in events})
    return {
        "steps": steps,
        "kv": {"source": "pw_kv allocator attached to the context (F_blk read every step)",
               "schedule": f"gen_kv_requests(200, seed={args.seed}): {n_req} requests, demand peak {peak} blocks",
               "budget_bytes": S, "block_bytes": B_KV, "T_blk": T_blk, "R": R, "dropped_requests": len(dropped),
               "F_blk": {"min": min(free_blk), "max": max(free_blk)}, "used_blocks_max": max(used)},
        "host_ms_per_step": wall * 1e3 / steps, "device_ms_per_step": dev_ms / steps,
        "tokens_per_s": T * L * steps / wall, "plans": {"none": kinds[0], "offload": kinds[1], "reload": kinds[2]},
        "offloaded_bytes": moved["offload"], "reloaded_bytes": moved["reload"],
        "resident_bytes": {"start": start, "min": min(resident), "end": resident[-1]}, "clocks": clk,
        # the stack's kernels, plus one page-table commit kernel per applied bitwidth change
        "gpu_launches": 5 * L * steps + applied,
    }


def stack_roofline(pw, ctx, shape, qs, L, T, kern):
    """Algorithmic bytes of the stack's layers (from the routing statistics of the timed
    steps), the per-kernel shares from the profiled pass, and the roofline of the dominant
    kernel: HBM GB/s at decode sizes, tensor TFLOP/s for prefill-sized batches."""
    bytes_l = []
    for l in range(L):
        cnt, _ = pw.pw_routing_stats(ctx, l, shape.E)
        bytes_l.append(layer_bytes(shape, qs[l], cnt, T))
    tot = {k: sum(b[k] for b in bytes_l) for k in bytes_l[0]}
    peak, peak_kind = peaks()
    # dominant kernel: the one with the largest share of the step
    share = kern.sum(axis=0) / kern.sum()
    names = ["route_kernel + gather_kernel", "tc_ffn_kernel<1> (gate_up + SiLU*up)", "tc_ffn_kernel<2> (down)",
             "combine_kernel"]
    dom = int(np.argmax(share))
    dom_bytes = {1: tot["gu"] + tot["sh_gu"] + T * shape.H * 2 * L,
                 2: tot["dn"] + tot["sh_dn"],
                 0: tot["router"] + T * shape.H * 2 * L,
                 3: T * shape.H * 2 * L}[dom]
    dom_ms = kern[:, dom].sum()
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    ratio = TRAFFIC_PER_ALGORITHMIC_BYTE.get((dom, T >= PREFILL_MIN_T)) if dom in (1, 2) else None
    roofline = {"bound": "hbm", "kernel": names[dom], "achieved": achieved, "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": ratio * dom_bytes / L if ratio else None,
                "algorithmic_bytes_per_launch": dom_bytes / L, "avg_launch_ms": dom_ms / L,
                "kernel_share": {n: float(s) for n, s in zip(names, share)}}
    flops = None
    if T >= PREFILL_MIN_T and dom in (1, 2):
        # prefill: the expert kernels are tensor-bound; algorithmic FLOPs of the dominant one
        # = 2 x (routed pairs x its block's N x K + tokens x the shared block's N x K)
        pairs = T * shape.K
        fl = {1: 2.0 * (pairs * 2 * shape.I * shape.H + T * 2 * shape.Is * shape.H),
              2: 2.0 * (pairs * shape.H * shape.I + T * shape.H * shape.Is)}
        flops = fl
        tp, tp_kind = tensor_peak()
        t_ach = fl[dom] * L / (dom_ms * 1e-3) / 1e12
        roofline.update({"bound": "tensor", "achieved": t_ach, "peak": tp, "peak_kind": tp_kind,
                         "unit": "TFLOP/s", "frac": t_ach / tp, "algorithmic_flops_per_launch": fl[dom],
                         "hbm_achieved_gbs": achieved})
    return {"bytes_l": bytes_l, "tot": tot, "roofline": roofline, "flops": flops}


def time_stack(pw, torch, ctx, shape, qs, L, T, steps, warmup, seed, local):
    """One more workload on an already loaded stack: warm-up, K timed steps (CUDA events on
    the launching stream, clocks sampled during them), a profiled pass for the kernel
    shares, and the dominant kernel's roofline."""
    stream = torch.cuda.Stream()
    pw.pw_set_stream(ctx, stream)
    x0 = torch.from_numpy(syn.gen_tokens_np(shape, seed, 0, T).view(np.int16)).cuda()
    xw = torch.empty_like(x0)
    torch.cuda.synchronize()

    def step():
        xw.copy_(x0)
        pw.pw_stack_forward(ctx, xw, T, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            step()
    stream.synchronize()
    for l in range(L):
        pw.pw_routing_stats(ctx, l, shape.E, reset=True)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
    stream.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    clk = clocks.stop()
    pw.pw_set_profiling(ctx, 1)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    stream.synchronize()
    kern = np.array([pw.pw_profile_read(ctx, l) for l in range(L)], dtype=np.float64)
    pw.pw_set_profiling(ctx, 0)
    rf = stack_roofline(pw, ctx, shape, qs, L, T, kern)
    out = {"config": workload_config(shape, T, L), "value": T * L / (ms * 1e-3), "unit": "tokens/s",
           "steps": steps, "warmup": max(warmup, 3), "ms_per_step": ms,
           "gbs": rf["tot"]["total"] / (ms * 1e-3) / 1e9, "roofline": rf["roofline"], "clocks": clk,
           "gpu_launches": 5 * L * steps}
    if rf["flops"] is not None:
        out["tflops"] = (rf["flops"][1] + rf["flops"][2]) * L / (ms * 1e-3) / 1e12
    return out


def run_ours(args, shape, L, T):
    import torch
    import any_precision_bit_gb300 as pw
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from any_precision_bit_gb300 import _build
    _build.build()
    t_setup = time.time()
    ctx, qs = load_stack(pw, torch, shape, L, T, args.seed, local)
    t_setup = time.time() - t_setup
    stream = torch.cuda.Stream()
    pw.pw_set_stream(ctx, stream)
    if args.gemv_tokens is not None:
        pw.pw_set_gemv_tokens(ctx, args.gemv_tokens)
    x0 = torch.from_numpy(syn.gen_tokens_np(shape, args.seed, 0, T).view(np.int16)).cuda()
    xw = torch.empty_like(x0)
    torch.cuda.synchronize()

    def step():
        xw.copy_(x0)
        pw.pw_stack_forward(ctx, xw, T, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    if args.paging:
        static_ms = None
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(20):
                step()
            ev1.record(stream)
        stream.synchronize()
        static_ms = ev0.elapsed_time(ev1) / 20
        res = run_paging(args, pw, torch, ctx, shape, L, T, stream, x0, xw, Clocks)
        line = {"metric": METRIC, "value": res["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
                "steps": res["steps"], "warmup": max(args.warmup, 3), "ms_per_step": res["host_ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
                "config": dict(workload_config(shape, T, L), workload=f"{shape.name}-shaped MoE stack decode with "
                               f"dynamic paging driven by the KV-block allocator: {L} layers, T={T}, 200 steps"),
                "static_ms_per_step": static_ms, "paging": res, "clocks": res["clocks"],
                "gpu_launches": res["gpu_launches"]}
        pw.pw_destroy(ctx)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    for l in range(L):
        pw.pw_routing_stats(ctx, l, shape.E, reset=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / args.steps
    clk = clocks.stop()
    if dist:
        dist.barrier()
    ms = reduce_max_over_ranks(dist, [ms], "cuda")[0]
    # Kernel durations, per layer: a second timed pass with CUDA events recorded between the
    # kernels on the launching stream.  The events serialise the kernels (the step above lets
    # each kernel start while its predecessor drains, through programmatic dependent launch),
    # so the step time is taken without them.
    pw.pw_set_profiling(ctx, 1)
    with torch.cuda.stream(stream):
        for _ in range(max(3, min(args.steps, 10))):
            step()
    stream.synchronize()
    kern = np.array([pw.pw_profile_read(ctx, l) for l in range(L)], dtype=np.float64)  # [L][4] ms
    pw.pw_set_profiling(ctx, 0)
    rf = stack_roofline(pw, ctx, shape, qs, L, T, kern)
    bytes_l, tot, roofline, flops = rf["bytes_l"], rf["tot"], rf["roofline"], rf["flops"]
    value = world * T * L / (ms * 1e-3)
    peak, _ = peaks()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(shape, T, L),
        "stack_tokens_per_s": world * T / (ms * 1e-3),
        "gbs": tot["total"] / (ms * 1e-3) / 1e9, "weight_gbs": tot["weights"] / (ms * 1e-3) / 1e9,
        "routed_gbs": (tot["gu"] + tot["dn"]) / (ms * 1e-3) / 1e9,
        "hbm_frac": tot["total"] / (ms * 1e-3) / 1e9 / peak,
        "bytes_per_step": tot["total"], "roofline": roofline, "clocks": clk,
        # algorithmic bytes of each layer's two expert kernels (gate_up with the shared gate_up and
        # the input rows; down with the shared down), for comparison with per-launch DRAM counters
        "expert_kernel_bytes_per_layer": [[b["gu"] + b["sh_gu"] + T * shape.H * 2, b["dn"] + b["sh_dn"]]
                                          for b in bytes_l] if L <= 4 else None,
        "gpu_launches": 5 * L * args.steps, "setup_s": round(t_setup, 1),
    }
    if flops is not None:
        tot_fl = (flops[1] + flops[2]) * L
        line["tflops"] = tot_fl / (ms * 1e-3) / 1e12
        line["ffn_tflops"] = {"gate_up": flops[1] * L / (kern[:, 1].sum() * 1e-3) / 1e12,
                              "down": flops[2] * L / (kern[:, 2].sum() * 1e-3) / 1e12}
    # end to end through the C ABI with pinned host buffers
    if not args.no_e2e:
        xh = torch.from_numpy(syn.gen_tokens_np(shape, args.seed, 0, T).view(np.int16)).pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        pw.pw_stack_forward_host(ctx, xh, T, yh)
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pw.pw_stack_forward_host(ctx, xh, T, yh)
        te = (time.perf_counter() - t0) / args.steps
        if dist:
            dist.barrier()
        te = reduce_max_over_ranks(dist, [te], "cuda")[0]
        line["e2e"] = {"value": world * T * L / te, "unit": "tokens/s", "ms_per_step": te * 1e3,
                       "h2d_bytes_per_step": T * shape.H * 2, "d2h_bytes_per_step": T * shape.H * 2}
    if rank == 0 and not args.no_cpu_baseline:
        line["_cpu_pending"] = True
    pw.pw_destroy(ctx)
    # The largest single-GPU configurations, on one loaded stack: the Mixtral-shaped stack with
    # all 32 layers, decoding a 256-token batch and running a 4096-token prefill.
    if world == 1 and not args.no_also and args.config == "qwen":
        mix = syn.SHAPES["mixtral"]
        t0 = time.time()
        mctx, mqs = load_stack(pw, torch, mix, mix.L, mix.prefill_T, args.seed, local)
        setup = round(time.time() - t0, 1)
        also = [time_stack(pw, torch, mctx, mix, mqs, mix.L, 256, max(args.steps, 10), args.warmup, args.seed, local),
                time_stack(pw, torch, mctx, mix, mqs, mix.L, mix.prefill_T, 5, 3, args.seed, local)]
        for a in also:
            a["setup_s"] = setup
        line["also"] = also
        pw.pw_destroy(mctx)
    if line.pop("_cpu_pending", False):
        Ts = min(T, 64)
        sample = oracle_sample(shape, args.seed, Ts)
        t = time_oracle(shape, sample)
        line["cpu_baseline"] = {"value": Ts / t, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"layer 0 of {L}, the first {Ts} of {T} tokens, one pass of the float64 "
                                          f"numpy oracle ({t:.1f} s); BLAS may use every core, the rest runs on one"}
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    shape = syn.SHAPES[args.config]
    L = args.layers or shape.L
    T = args.tokens
    if args.impl == "reference":
        run_reference(args, shape, L, T)
    else:
        run_ours(args, shape, L, T)


if __name__ == "__main__":
    main()
