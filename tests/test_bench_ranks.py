"""bench.py's multi-rank host logic: the max-over-ranks reduction with two gloo ranks on CPU,
and the reference arm under a launcher (rank 0 alone runs and prints; the others exit 0)."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed (1 + r) ms per step and (5 - r) ms end to end
        got = bench.reduce_max_over_ranks(dist, [1.0 + rank, 5.0 - rank], "cpu")
        dist.barrier()
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_times_are_the_slowest_ranks_with_gloo():
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = dict(out.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert got == {0: [2.0, 5.0], 1: [2.0, 5.0]}


def test_single_process_reduction_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_over_ranks(None, [3, 4.5], "cpu") == [3.0, 4.5]


def _reference_arm(rank):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2")
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "qwen", "--tokens", "1",
                           "--layers", "1", "--steps", "1", "--warmup", "1", "--gpus", "2"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_other_ranks_exit_quietly():
    r = _reference_arm(1)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.gpu
def test_reference_arm_rank0_prints_one_line():
    """Rank 0 times the oracle on the host cores (the sample's weights are drawn with the
    GPU run's device generator, hence a GPU)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = _reference_arm(0)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
