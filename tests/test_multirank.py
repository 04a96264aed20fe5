"""Multi-rank host logic on the CPU (world size 2, gloo): the benchmark's barrier, max and sum
over ranks and its reference arm on rank 0 only; and the one cross-shard step of the path, the
sink gradient's gather of per-shard chunk partials and their left-to-right merge."""

import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        mx = bench.max_over_ranks(dist, 1.5 + rank, "cpu")   # per-rank ms per step
        sm = bench.sum_over_ranks(dist, 100.0 * (rank + 1), "cpu")  # per-rank bytes
        out.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_max_and_sum_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]      # the slowest rank's time, on every rank
    assert [r[2] for r in res] == [300.0, 300.0]  # all ranks' bytes


def test_reference_arm_runs_on_rank_0_only():
    # a non-zero rank of a torchrun launch exits 0 without work and prints nothing
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_line_on_a_single_rank():
    import json

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["steps"] == 3 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["config"]["workload"] == "qwen_image_bf16"
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["sample"]
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def _sink_worker(rank, world, port, out):
    import numpy as np
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    from deterministic_attention_softmax_gb300.shard import sharded_sink_grad

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(17)  # the same global partials on both ranks
        full = (rng.standard_normal((3, 11)) * 10.0 ** rng.integers(-5, 5, (3, 11))).astype(np.float32)
        cols = [(0, 5), (5, 11)][rank]  # rank 0 holds chunks 0..4, rank 1 chunks 5..10
        mine = torch.from_numpy(np.ascontiguousarray(full[:, cols[0]:cols[1]]))
        d = sharded_sink_grad(mine)
        out.put((rank, d.numpy().tobytes(), full.tobytes()))
    finally:
        dist.destroy_process_group()


def test_sharded_sink_grad_gathers_in_rank_order_and_merges_left_to_right():
    import numpy as np

    import deterministic_attention_softmax_gb300 as fos

    fos.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sink_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = np.frombuffer(res[0][2], dtype=np.float32).reshape(3, 11)
    want = np.empty(3, dtype=np.float32)
    for h in range(3):  # one float32 rounding per addition, chunks in order, from +0
        t = np.float32(0.0)
        for c in range(11):
            t = np.float32(t + full[h, c])
        want[h] = t
    assert res[0][1] == want.tobytes() and res[1][1] == want.tobytes()
