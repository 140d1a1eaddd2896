"""The multi-process path of bench.py on CPU (gloo, world size 2): one process per
GPU is how the bench runs replicas, and every (batch, head) scan is independent, so
the path shards over (batch, head) with no collective in the data path."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world), CUDA_VISIBLE_DEVICES="")


def _max_worker(rank, world, port, q):
    _env(rank, world, port)
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    q.put((r, w, bench.max_over_ranks(w, 1.5 + r)))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 2.5), (1, 2, 2.5)]


SHARD_CFG = dict(B=3, H=3, L=64)   # 9 (batch, head) rows: rank 1's range starts mid-batch


def _row_outputs(cfg, x, r0, r1):
    """Oracle outputs of rows r0..r1-1 of the B*H grid (row b*H + h), one row at a time."""
    import oracle
    pairs = [divmod(r, cfg.H) for r in range(r0, r1)]
    res = oracle.run_pairs(cfg.kind, x, pairs, threads=1, mini_batch=cfg.mini_batch, ln=cfg.ln,
                           eps=cfg.eps)
    return [[np.asarray(a)[0, 0] for a in res[pr]] for pr in pairs]


def _shard_worker(rank, world, port, q):
    _env(rank, world, port)
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    import test_sequence_layers_08_b300 as ttt
    from test_sequence_layers_08_b300.inputs import CONFIGS, make_inputs
    dist.init_process_group("gloo")
    cfg = CONFIGS["linear_ln_bf16_B4_H16_L8192"].with_(name="shard", **SHARD_CFG)
    x = make_inputs(cfg, 0)
    if "eta" not in x:
        x["eta"] = oracle.eta_gate(x["x"], x["theta"], x["eta_base"])
    r0, r1 = ttt.partition_rows(cfg.B * cfg.H, world, rank)   # the library's partition
    mine = (r0, r1, _row_outputs(cfg, x, r0, r1))
    shards = [None] * world
    dist.all_gather_object(shards, mine)   # gathering is the test's check, not the data path
    q.put((rank, shards))
    dist.destroy_process_group()


def test_row_partition_reassembles_the_single_process_result():
    """Each rank takes its row range from the library's partition_rows and computes those
    rows; the ranges tile the grid in rank order and the rows reassemble the result of one
    process over every row."""
    sys.path.insert(0, ROOT)
    import oracle
    from test_sequence_layers_08_b300.inputs import CONFIGS, make_inputs
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg = CONFIGS["linear_ln_bf16_B4_H16_L8192"].with_(name="shard", **SHARD_CFG)
    x = make_inputs(cfg, 0)
    if "eta" not in x:
        x["eta"] = oracle.eta_gate(x["x"], x["theta"], x["eta_base"])
    full = _row_outputs(cfg, x, 0, cfg.B * cfg.H)
    shards = out[0]
    assert shards[0][0] == 0 and shards[-1][1] == cfg.B * cfg.H
    assert shards[0][1] == shards[1][0] and shards[1][0] % cfg.H != 0   # crosses a batch
    joined = [row for (_, _, rows) in shards for row in rows]
    assert len(joined) == len(full)
    for got, ref in zip(joined, full):
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a, b)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched by torchrun with two ranks: rank 0 alone
    runs the oracle and prints one JSON line; rank 1 exits 0 without work."""
    port = free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "linear_f32_B1_H2_L256", "--ref-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
