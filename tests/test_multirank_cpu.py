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


def _shard_worker(rank, world, port, q):
    _env(rank, world, port)
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from test_sequence_layers_08_b300.inputs import CONFIGS, make_inputs
    dist.init_process_group("gloo")
    cfg = CONFIGS["linear_ln_bf16_B4_H16_L8192"].with_(name="shard", B=2, H=3, L=64)
    x = make_inputs(cfg, 0)
    if "eta" not in x:
        x["eta"] = oracle.eta_gate(x["x"], x["theta"], x["eta_base"])
    pairs = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    mine = pairs[rank::world]                      # (batch, head) shard of this rank
    res = oracle.run_pairs(cfg.kind, x, mine, threads=1, mini_batch=cfg.mini_batch, ln=cfg.ln,
                           eps=cfg.eps)
    shards = [None] * world
    mine_out = {pr: [np.asarray(a) for a in res[pr]] for pr in mine}
    dist.all_gather_object(shards, mine_out)   # gathering is the test's check, not the data path
    q.put((rank, shards))
    dist.destroy_process_group()


def test_head_shards_reassemble_the_single_process_result():
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
    cfg = CONFIGS["linear_ln_bf16_B4_H16_L8192"].with_(name="shard", B=2, H=3, L=64)
    x = make_inputs(cfg, 0)
    if "eta" not in x:
        x["eta"] = oracle.eta_gate(x["x"], x["theta"], x["eta_base"])
    pairs = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    full = oracle.run_pairs(cfg.kind, x, pairs, threads=1, mini_batch=cfg.mini_batch, ln=cfg.ln,
                            eps=cfg.eps)
    seen = set()
    for shard in out[0]:
        for pr, res in shard.items():
            seen.add(pr)
            for a, f in zip(res, full[pr]):
                np.testing.assert_array_equal(a, np.asarray(f))
    assert seen == set(pairs)
    assert all(len(sh) == len(pairs) // 2 for sh in out[0])   # disjoint halves


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
