"""Throughput of the TTT inner-loop forward on one B300 (or N, one replica per
GPU under torchrun), plus roofline fraction, clocks, an end-to-end number
through host buffers and the CPU oracle as a reported baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--decode T] [--gated] [--split]

A step is one call of the library entry point over one batch of the workload
(the whole hot path: every mini-batch of every (batch, head) scan).  Inputs are
synthetic (seeded, see test_sequence_layers_08_b300/inputs.py) and resident in
HBM; consecutive steps rotate through enough input/output copies that their
union exceeds the 126 MB L2, so no step starts with its inputs in L2.

Under torchrun (N > 1) every rank runs a replica of the workload by default
(weak scaling); --split gives each rank its contiguous range of (batch, head)
rows of one workload instead (partition_rows; strong scaling, no collective).
--gated puts the learning-rate gate (ttt_eta_gate, eta from the layer input)
in every step.

--decode T times the decode step instead (ttt_linear_step: T tokens per call, one
at a time, from a state carried in device memory between calls) on a linear
workload's batch, heads and head width.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from test_sequence_layers_08_b300.inputs import CONFIGS, make_inputs  # noqa: E402

DEFAULT_WORKLOAD = "linear_ln_bf16_B4_H16_L8192"
L2_BYTES = 126 * 2 ** 20
METRIC = "TTT-layer fwd tokens/s at 1 B300 and % of roofline (TC peak vs HBM GB/s)"


def flops_per_head_token(cfg) -> float:
    """Algorithmic FLOPs of one head-token (dense contractions only).
    Linear: key product, query product and update (3 d^2 MACs) plus Q K^T and
    the masked (Q K^T + 1) G product (2 b d MACs).  MLP: 7 d dh MACs (two key
    layers, G2 W2^T, two updates, two query layers) plus 2 b (d + dh)."""
    d, b = cfg.d, cfg.mini_batch
    if cfg.kind == "linear":
        return 2.0 * (3 * d * d + 2 * b * d)
    return 2.0 * (7 * d * cfg.dh + 2 * b * (d + cfg.dh))


def algorithmic_bytes(cfg) -> float:
    """Bytes one launch must move at minimum: Q, K, V read and Z written in the
    I/O type, eta read (fp32), initial state read once per head, final state
    written once per (batch, head) in fp32."""
    es = 2 if cfg.io == "bf16" else 4
    seq = cfg.B * cfg.H * cfg.L
    io = seq * (4 * cfg.d * es + 4)
    if cfg.kind == "linear":
        state = (cfg.d * cfg.d + cfg.d) * 4
    else:
        state = (2 * cfg.d * cfg.dh + cfg.dh + cfg.d) * 4
    ln = 2 * cfg.H * cfg.d * 4 if cfg.ln else 0
    return float(io + state * cfg.H + state * cfg.B * cfg.H + ln)


KERNEL_SOURCES = {"ttt_linear_fused": "ttt_linear_tc.cu", "ttt_linear_chunked": "ttt_linear_chunk.cu",
                  "ttt_mlp_fused": "ttt_mlp_tc.cu", "ttt_mlp_tmem": "ttt_mlp_tmem.cu",
                  "ttt_linear_decode": "ttt_decode.cu",
                  "ttt_linear_bwd": "ttt_backward.cu",
                  "ttt_linear_generic": "ttt_generic.cu", "ttt_mlp_generic": "ttt_generic.cu",
                  "ttt_linear_cols": "ttt_linear_cols.cu", "ttt_qkv_proj": "ttt_proj.cu"}


def measured_traffic(kname, workload):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu
    summary committed under profiles/ for this kernel and workload, if that capture was
    taken of the kernel source as it is now (its sha256 is recorded in the summary);
    otherwise None."""
    import hashlib
    import re
    src = KERNEL_SOURCES.get(kname)
    summary = os.path.join(ROOT, "profiles", f"{kname}_ncu_{workload}.md")
    if src is None or not os.path.exists(summary):
        return None
    text = open(summary).read()
    m_bytes = re.search(r"^traffic_bytes_per_launch:\s*(\d+)", text, re.M)
    m_sha = re.search(r"^kernel_source_sha256:\s*([0-9a-f]{64})", text, re.M)
    if not m_bytes or not m_sha:
        return None
    path = os.path.join(ROOT, "test_sequence_layers_08_b300", "csrc", src)
    if hashlib.sha256(open(path, "rb").read()).hexdigest() != m_sha.group(1):
        return None
    return float(m_bytes.group(1))


# FP32 FFMA peak of one B300: 148 SMs x 128 lanes x 2 FLOP per FMA x 2.032 GHz (TFLOP/s)
ALU_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        m = json.load(open(p))
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if t0 <= ts <= t1:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_inputs(x):
    """The workload's inputs for the oracle: eta given, or from the oracle's own gate."""
    import oracle
    if "eta" in x:
        return x
    y = dict(x)
    y["eta"] = oracle.eta_gate(x["x"], x["theta"], x["eta_base"])
    return y


def oracle_rate(cfg, x, budget_s: float, threads: int, variant=None):
    """Time the oracle as it stands on whole (batch, head) scans of the
    workload, in chunks of at least one scan per thread, until the time budget
    is spent (cycling over the workload's scans).  Returns (tokens/s, text).
    eta is computed (by the oracle's gate, for gated workloads) before timing."""
    import oracle
    x = oracle_inputs(x)
    pairs = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    kw = dict(mini_batch=cfg.mini_batch, ln=cfg.ln, eps=cfg.eps, **(variant or {}))
    chunk = max(threads, min(len(pairs), 2 * threads))
    done, i = 0, 0
    t0 = time.perf_counter()
    while True:
        todo = [pairs[(i + j) % len(pairs)] for j in range(chunk)]
        i += chunk
        oracle.run_pairs(cfg.kind, x, todo, threads=threads, **kw)
        done += chunk
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    desc = (f"{done} (batch, head) scans at full L={cfg.L} ({done / len(pairs):.2f} x the "
            f"{len(pairs)}-scan workload) in {dt:.1f} s on {threads} threads; "
            f"tokens/s = head-tokens/s / H")
    return done * cfg.L / cfg.H / dt, desc


def run_reference(args, cfg, world, rank):
    if rank != 0:
        return
    x = make_inputs(cfg, 0)
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    budget = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rate(cfg, x, budget / 4, threads)
    rates, sample = [], ""
    for _ in range(args.steps):
        r, sample = oracle_rate(cfg, x, budget, threads)
        rates.append(r)
    value = statistics.median(rates)
    sample = "per step: " + sample
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": cfg.tokens / value * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "B": cfg.B, "H": cfg.H, "L": cfg.L, "d": cfg.d,
                       "mini_batch": cfg.mini_batch, "io": cfg.io, "residual_ln": cfg.ln,
                       "kind": cfg.kind},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def packed(specs, device, pin=False):
    """One flat byte buffer holding tensors of the given (shape, dtype), each at a 256-byte
    aligned offset.  Returns (flat buffer, [tensor views])."""
    import torch
    offs, total = [], 0
    for shape, dt in specs:
        nbytes = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        offs.append((total, nbytes))
        total += (nbytes + 255) // 256 * 256
    flat = torch.empty(total, dtype=torch.uint8, device=device)
    if pin:
        flat = flat.pin_memory()
    views = [flat[o:o + n].view(dt).view(shape) for (o, n), (shape, dt) in zip(offs, specs)]
    return flat, views


def run_ours(args, cfg, world, rank, local):
    import torch
    import test_sequence_layers_08_b300 as ttt
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = make_inputs(cfg, 0)
    io = torch.bfloat16 if cfg.io == "bf16" else torch.float32
    state_keys = ["W0", "b0"] if cfg.kind == "linear" else ["W1", "b1", "W2", "b2"]

    gated = "eta" not in x
    if gated:   # the gate's inputs on the device; eta from the library's gate
        x_dev = torch.from_numpy(x["x"]).to(dev).to(io)
        theta_dev = torch.from_numpy(x["theta"]).to(dev)
        eta_dev = ttt.ttt_eta_gate(x_dev, theta_dev, x["eta_base"])
        ttt.ttt_sync_status()
    else:
        eta_dev = torch.from_numpy(x["eta"]).to(dev)

    def dev_inputs():
        d = {}
        for k in ("Q", "K", "V"):
            d[k] = rows(torch.from_numpy(x[k]).to(dev).to(io))
        for k in ["gamma", "beta"] + state_keys:
            d[k] = None if x[k] is None else torch.from_numpy(x[k]).to(dev)
        d["eta"] = rows(eta_dev.clone())
        return d

    # --split: this rank's contiguous range of (batch, head) rows (the library's partition);
    # otherwise every rank runs the whole workload (a replica)
    # the inner learner (default: squared-error loss, no weight decay)
    variant = dict(loss=args.loss, weight_decay=args.weight_decay)
    learner_tag = ("" if args.loss == "mse" else f"+loss_{args.loss}") + \
                  ("" if args.weight_decay == 0 else f"+wd{args.weight_decay:g}")
    split = args.split and world > 1
    r0, r1 = ttt.partition_rows(cfg.B * cfg.H, world, rank) if split else (0, cfg.B * cfg.H)
    part_kw = dict(heads=cfg.H, bh_offset=r0) if split else {}

    def rows(t):   # this rank's rows of a [B, H, ...] tensor
        return t.reshape((-1,) + tuple(t.shape[2:]))[r0:r1].contiguous() if split else t

    per_set = algorithmic_bytes(cfg) * (r1 - r0) / (cfg.B * cfg.H)
    n_sets = max(1, min(8, math.ceil(3 * L2_BYTES / per_set)))
    sets = [dev_inputs() for _ in range(n_sets)]
    outs = [None] * n_sets
    stream = torch.cuda.current_stream(dev)

    def step(i):
        s = sets[i % n_sets]
        if args.gated:   # the learning-rate gate is part of the step
            ttt.ttt_eta_gate(x_dev, theta_dev, x["eta_base"], out=s["eta"], stream=stream)
        kw = dict(mini_batch=cfg.mini_batch, residual_ln=cfg.ln, ln_eps=cfg.eps,
                  out=outs[i % n_sets], stream=stream, **part_kw, **variant)
        if cfg.kind == "linear":
            o = ttt.ttt_linear_fwd(s["Q"], s["K"], s["V"], s["eta"], s["W0"], s["b0"],
                                   s["gamma"], s["beta"], **kw)
        else:
            o = ttt.ttt_mlp_fwd(s["Q"], s["K"], s["V"], s["eta"], s["W1"], s["b1"], s["W2"],
                                s["b2"], s["gamma"], s["beta"], **kw)
        outs[i % n_sets] = o

    desc = ttt.make_desc(sets[0]["Q"], cfg.mini_batch, cfg.ln, cfg.eps,
                         d_hidden=cfg.dh if cfg.kind == "mlp" else 0, **part_kw, **variant)
    kname = ttt.kernel_name(desc, cfg.kind == "mlp")

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    ttt.ttt_sync_status(stream)
    # soak: keep the same load running for ~1.5 s so the clock samples taken
    # around the timed region describe this workload
    t_soak = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    step(0)
    e1.record(stream)
    e1.synchronize()
    one_ms = max(e0.elapsed_time(e1), 1e-3)
    soak_n = int(min(20000, max(0, args.soak_ms / one_ms)))
    for i in range(soak_n):
        step(i)
    torch.cuda.synchronize(dev)

    barrier(world)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    ttt.ttt_sync_status(stream)
    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(world, ms_total)
    ms_step = ms_total / args.steps
    # replicas: every rank runs the whole workload; split: the ranks share one workload
    value = (1 if split else world) * cfg.tokens / (ms_step * 1e-3)
    if time.time() - t_wall1 < 0.4:
        time.sleep(0.4)   # let the sampler log past the end of the timed region
    clk = clocks.summary(t_soak, time.time())

    # ---- end to end through host buffers (pinned), copies inside the timed region.  Every
    # step copies its inputs host -> device, runs the kernel and reads its outputs back.  The
    # per-step inputs (and the outputs) sit in one flat buffer each, so a step is one copy in,
    # one call, one copy out.  The two copy directions and the kernel run on three streams over
    # two device buffer sets, so the copies of neighbouring steps overlap the kernel (a
    # streaming job's steady state).
    # with --gated a step copies the layer input x (the gate computes eta on the device)
    in_keys = ["Q", "K", "V", "x" if args.gated else "eta"] + state_keys
    shapes = {k: (tuple(sets[0][k].shape), sets[0][k].dtype) for k in in_keys if k != "x"}
    if args.gated:
        shapes["x"] = (tuple(x_dev.shape), x_dev.dtype)
    in_specs = [shapes[k] for k in in_keys]
    out_specs = [(tuple(o.shape), o.dtype) for o in outs[0]]
    hin_flat, hin = packed(in_specs, "cpu", pin=True)
    for k, hv in zip(in_keys, hin):
        src = eta_dev.cpu() if k == "eta" else torch.from_numpy(x[k]).to(hv.dtype)
        hv.copy_(rows(src) if k in ("Q", "K", "V", "eta") else src)
    dsets, douts, din_flat, dout_flat, hout_flat = [], [], [], [], []
    for _ in range(2):
        f, views = packed(in_specs, dev)
        d = dict(zip(in_keys, views))
        d["gamma"], d["beta"] = sets[0]["gamma"], sets[0]["beta"]
        if args.gated:
            d["eta"] = torch.empty_like(eta_dev)
        dsets.append(d)
        din_flat.append(f)
        f, views = packed(out_specs, dev)
        douts.append(tuple(views))
        dout_flat.append(f)
        hout_flat.append(packed(out_specs, "cpu", pin=True)[0])
    h2d = hin_flat.numel()
    d2h = hout_flat[0].numel()
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run_on(b):
        s_ = dsets[b]
        if args.gated:
            ttt.ttt_eta_gate(s_["x"], theta_dev, x["eta_base"], out=s_["eta"], stream=stream)
        kw = dict(mini_batch=cfg.mini_batch, residual_ln=cfg.ln, ln_eps=cfg.eps,
                  out=douts[b], stream=stream, **part_kw, **variant)
        if cfg.kind == "linear":
            douts[b] = ttt.ttt_linear_fwd(s_["Q"], s_["K"], s_["V"], s_["eta"], s_["W0"], s_["b0"],
                                          s_["gamma"], s_["beta"], **kw)
        else:
            douts[b] = ttt.ttt_mlp_fwd(s_["Q"], s_["K"], s_["V"], s_["eta"], s_["W1"], s_["b1"],
                                       s_["W2"], s_["b2"], s_["gamma"], s_["beta"], **kw)

    def e2e_step(i):
        b = i % 2
        s_h2d.wait_event(ev_done[b])          # kernel i - 2 no longer reads set b
        with torch.cuda.stream(s_h2d):
            din_flat[b].copy_(hin_flat, non_blocking=True)
        ev_in[b].record(s_h2d)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])          # outputs b of step i - 2 have been read back
        run_on(b)
        ev_done[b].record(stream)
        s_d2h.wait_event(ev_done[b])
        with torch.cuda.stream(s_d2h):
            hout_flat[b].copy_(dout_flat[b], non_blocking=True)
        ev_out[b].record(s_d2h)

    for b in range(2):   # first recordings, so that every wait has an event to wait on
        run_on(b)
        for ev in (ev_in[b], ev_done[b], ev_out[b]):
            ev.record(stream)
    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    n_e2e = max(3, min(args.steps, 50))
    barrier(world)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    s_h2d.wait_event(s0)
    for i in range(n_e2e):
        e2e_step(i)
    stream.wait_event(ev_out[(n_e2e - 1) % 2])
    s1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(world, s0.elapsed_time(s1)) / n_e2e
    e2e_value = (1 if split else world) * cfg.tokens / (e2e_ms * 1e-3)

    clocks.stop()
    peaks = load_peaks()
    alg_bytes = per_set
    alg_flops = flops_per_head_token(cfg) * cfg.L * (r1 - r0)
    if args.gated:   # the gate reads x and writes eta (the scan's read of eta is counted)
        alg_bytes += x_dev.numel() * x_dev.element_size() + cfg.head_tokens * 4   # (replicas)
        alg_flops += 2.0 * x_dev.numel() * cfg.H
    achieved_gbs = alg_bytes / (ms_step * 1e-3) / 1e9
    achieved_tf = alg_flops / (ms_step * 1e-3) / 1e12
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    # the FP32 FFMA kernels' arithmetic peak is the ALU's (148 SMs x 128 lanes x 2 FLOP x
    # 2.032 GHz), the tensor-core kernels' the measured bf16 peak
    ffma = kname in ("ttt_linear_generic", "ttt_linear_cols", "ttt_mlp_generic")
    c_peak = ALU_PEAK_TFLOPS if ffma else peaks["bf16_tflops"]
    t_tc = alg_flops / (c_peak * 1e12)
    if t_tc > t_hbm:
        roof = {"bound": "alu" if ffma else "tensor", "achieved": achieved_tf, "peak": c_peak,
                "unit": "TFLOP/s", "frac": achieved_tf / c_peak}
    else:
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"]}
    roof.update({"traffic": measured_traffic(kname, cfg.name), "peak_source": peaks["source"], "kernel": kname,
                 "algorithmic_bytes": alg_bytes, "algorithmic_flops": alg_flops,
                 "roofline_ms": max(t_hbm, t_tc) * 1e3})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 1
        rate, sample = oracle_rate(cfg, x, args.cpu_seconds, threads, variant)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": sample}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "strong" if split else "weak",
                "vs_baseline": None,
                "dtype": "bf16" if cfg.io == "bf16" else "f32", "data": "synthetic",
                "config": {"workload": cfg.name + ("+gate" if args.gated else "") + learner_tag,
                           "kind": cfg.kind, "B": cfg.B, "H": cfg.H,
                           "eta": ("gate in the step (ttt_eta_gate)" if args.gated else
                                   "input (computed once by ttt_eta_gate)" if gated else "constant"),
                           "L": cfg.L, "d": cfg.d, "mini_batch": cfg.mini_batch,
                           "io": cfg.io, "state": "f32", "residual_ln": cfg.ln,
                           "learner": {"loss": args.loss, "weight_decay": args.weight_decay},
                           "l2": f"inputs rotate over {n_sets} copies "
                                 f"({n_sets * alg_bytes / 1e6:.0f} MB > L2)",
                           "parallelism": (f"(batch, head) rows split over {world} GPUs "
                                           f"(rank 0: rows {r0}..{r1 - 1}), one CTA per row"
                                           if split else
                                           f"replica x{world}, one CTA per (batch, head)")},
                "head_tokens_per_s": value * cfg.H, "roofline": roof, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h,
                        "schedule": "per step: one host->device copy of the inputs, the call, one "
                                    "device->host copy of the outputs; three streams over two "
                                    "buffer sets"},
                "gpu_launches": args.steps * (2 if args.gated else 1), "clocks": clk,
                "wall_s_timed": t_wall1 - t_wall0}
        print(json.dumps(line), flush=True)


def run_decode(args, cfg, world, rank, local):
    """Decode: `ttt_linear_step` on the workload's (B, H, d, I/O type, LayerNorm) with
    args.decode tokens per call, processed one at a time from a state carried in device memory
    between calls.  Consecutive calls rotate over enough (inputs, state) sets that their union
    exceeds L2; each set carries its own state from call to call.  A decode call is a few
    microseconds of GPU work, less than the Python binding's host cost, so the calls are
    captured in a CUDA graph (as a serving loop would run them) and the graph is replayed."""
    import torch
    import test_sequence_layers_08_b300 as ttt
    if cfg.kind != "linear":
        raise SystemExit("--decode runs the TTT-Linear decode step: pick a linear workload")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T = args.decode
    dcfg = cfg.with_(L=T, mini_batch=1)
    x = make_inputs(dcfg, 0)
    io = torch.bfloat16 if cfg.io == "bf16" else torch.float32
    es = 2 if cfg.io == "bf16" else 4
    BH, d = cfg.B * cfg.H, cfg.d
    state_bytes = BH * (d * d + d) * 4
    io_bytes = BH * T * (4 * d * es + 4)
    alg_bytes = 2 * state_bytes + io_bytes            # state read and written once per call
    alg_flops = 2 * 3 * d * d * BH * T                # k W, the rank-1 update, q W per token
    n_sets = max(2, min(128, math.ceil(3 * L2_BYTES / (state_bytes + io_bytes))))
    W0 = np.broadcast_to(x["W0"], (cfg.B, cfg.H, d, d))
    b0 = np.broadcast_to(x["b0"], (cfg.B, cfg.H, d))
    gamma = None if x["gamma"] is None else torch.from_numpy(x["gamma"]).to(dev)
    beta = None if x["beta"] is None else torch.from_numpy(x["beta"]).to(dev)
    qkv = {k: torch.from_numpy(x[k]).to(dev).to(io) for k in ("Q", "K", "V")}
    if "eta" in x:
        eta = torch.from_numpy(x["eta"]).to(dev)
    else:
        eta = ttt.ttt_eta_gate(torch.from_numpy(x["x"]).to(dev).to(io),
                               torch.from_numpy(x["theta"]).to(dev), x["eta_base"])
        ttt.ttt_sync_status()
    sets = []
    for _ in range(n_sets):
        sets.append(dict(Q=qkv["Q"].clone(), K=qkv["K"].clone(), V=qkv["V"].clone(),
                         eta=eta.clone(), W=torch.from_numpy(np.ascontiguousarray(W0)).to(dev),
                         b=torch.from_numpy(np.ascontiguousarray(b0)).to(dev),
                         Z=torch.empty_like(qkv["Q"])))
    stream = torch.cuda.current_stream(dev)

    def call(s_):   # on the current stream (the capture stream inside a graph capture)
        ttt.ttt_linear_step(s_["Q"], s_["K"], s_["V"], s_["eta"], s_["W"], s_["b"], gamma, beta,
                            residual_ln=cfg.ln, ln_eps=cfg.eps, out=s_["Z"])

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(max(args.warmup, n_sets)):
        call(sets[i % n_sets])
    ttt.ttt_sync_status(stream)
    per_graph = n_sets                      # one call on every set per replay
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(per_graph):
            call(sets[i])
    replays = max(1, math.ceil(args.steps / per_graph))
    t_soak = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    e1.synchronize()
    soak_n = int(min(20000, max(0, args.soak_ms / max(e0.elapsed_time(e1), 1e-3))))
    for _ in range(soak_n):
        graph.replay()
    barrier(world)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(replays):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ttt.ttt_sync_status(stream)
    n_calls = replays * per_graph
    ms_step = max_over_ranks(world, start.elapsed_time(end)) / n_calls
    value = world * cfg.B * T / (ms_step * 1e-3)
    time.sleep(0.4)
    clk = clocks.summary(t_soak, time.time())

    # end to end: every call copies its tokens in and its outputs out; the state stays on
    # the device (the decode cache)
    s0_ = sets[0]
    in_keys = ["Q", "K", "V", "eta"]
    hin_flat, hin = packed([(tuple(s0_[k].shape), s0_[k].dtype) for k in in_keys], "cpu", pin=True)
    for k, hv in zip(in_keys, hin):
        hv.copy_(s0_[k].cpu())
    din_flat, din = packed([(tuple(s0_[k].shape), s0_[k].dtype) for k in in_keys], dev)
    e2e_set = dict(zip(in_keys, din), W=s0_["W"], b=s0_["b"], Z=s0_["Z"])
    hz = torch.empty(s0_["Z"].shape, dtype=s0_["Z"].dtype).pin_memory()

    def e2e_call():
        din_flat.copy_(hin_flat, non_blocking=True)
        call(e2e_set)
        hz.copy_(e2e_set["Z"], non_blocking=True)

    for _ in range(args.warmup):
        e2e_call()
    torch.cuda.synchronize(dev)
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        for _ in range(per_graph):
            e2e_call()
    e2e_graph.replay()
    torch.cuda.synchronize(dev)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(replays):
        e2e_graph.replay()
    s1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(world, s0.elapsed_time(s1)) / n_calls
    e2e_value = world * cfg.B * T / (e2e_ms * 1e-3)
    clocks.stop()

    peaks = load_peaks()
    achieved = alg_bytes / (ms_step * 1e-3) / 1e9
    dkname = "ttt_linear_decode" if d == 64 else "ttt_linear_generic"
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"],
            "traffic": measured_traffic(dkname, f"decode_{cfg.name}_T{T}"),
            "peak_source": peaks["source"], "kernel": dkname,
            "algorithmic_bytes": alg_bytes, "algorithmic_flops": alg_flops,
            "roofline_ms": alg_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 1
        rate, sample = oracle_rate(dcfg, x, args.cpu_seconds, threads)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": sample.replace("scans at full", "decode calls of")}
    if rank == 0:
        line = {"metric": "TTT-Linear decode tokens/s (one token at a time from a carried "
                          "state) at 1 B300 and % of roofline",
                "value": value, "unit": "tokens/s", "n_gpus": world, "steps": n_calls,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if cfg.io == "bf16" else "f32", "data": "synthetic",
                "config": {"workload": f"decode_{cfg.name}_T{T}", "kind": "linear_decode",
                           "B": cfg.B, "H": cfg.H, "tokens_per_call": T, "d": d, "io": cfg.io,
                           "state": "f32", "residual_ln": cfg.ln,
                           "l2": f"calls rotate over {n_sets} (inputs, state) sets "
                                 f"({n_sets * (state_bytes + io_bytes) / 1e6:.0f} MB > L2)",
                           "parallelism": f"replica x{world}, one warp per (batch, head)"},
                "roofline": roof, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "tokens/s",
                        "h2d_bytes_per_step": hin_flat.numel(),
                        "d2h_bytes_per_step": hz.numel() * hz.element_size(),
                        "schedule": "per call: one host->device copy of the tokens, the call, "
                                    "one device->host copy of Z; the state stays on the device; "
                                    "CUDA graph of the calls"},
                "gpu_launches": n_calls, "clocks": clk,
                "launch": f"CUDA graph of {per_graph} calls, replayed {replays} times"}
        print(json.dumps(line), flush=True)


def run_backward(args, cfg, world, rank, local):
    """Backward: `ttt_linear_bwd` (the vector-Jacobian product of the TTT-Linear forward) on
    a linear workload (with its residual LayerNorm if it has one), with a seeded random dZ,
    dW_final, db_final.  Each
    step is one library call (the backward kernel and, for the head-shared initial state,
    the two per-head sums); consecutive steps rotate over input/output/workspace sets whose
    union exceeds L2.  FP32 FFMA arithmetic: the roofline is the FP32 ALU peak derived from
    the SM count and the maximum clock (148 SMs x 128 lanes x 2 FLOP x 2.032 GHz)."""
    import torch
    import test_sequence_layers_08_b300 as ttt
    if cfg.kind != "linear":
        raise SystemExit("--backward runs the TTT-Linear backward: pick a linear workload")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = make_inputs(cfg, 0)
    io = torch.bfloat16 if cfg.io == "bf16" else torch.float32
    es = 2 if cfg.io == "bf16" else 4
    if "eta" not in x:   # eta from the library's gate
        eta_dev = ttt.ttt_eta_gate(torch.from_numpy(x["x"]).to(dev).to(io),
                                   torch.from_numpy(x["theta"]).to(dev), x["eta_base"])
        ttt.ttt_sync_status()
    else:
        eta_dev = torch.from_numpy(x["eta"]).to(dev)
    rng = np.random.default_rng(1)
    B, H, L, d = cfg.B, cfg.H, cfg.L, cfg.d
    dZ_h = rng.standard_normal((B, H, L, d)).astype(np.float32)
    dWf_h = rng.standard_normal((B, H, d, d)).astype(np.float32)
    dbf_h = rng.standard_normal((B, H, d)).astype(np.float32)
    seq = B * H * L
    alg_bytes = float(seq * (7 * d * es + 8) + 2 * H * (d * d + d) * 4 + 2 * B * H * (d * d + d) * 4)
    alg_flops = float(2 * ((12 if cfg.ln else 11) * d * d + 4 * cfg.mini_batch * d) * seq)
    n_sets = max(1, min(4, math.ceil(3 * L2_BYTES / alg_bytes)))
    learner_tag = ("" if args.loss == "mse" else f"+loss_{args.loss}") + \
                  ("" if args.weight_decay == 0 else f"+wd{args.weight_decay:g}")

    def make_set():
        t = {k: torch.from_numpy(x[k]).to(dev).to(io) for k in ("Q", "K", "V")}
        t["dZ"] = torch.from_numpy(dZ_h).to(dev).to(io)
        t["eta"] = eta_dev.clone()
        t["W0"], t["b0"] = torch.from_numpy(x["W0"]).to(dev), torch.from_numpy(x["b0"]).to(dev)
        t["gamma"] = None if x["gamma"] is None else torch.from_numpy(x["gamma"]).to(dev)
        t["beta"] = None if x["beta"] is None else torch.from_numpy(x["beta"]).to(dev)
        t["dWf"], t["dbf"] = torch.from_numpy(dWf_h).to(dev), torch.from_numpy(dbf_h).to(dev)
        t["ws"] = torch.empty(ttt.ttt_linear_bwd_workspace_size(t["Q"], mini_batch=cfg.mini_batch,
                                                               residual_ln=cfg.ln, ln_eps=cfg.eps,
                                                               loss=args.loss,
                                                               weight_decay=args.weight_decay),
                              dtype=torch.uint8, device=dev)
        t["out"] = (torch.empty_like(t["Q"]), torch.empty_like(t["K"]), torch.empty_like(t["V"]),
                    torch.empty_like(t["eta"]), torch.empty_like(t["W0"]), torch.empty_like(t["b0"]))
        if cfg.ln:
            t["out"] += (torch.empty_like(t["gamma"]), torch.empty_like(t["beta"]))
        return t
    sets = [make_set() for _ in range(n_sets)]
    stream = torch.cuda.current_stream(dev)

    def call(t, strm):
        ttt.ttt_linear_bwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], t["b0"], t["dZ"], t["dWf"],
                           t["dbf"], t["gamma"], t["beta"], mini_batch=cfg.mini_batch,
                           residual_ln=cfg.ln, ln_eps=cfg.eps, loss=args.loss,
                           weight_decay=args.weight_decay, out=t["out"], workspace=t["ws"],
                           stream=strm)

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        call(sets[i % n_sets], stream)
    ttt.ttt_sync_status(stream)
    t_soak = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    call(sets[0], stream)
    e1.record(stream)
    e1.synchronize()
    soak_n = int(min(2000, max(0, args.soak_ms / max(e0.elapsed_time(e1), 1e-3))))
    for i in range(soak_n):
        call(sets[i % n_sets], stream)
    barrier(world)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        call(sets[i % n_sets], stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ttt.ttt_sync_status(stream)
    ms_step = max_over_ranks(world, start.elapsed_time(end)) / args.steps
    value = world * cfg.tokens / (ms_step * 1e-3)
    time.sleep(0.4)
    clk = clocks.summary(t_soak, time.time())

    # end to end: every step copies its inputs in from pinned host memory and its gradients out
    t0 = sets[0]
    in_keys = ["Q", "K", "V", "eta", "dZ", "dWf", "dbf"]
    hin_flat, hin = packed([(tuple(t0[k].shape), t0[k].dtype) for k in in_keys], "cpu", pin=True)
    for k, hv in zip(in_keys, hin):
        hv.copy_(t0[k].cpu())
    din_flat, din = packed([(tuple(t0[k].shape), t0[k].dtype) for k in in_keys], dev)
    e2e = dict(t0)
    e2e.update(zip(in_keys, din))
    out_specs = [(tuple(o.shape), o.dtype) for o in t0["out"]]
    dout_flat, dout = packed(out_specs, dev)
    hout_flat = packed(out_specs, "cpu", pin=True)[0]
    e2e["out"] = tuple(dout)
    n_e2e = max(3, min(args.steps, 20))
    for _ in range(2):
        din_flat.copy_(hin_flat, non_blocking=True)
        call(e2e, stream)
        hout_flat.copy_(dout_flat, non_blocking=True)
    torch.cuda.synchronize(dev)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(n_e2e):
        din_flat.copy_(hin_flat, non_blocking=True)
        call(e2e, stream)
        hout_flat.copy_(dout_flat, non_blocking=True)
    s1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(world, s0.elapsed_time(s1)) / n_e2e
    e2e_value = world * cfg.tokens / (e2e_ms * 1e-3)
    clocks.stop()

    peaks = load_peaks()
    alu_peak = ALU_PEAK_TFLOPS
    achieved = alg_flops / (ms_step * 1e-3) / 1e12
    roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
            "frac": achieved / alu_peak, "traffic": measured_traffic("ttt_linear_bwd", cfg.name),
            "peak_source": "derived: 148 SMs x 128 FP32 lanes x 2 FLOP x 2.032 GHz",
            "kernel": "ttt_linear_bwd", "algorithmic_bytes": alg_bytes, "algorithmic_flops": alg_flops,
            "hbm_frac": alg_bytes / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "roofline_ms": alg_flops / (alu_peak * 1e12) * 1e3}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle.backward import ttt_linear_grad
        threads = torch.get_num_threads()
        eta_h = eta_dev.cpu().numpy()
        t_start, done = time.perf_counter(), 0
        while True:   # whole (batch, head) scans at full L, one at a time
            bi, hi = divmod(done % (B * H), H)
            sl = lambda a: a[bi:bi + 1, hi:hi + 1]
            ttt_linear_grad(sl(x["Q"]), sl(x["K"]), sl(x["V"]), sl(eta_h), x["W0"][hi:hi + 1],
                            x["b0"][hi:hi + 1],
                            None if x["gamma"] is None else x["gamma"][hi:hi + 1],
                            None if x["beta"] is None else x["beta"][hi:hi + 1], sl(dZ_h), sl(dWf_h),
                            sl(dbf_h), mini_batch=cfg.mini_batch, ln=cfg.ln, eps=cfg.eps,
                            loss=args.loss, weight_decay=args.weight_decay)
            done += 1
            dt = time.perf_counter() - t_start
            if dt >= args.cpu_seconds:
                break
        cpu = {"value": done * L / H / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} (batch, head) backward scans at full L={L} in {dt:.1f} s "
                         f"(torch autograd, float64); tokens/s = head-tokens/s / H"}
    if rank == 0:
        line = {"metric": "TTT-Linear backward tokens/s at 1 B300 and % of roofline (FP32 ALU)",
                "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": {"workload": cfg.name + "+backward" + learner_tag, "kind": "linear_backward",
                           "learner": {"loss": args.loss, "weight_decay": args.weight_decay},
                           "B": B, "H": H, "L": L, "d": d, "mini_batch": cfg.mini_batch, "io": cfg.io,
                           "l2": f"inputs rotate over {n_sets} sets "
                                 f"({n_sets * alg_bytes / 1e6:.0f} MB of I/O, plus the checkpoint "
                                 f"workspaces)",
                           "parallelism": f"replica x{world}, one CTA per (batch, head)"},
                "roofline": roof, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "tokens/s",
                        "h2d_bytes_per_step": hin_flat.numel(), "d2h_bytes_per_step": hout_flat.numel(),
                        "schedule": "per step: one host->device copy of the inputs and dZ, the call, "
                                    "one device->host copy of the gradients, one stream"},
                "gpu_launches": args.steps * (5 if cfg.ln else 3), "clocks": clk}
        print(json.dumps(line), flush=True)


def run_project(args, cfg, world, rank, local):
    """The whole layer from its input tokens: each step is the input projections
    (ttt_qkv_proj: Q, K, V = views of x through the stacked projection matrices, tcgen05),
    the learning-rate gate (ttt_eta_gate) and the scan, on a gated workload (x [B, L, 768],
    seeded random projection matrices [3 H d, 768] ~ N(0, 1/768)).  Consecutive steps rotate
    over two input/output sets (each step writes 3 B H L d bf16 of Q, K, V: more than L2).
    Steps are pipelined: the scan of step i runs on a high-priority stream and holds one SM
    per (batch, head); the projections and gate of step i + 1 run beside it on a low-priority
    stream, their grids capped at the SMs the scan leaves idle (every step's work is in the
    timed region, the first step's projections included).  The projection call is also timed
    alone: its roofline is the bf16 tensor peak."""
    import torch
    import test_sequence_layers_08_b300 as ttt
    if cfg.eta != "gate" or cfg.io != "bf16":
        raise SystemExit("--project needs a bf16 workload with the per-token gate")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = make_inputs(cfg, 0)
    B, H, L, d = cfg.B, cfg.H, cfg.L, cfg.d
    Dx = x["x"].shape[-1]
    rng = np.random.default_rng(2)
    W_h = (rng.standard_normal((3 * H * d, Dx)) / np.sqrt(Dx)).astype(np.float32)
    theta = torch.from_numpy(x["theta"]).to(dev)
    W = torch.from_numpy(W_h).to(dev).to(torch.bfloat16)
    state = {k: (None if x.get(k) is None else torch.from_numpy(x[k]).to(dev))
             for k in ("W0", "b0", "W1", "b1", "W2", "b2", "gamma", "beta")}
    proj_flops = 2.0 * B * L * Dx * 3 * H * d
    learner_tag = ("" if args.loss == "mse" else f"+loss_{args.loss}") + \
                  ("" if args.weight_decay == 0 else f"+wd{args.weight_decay:g}")
    variant = dict(loss=args.loss, weight_decay=args.weight_decay)

    def make_set():
        t = {"x": torch.from_numpy(x["x"]).to(dev).to(torch.bfloat16)}
        t["qkv"] = tuple(torch.empty((B, H, L, d), device=dev, dtype=torch.bfloat16) for _ in range(3))
        t["eta"] = torch.empty((B, H, L), device=dev, dtype=torch.float32)
        return t
    sets = [make_set() for _ in range(2)]
    stream = torch.cuda.current_stream(dev)
    # the scan on a high-priority stream, the next step's projections and gate beside it
    s_scan = torch.cuda.Stream(dev, priority=-1)
    s_side = torch.cuda.Stream(dev, priority=0)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    scan_ctas = B * H   # one CTA per (batch, head)
    side_sms = n_sm - scan_ctas if scan_ctas <= n_sm - 16 else 0   # 0: no cap (all SMs)

    def prep(t, st, cap=0):
        ttt.ttt_qkv_proj(t["x"], W, H, d, out=t["qkv"], stream=st, max_sms=cap)
        ttt.ttt_eta_gate(t["x"], theta, x["eta_base"], out=t["eta"], stream=st, max_sms=cap)

    def scan(t, st, out=None):
        kw = dict(mini_batch=cfg.mini_batch, residual_ln=cfg.ln, ln_eps=cfg.eps, stream=st, **variant)
        Q, K, V = t["qkv"]
        if cfg.kind == "linear":
            return ttt.ttt_linear_fwd(Q, K, V, t["eta"], state["W0"], state["b0"], state["gamma"],
                                      state["beta"], out=out, **kw)
        return ttt.ttt_mlp_fwd(Q, K, V, t["eta"], state["W1"], state["b1"], state["W2"], state["b2"],
                               state["gamma"], state["beta"], out=out, **kw)

    def layer(t, out=None):   # one step, serial on the current stream
        prep(t, stream)
        return scan(t, stream, out)

    ev_prep = [torch.cuda.Event() for _ in range(2)]
    ev_scan = [torch.cuda.Event() for _ in range(2)]

    def pipeline(nsteps, first=None):
        """nsteps layer steps: scan i on s_scan, projections and gate of step i + 1 on s_side
        once scan i - 1 no longer reads their set.  Starts after `first` (an event on the
        current stream) and everything queued before; ends with the current stream waiting
        for both."""
        s_scan.wait_stream(stream)
        s_side.wait_stream(stream)
        if first is not None:
            s_scan.wait_event(first)
            s_side.wait_event(first)
        prep(sets[0], s_side, side_sms)
        ev_prep[0].record(s_side)
        for i in range(nsteps):
            b = i % 2
            s_scan.wait_event(ev_prep[b])
            scan(sets[b], s_scan, outs[b])
            ev_scan[b].record(s_scan)
            if i + 1 < nsteps:
                nb = (i + 1) % 2
                if i >= 1:
                    s_side.wait_event(ev_scan[nb])
                prep(sets[nb], s_side, side_sms)
                ev_prep[nb].record(s_side)
        stream.wait_stream(s_scan)
        stream.wait_stream(s_side)

    outs = [layer(t) for t in sets]
    ttt.ttt_sync_status(stream)
    clocks = ClockSampler(local)
    clocks.start()
    pipeline(max(2, args.warmup))
    ttt.ttt_sync_status(stream)
    t_soak = time.time()
    soak_end = time.time() + args.soak_ms / 1e3
    while time.time() < soak_end:
        pipeline(16)
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    pipeline(args.steps, first=start)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ttt.ttt_sync_status(stream)
    ms_step = max_over_ranks(world, start.elapsed_time(end)) / args.steps
    # the same steps one after another on one stream (no overlap), for comparison
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    q0.record(stream)
    for i in range(args.steps):
        layer(sets[i % 2], outs[i % 2])
    q1.record(stream)
    torch.cuda.synchronize(dev)
    ttt.ttt_sync_status(stream)
    ms_serial = max_over_ranks(world, q0.elapsed_time(q1)) / args.steps
    # the faster of the two schedules is the step (both run every step's whole work); the
    # overlap pays when the capped projections and gate take less than the scan
    ms_pipe = ms_step
    pipelined = ms_pipe <= ms_serial
    ms_step = min(ms_pipe, ms_serial)
    # the projection call alone (same rotation)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for i in range(args.steps):
        ttt.ttt_qkv_proj(sets[i % 2]["x"], W, H, d, out=sets[i % 2]["qkv"], stream=stream)
    p1.record(stream)
    torch.cuda.synchronize(dev)
    ttt.ttt_sync_status(stream)
    ms_proj = max_over_ranks(world, p0.elapsed_time(p1)) / args.steps
    value = world * cfg.tokens / (ms_step * 1e-3)
    time.sleep(0.4)
    clk = clocks.summary(t_soak, time.time())

    # end to end: every step copies x in from pinned host memory and Z out
    hx = torch.from_numpy(x["x"]).to(torch.bfloat16).pin_memory()
    hz = torch.empty(tuple(outs[0][0].shape), dtype=outs[0][0].dtype).pin_memory()
    n_e2e = max(3, min(args.steps, 20))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s0.record(stream)
    for i in range(n_e2e):
        sets[0]["x"].copy_(hx, non_blocking=True)
        layer(sets[0], outs[0])
        hz.copy_(outs[0][0], non_blocking=True)
    s1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(world, s0.elapsed_time(s1)) / n_e2e
    clocks.stop()

    peaks = load_peaks()
    achieved = proj_flops / (ms_proj * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "traffic": measured_traffic("ttt_qkv_proj", cfg.name + "_proj"),
            "peak_source": peaks["source"], "kernel": "ttt_qkv_proj", "algorithmic_flops": proj_flops,
            "ms_per_call": ms_proj, "roofline_ms": proj_flops / (peaks["bf16_tflops"] * 1e12) * 1e3}
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": cfg.name + "+proj+gate" + learner_tag, "kind": cfg.kind, "B": B, "H": H,
                           "L": L, "d": d, "d_model": Dx, "mini_batch": cfg.mini_batch, "io": "bf16",
                           "step": "ttt_qkv_proj + ttt_eta_gate + scan from the layer input x",
                           "schedule": ((f"pipelined: step i + 1's projections and gate beside the scan of step i, "
                                         f"capped at {side_sms or n_sm} SMs (serial: {ms_serial * 1e3:.1f} us per step)")
                                        if pipelined else
                                        (f"serial on one stream (pipelined with the projections and gate capped at "
                                         f"{side_sms or n_sm} SMs: {ms_pipe * 1e3:.1f} us per step)")),
                           "l2": "two input/output sets; each step writes 3 B H L d bf16 (> L2)",
                           "parallelism": f"replica x{world}"},
                "roofline": roof, "cpu_baseline": None,
                "e2e": {"value": world * cfg.tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                        "h2d_bytes_per_step": int(hx.numel() * hx.element_size()),
                        "d2h_bytes_per_step": int(hz.numel() * hz.element_size())},
                "gpu_launches": args.steps * 3, "clocks": clk}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: host time spread over warm-up and timed steps")
    ap.add_argument("--decode", type=int, default=0, metavar="T",
                    help="time the decode step instead: T tokens per call, one at a time, from a "
                         "state carried between calls (a linear workload's B, H, d)")
    ap.add_argument("--backward", action="store_true",
                    help="time the TTT-Linear backward pass (ttt_linear_bwd) instead (a linear "
                         "workload, with or without its residual LayerNorm)")
    ap.add_argument("--split", action="store_true",
                    help="with N > 1 GPUs, split one workload's (batch, head) rows over the ranks "
                         "(strong scaling) instead of running a replica on each")
    ap.add_argument("--loss", choices=["mse", "ip"], default="mse",
                    help="inner-learner loss: squared error (default) or inner product")
    ap.add_argument("--weight-decay", type=float, default=0.0,
                    help="inner-learner weight decay lambda on the fast weights")
    ap.add_argument("--gated", action="store_true",
                    help="each step also computes eta from the layer input with the learning-rate "
                         "gate (ttt_eta_gate) before the scan")
    ap.add_argument("--project", action="store_true",
                    help="time the whole layer from its input tokens: the input projections "
                         "(ttt_qkv_proj), the gate and the scan per step (a gated bf16 workload)")
    ap.add_argument("--mlp-kernel", choices=["fused", "tmem"], default=None,
                    help="TTT-MLP kernel: the warp-MMA one (default) or the tcgen05 one with the "
                         "fast weights in tensor memory (sets TTT_MLP_KERNEL)")
    ap.add_argument("--soak-ms", type=float, default=1500.0,
                    help="untimed load before the timed region, so the clock samples describe "
                         "this workload (0 under a profiler)")
    args = ap.parse_args()
    if args.mlp_kernel:
        os.environ["TTT_MLP_KERNEL"] = args.mlp_kernel
    if args.warmup < 3:
        args.warmup = 3
    cfg = CONFIGS[args.workload]
    if args.gated and cfg.eta != "gate":
        raise SystemExit("--gated needs a workload with the per-token gate")
    if args.gated and args.split:
        raise SystemExit("--gated and --split are not combined")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, cfg, world, rank)
        elif args.decode > 0:
            run_decode(args, cfg, world, rank, local)
        elif args.backward:
            run_backward(args, cfg, world, rank, local)
        elif args.project:
            run_project(args, cfg, world, rank, local)
        else:
            run_ours(args, cfg, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
