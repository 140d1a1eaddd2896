"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases compare every output element; the five full-size workloads are
run in the launch configuration the benchmark times and compared on sampled
(batch, head) scans that the oracle recomputes whole.  Tolerances are the
relative L2 errors fixed for the workloads: 1e-5 with fp32 I/O, 2e-2 with
bf16 I/O and fp32 state.
"""
import numpy as np
import pytest
import torch

import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS

from gpu_util import (TOL, compare_all, compare_pairs, inputs, rel_l2, run_gpu, run_oracle,
                      sample_pairs, to_device)

pytestmark = pytest.mark.gpu

LIN = CONFIGS["linear_bf16_B8_H12_L2048"]
LIN_LN = CONFIGS["linear_ln_bf16_B4_H16_L8192"]
MLP = CONFIGS["mlp_ln_bf16_B4_H12_L4096"]


def small_cases():
    cases = []
    for io in ("f32", "bf16"):
        for ln in (False, True):
            # several mini-batches, a grid that is no multiple of anything
            cases.append(LIN.with_(name=f"lin_{io}_ln{int(ln)}", B=3, H=5, L=96, io=io, ln=ln))
            cases.append(LIN.with_(name=f"lin1_{io}_ln{int(ln)}", B=1, H=1, L=16, io=io, ln=ln))
            cases.append(MLP.with_(name=f"mlp_{io}_ln{int(ln)}", B=2, H=3, L=48, io=io, ln=ln))
    return cases


@pytest.mark.parametrize("cfg", small_cases(), ids=lambda c: c.name)
def test_small_all_elements(cfg):
    x = inputs(cfg, seed=3)
    got = run_gpu(cfg, to_device(cfg, x))
    ref = run_oracle(cfg, x)
    compare_all(cfg, got, ref)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_full_size_workloads(name):
    cfg = CONFIGS[name]
    x = inputs(cfg, seed=0)
    got = run_gpu(cfg, to_device(cfg, x))
    pairs = sample_pairs(cfg, 6 if cfg.kind == "mlp" else 8)
    ref = run_oracle(cfg, x, pairs)
    compare_pairs(cfg, got, ref)


@pytest.mark.parametrize("mb,d", [(1, 64), (4, 64), (8, 32), (32, 64), (16, 128), (64, 16)])
def test_generic_shapes(mb, d):
    cfg = LIN_LN.with_(name="g", B=2, H=2, L=128, d=d, mini_batch=mb, io="f32")
    x = inputs(cfg, seed=5)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


@pytest.mark.parametrize("kind", ["linear", "mlp"])
def test_eta_zero_returns_initial_state(kind):
    cfg = (LIN_LN if kind == "linear" else MLP).with_(name="z", B=2, H=2, L=64)
    x = inputs(cfg, seed=6)
    x["eta"] = np.zeros((cfg.B, cfg.H, cfg.L), np.float32)
    got = run_gpu(cfg, to_device(cfg, x))
    ref = run_oracle(cfg, x)
    compare_all(cfg, got, ref)
    init = [x["W0"], x["b0"]] if kind == "linear" else [x["W1"], x["b1"], x["W2"], x["b2"]]
    for g, w in zip(got[1:], init):
        np.testing.assert_array_equal(g, np.broadcast_to(w, g.shape))


@pytest.mark.parametrize("kind", ["linear", "mlp"])
def test_state_carry_in_place(kind):
    """Two calls, the second started in place from the first's final state,
    equal one call over the whole sequence."""
    cfg = (LIN_LN if kind == "linear" else MLP).with_(name="carry", B=2, H=3, L=128)
    x = inputs(cfg, seed=7)
    dev = to_device(cfg, x)
    full = run_gpu(cfg, dev)
    half = cfg.with_(L=64)
    d1 = {k: (v[:, :, :64].contiguous() if k in ("Q", "K", "V", "eta") else v)
          for k, v in dev.items()}
    d2 = {k: (v[:, :, 64:].contiguous() if k in ("Q", "K", "V", "eta") else v)
          for k, v in dev.items()}
    first = run_gpu(half, d1)
    state = [torch.from_numpy(a.astype(np.float32)).cuda() for a in first[1:]]
    names = ["W0", "b0"] if kind == "linear" else ["W1", "b1", "W2", "b2"]
    for n, s in zip(names, state):
        d2[n] = s
    out = (torch.empty_like(d2["Q"]),) + tuple(state)   # final state written over the initial
    second = run_gpu(half, d2, out=out, init_per_batch=True)
    z = np.concatenate([first[0], second[0]], axis=2)
    compare_all(cfg, [z] + list(second[1:]), full)


def test_non_default_stream_and_reuse():
    cfg = LIN.with_(name="s", B=2, H=2, L=64)
    x = inputs(cfg, seed=8)
    dev = to_device(cfg, x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = run_gpu(cfg, dev, stream=s)
    b = run_gpu(cfg, dev)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)   # deterministic kernels


def test_ttt_sync_status_clean():
    ttt.ttt_sync_status()
