"""The per-token learning-rate gate on the GPU (ttt_eta_gate, through the C ABI) against
the oracle's gate: eta[b, h, t] = eta_base * sigmoid(theta[h] . x[b, t]) (lryc.cn TTT
article, section 2.2).  The contraction is carried in fp32 on both token types, so the
bound is the fp32 one (relative L2 1e-5) for bf16 tokens too."""
import numpy as np
import pytest
import torch

import oracle
import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS, make_inputs, round_bf16

from gpu_util import check_scan, current_case

pytestmark = pytest.mark.gpu
TOL = 1e-5


def problem(B, L, H, Dx, io, seed, scale=0.02):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, L, Dx)).astype(np.float32)
    if io == "bf16":
        x = round_bf16(x)
    theta = (scale * rng.standard_normal((H, Dx))).astype(np.float32)
    return x, theta


def run(x, theta, eta_base, io, max_sms=0):
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    eta = ttt.ttt_eta_gate(torch.from_numpy(x).cuda().to(dt), torch.from_numpy(theta).cuda(),
                           eta_base, max_sms=max_sms)
    ttt.ttt_sync_status()
    return eta.cpu().numpy()


def compare(got, ref):
    case = current_case("gate")
    for bi in range(got.shape[0]):
        for hi in range(got.shape[1]):
            check_scan(case, "eta", got[bi, hi], ref[bi, hi], TOL)


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("B,L,H,Dx", [(1, 1, 1, 768), (3, 31, 5, 768), (2, 33, 12, 768),
                                      (1, 100, 16, 768), (2, 40, 17, 64), (1, 70, 32, 768),
                                      (2, 17, 3, 16), (1, 9, 40, 128), (1, 5, 2, 24)])
def test_gate_shapes(io, B, L, H, Dx):
    """Token counts that end inside a 32-token tile and cross batch rows, head counts that
    leave a partial 8-head MMA tile, more than 32 heads and widths that are no multiple of
    16 (the FP32 kernel)."""
    x, theta = problem(B, L, H, Dx, io, seed=B * 1000 + L * 10 + H)
    compare(run(x, theta, 0.25, io), oracle.eta_gate(x, theta, 0.25))


def test_gate_large_logits_saturate():
    x, theta = problem(2, 50, 8, 768, "bf16", seed=3, scale=1.0)   # |logit| up to ~100
    got = run(x, theta, 1.0, "bf16")
    assert np.isfinite(got).all() and got.min() >= 0.0 and got.max() <= 1.0
    compare(got, oracle.eta_gate(x, theta, 1.0))


@pytest.mark.parametrize("name", ["linear_bf16_B8_H12_L2048", "linear_ln_bf16_B4_H16_L8192",
                                  "mlp_ln_bf16_B4_H12_L4096", "linear_ln_drift_bf16_B1_H32_L32768"])
def test_gate_full_size(name):
    """The gate of every gated workload at its full size, every element."""
    cfg = CONFIGS[name]
    x = make_inputs(cfg, 0)
    compare(run(x["x"], x["theta"], x["eta_base"], cfg.io),
            oracle.eta_gate(x["x"], x["theta"], x["eta_base"]))


def test_gate_reuses_output_and_stream():
    x, theta = problem(2, 64, 16, 768, "bf16", seed=9)
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    td = torch.from_numpy(theta).cuda()
    out = torch.full((2, 16, 64), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ttt.ttt_eta_gate(xd, td, 0.5, out=out, stream=s)
    ttt.ttt_sync_status(s)
    compare(out.cpu().numpy(), oracle.eta_gate(x, theta, 0.5))


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("max_sms", [1, 7])
def test_gate_sm_cap(io, max_sms):
    """A grid capped at a few SMs still covers every tile of tokens."""
    x, theta = problem(2, 700, 16, 768, io, seed=50 + max_sms)
    compare(run(x, theta, 0.3, io, max_sms=max_sms), oracle.eta_gate(x, theta, 0.3))
