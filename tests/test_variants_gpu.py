"""GPU parity of the inner-learner variants (ai-feeds Modular TTT page, design dimensions
"loss" and "weight decay"): the inner-product loss -<f(k), v> and weight decay lambda on the
fast weights, alone and together, for every kernel family, against the oracle.

The tensor-core bf16 kernels run them in place of the default learner (for TTT-Linear the
chunked kernel without the residual LayerNorm and the fused one with it, for TTT-MLP the fused
kernel); every fp32 case runs on the FFMA kernels; the decode step has its own."""
import numpy as np
import pytest
import torch

import oracle
import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS

from gpu_util import (compare_all, compare_pairs, inputs, run_gpu, run_oracle, sample_pairs,
                      to_device, with_oracle_eta)

pytestmark = pytest.mark.gpu

LIN = CONFIGS["linear_bf16_B8_H12_L2048"]
LIN_LN = CONFIGS["linear_ln_bf16_B4_H16_L8192"]
MLP = CONFIGS["mlp_ln_bf16_B4_H12_L4096"]

VARIANTS = [("ip", 0.0), ("mse", 0.5), ("ip", 0.5)]
VID = lambda v: f"{v[0]}-wd{v[1]}"


def kernel(cfg, mlp=False, loss="mse", weight_decay=0.0):
    dev = torch.empty((cfg.B, cfg.H, cfg.L, cfg.d),
                      dtype=torch.bfloat16 if cfg.io == "bf16" else torch.float32)
    desc = ttt.make_desc(dev, cfg.mini_batch, cfg.ln, cfg.eps, d_hidden=cfg.dh if mlp else 0,
                         loss=loss, weight_decay=weight_decay)
    return ttt.kernel_name(desc, mlp)


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_linear_variants(io, ln, variant):
    loss, wd = variant
    # bf16: chunked (no LN) or fused (LN), 65 mini-batches (a ragged last 64-token stage);
    # f32: the column-split (no LN) or generic (LN) kernel
    L = 1040 if io == "bf16" else 272
    cfg = (LIN_LN if ln else LIN).with_(name=f"lin_var_{io}", B=2, H=3, L=L, io=io)
    if io == "bf16":
        assert kernel(cfg) in ("ttt_linear_fused", "ttt_linear_chunked")
    x = inputs(cfg, seed=71)
    got = run_gpu(cfg, to_device(cfg, x), loss=loss, weight_decay=wd)
    compare_all(cfg, got, run_oracle(cfg, x, loss=loss, weight_decay=wd))


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_mlp_variants(io, ln, variant):
    loss, wd = variant
    cfg = MLP.with_(name=f"mlp_var_{io}", B=2, H=2, L=80, io=io, ln=ln)
    x = inputs(cfg, seed=73)
    got = run_gpu(cfg, to_device(cfg, x), loss=loss, weight_decay=wd)
    compare_all(cfg, got, run_oracle(cfg, x, loss=loss, weight_decay=wd))


def test_tiny_weight_decay_is_the_default_learner():
    """lambda = 1e-30 selects the weight-decay code of the fused kernel, where every factor
    1 - lambda S rounds to 1 in fp32: its outputs equal the default kernel's bit for bit."""
    cfg = LIN_LN.with_(name="lin_wd_tiny", B=2, H=3, L=512)
    dev = to_device(cfg, inputs(cfg, seed=75))
    base = run_gpu(cfg, dev)
    tiny = run_gpu(cfg, dev, weight_decay=1e-30)
    for a, b in zip(base, tiny):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
def test_full_size_linear_ln_variants(variant):
    """The 4 x 16 x 8192 residual-LN workload with a variant learner, sampled (batch, head)."""
    loss, wd = variant
    cfg = LIN_LN
    x = inputs(cfg, seed=0)
    got = run_gpu(cfg, to_device(cfg, x), loss=loss, weight_decay=wd)
    pairs = sample_pairs(cfg, 4, seed=7)
    compare_pairs(cfg, got, run_oracle(cfg, x, pairs, loss=loss, weight_decay=wd))


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_variants(io, ln, variant):
    loss, wd = variant
    cfg = (LIN_LN if ln else LIN).with_(name=f"dec_var_{io}", B=2, H=3, L=33, io=io)
    x = inputs(cfg, seed=77)
    rng = np.random.default_rng(78)
    W = (x["W0"][None] + 0.01 * rng.standard_normal((cfg.B, cfg.H, cfg.d, cfg.d))).astype(np.float32)
    b = (np.broadcast_to(x["b0"], (cfg.B, cfg.H, cfg.d))
         + 0.01 * rng.standard_normal((cfg.B, cfg.H, cfg.d))).astype(np.float32)
    d = to_device(cfg, {k: v for k, v in x.items() if k not in ("W0", "b0")})
    Wd, bd = torch.from_numpy(W.copy()).cuda(), torch.from_numpy(b.copy()).cuda()
    Z = ttt.ttt_linear_step(d["Q"], d["K"], d["V"], d["eta"], Wd, bd, d["gamma"], d["beta"],
                            residual_ln=ln, ln_eps=cfg.eps, loss=loss, weight_decay=wd)
    ttt.ttt_sync_status()
    xo = with_oracle_eta(x)
    ref = oracle.ttt_linear(xo["Q"], xo["K"], xo["V"], xo["eta"], W, b, xo["gamma"], xo["beta"],
                            mini_batch=1, ln=ln, eps=cfg.eps, init_per_batch=True, loss=loss,
                            weight_decay=wd)
    compare_all(cfg, [Z.float().cpu().numpy(), Wd.cpu().numpy(), bd.cpu().numpy()], ref)


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
def test_full_size_mlp_variants(variant):
    """The 4 x 12 x 4096 TTT-MLP workload with a variant learner (the fused MLP kernel),
    sampled (batch, head)."""
    loss, wd = variant
    cfg = MLP
    assert kernel(cfg, mlp=True, loss=loss, weight_decay=wd) == "ttt_mlp_fused"
    x = inputs(cfg, seed=0)
    got = run_gpu(cfg, to_device(cfg, x), loss=loss, weight_decay=wd)
    pairs = sample_pairs(cfg, 2, seed=11)
    compare_pairs(cfg, got, run_oracle(cfg, x, pairs, loss=loss, weight_decay=wd))
