"""GPU parity of the column-split TTT-Linear kernel (ttt_linear_cols).  Without the residual
LayerNorm, column j of the state (W[:, j], c_j) evolves from column j of K W + c, V and G
alone (damodev TTT article, sections 4.1-4.2), so a (batch, head) scan is split over d / dc
CTAs of dc output columns.  Every output of every (batch, head) is compared with the oracle
for each column width (4, 8, 16: chosen by the number of rows), head dims 8-128, mini-batch
sizes 1-64, both I/O types, both losses and weight decay."""
import numpy as np
import pytest
import torch

import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS

from gpu_util import compare_all, inputs, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

F32_WL = CONFIGS["linear_f32_B1_H2_L256"]          # fp32, const eta 0.1, no LN
LIN = CONFIGS["linear_bf16_B8_H12_L2048"]      # gated eta, b0 != 0, no LN

VARIANTS = [("mse", 0.0), ("ip", 0.0), ("mse", 0.5), ("ip", 0.5)]


def kernel(cfg):
    dev = torch.empty((cfg.B, cfg.H, cfg.L, cfg.d),
                      dtype=torch.bfloat16 if cfg.io == "bf16" else torch.float32)
    return ttt.kernel_name(ttt.make_desc(dev, cfg.mini_batch, cfg.ln, cfg.eps), False)


def check(cfg, seed, **variant):
    assert kernel(cfg) == "ttt_linear_cols"
    x = inputs(cfg, seed=seed)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x), **variant), run_oracle(cfg, x, **variant))


def test_cols_full_fp32_workload():
    """The 1 x 2 x 256 fp32 workload itself (16 CTAs of 4 columns per head)."""
    check(F32_WL, seed=0)


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: f"{v[0]}-wd{v[1]}")
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_cols_variants(io, variant):
    loss, wd = variant
    # bf16 I/O with d = 32 (the tensor-core kernels take d = 64 only); gated eta, b0 != 0
    cfg = LIN.with_(name="cols_var", B=1, H=3, L=160, d=32, io=io)
    check(cfg, seed=81, loss=loss, weight_decay=wd)


@pytest.mark.parametrize("d,mb", [(8, 1), (16, 4), (32, 8), (128, 16), (64, 64), (128, 64), (64, 2)])
def test_cols_shapes(d, mb):
    cfg = F32_WL.with_(name=f"cols_d{d}_b{mb}", B=1, H=2, L=5 * mb if mb > 2 else 40, d=d, mini_batch=mb)
    check(cfg, seed=83 + d + mb)


@pytest.mark.parametrize("B,H", [(1, 1), (4, 8), (8, 6), (3, 7)])
def test_cols_widths(B, H):
    """1 row: 16 CTAs of 4 columns; 32 rows: 8 columns; 48 rows: 16 columns; 21 rows: 8."""
    cfg = LIN.with_(name=f"cols_B{B}_H{H}", B=B, H=H, L=96, io="f32")
    check(cfg, seed=87 + B * H)


def test_cols_single_mini_batch():
    cfg = F32_WL.with_(name="cols_one_step", L=16)
    check(cfg, seed=89)


def test_cols_per_batch_initial_state():
    cfg = LIN.with_(name="cols_per_batch", B=2, H=2, L=64, io="f32")
    x = inputs(cfg, seed=91)
    rng = np.random.default_rng(92)
    for k in ("W0", "b0"):
        per = np.broadcast_to(x[k], (cfg.B,) + x[k].shape).copy()
        x[k] = per + (0.02 * rng.standard_normal(per.shape)).astype(np.float32)
    got = run_gpu(cfg, to_device(cfg, x), init_per_batch=True)
    compare_all(cfg, got, run_oracle(cfg, x, init_per_batch=True))
