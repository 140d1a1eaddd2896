"""The fused TTT-MLP kernel (bf16 I/O, d = 64, d_hidden = 256, b = 16): it is the
kernel the library picks, it matches the oracle on edge shapes, and its bounded
waits report a timeout instead of hanging."""
import numpy as np
import pytest
import torch

import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS, uniform_eta

from gpu_util import compare_all, inputs, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

MLP = CONFIGS["mlp_ln_bf16_B4_H12_L4096"]


def test_fused_mlp_is_selected():
    cfg = MLP
    q = torch.empty((cfg.B, cfg.H, cfg.L, cfg.d), dtype=torch.bfloat16, device="cuda")
    desc = ttt.make_desc(q, cfg.mini_batch, cfg.ln, cfg.eps, d_hidden=cfg.dh)
    assert ttt.kernel_name(desc, mlp=True) == "ttt_mlp_fused"


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("L", [16, 48, 64, 80, 272])
def test_fused_mlp_lengths(ln, L):
    """Lengths that end inside a 64-token pipeline stage, one to several ring turns."""
    cfg = MLP.with_(name="len", B=2, H=2, L=L, ln=ln)
    x = inputs(cfg, seed=23 + L)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_fused_mlp_more_ctas_than_sms():
    """Several waves of CTAs (B*H > 148)."""
    cfg = MLP.with_(name="waves", B=13, H=12, L=32)
    x = inputs(cfg, seed=29)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_fused_mlp_large_eta():
    """An eta large enough to move the state far from its start within a few mini-batches.
    (Per-(batch, head) initial state is covered by the state-carry test.)"""
    cfg = MLP.with_(name="bigeta", B=2, H=2, L=128)
    x = inputs(cfg, seed=31)
    x["eta"] = uniform_eta(cfg.B, cfg.H, cfg.L, 0.0, 0.25, seed=31)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_fused_mlp_bounded_wait_reports_timeout():
    cfg = MLP.with_(name="timeout", B=1, H=2, L=128)
    x = inputs(cfg, seed=37)
    dev = to_device(cfg, x)
    try:
        ttt.set_wait_timeout_ns(5_000_000)     # 5 ms
        ttt.debug_withhold_loads(True)
        with pytest.raises(ttt.TTTError) as ei:
            run_gpu(cfg, dev)
        assert ei.value.status == 4            # TTT_ERR_TIMEOUT
    finally:
        ttt.debug_withhold_loads(False)
        ttt.set_wait_timeout_ns(0)
    ttt.ttt_sync_status()
    compare_all(cfg, run_gpu(cfg, dev), run_oracle(cfg, x))
