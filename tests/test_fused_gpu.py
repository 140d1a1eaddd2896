"""The tensor-core TTT-Linear kernels (bf16 I/O, d = 64, b = 16): the fused kernel (residual
LayerNorm, weight decay) and the chunked kernel (no LayerNorm) are the kernels the library
picks, they match the oracle on edge shapes, and their bounded waits report a timeout
instead of hanging."""
import numpy as np
import pytest
import torch

import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS, uniform_eta

from gpu_util import compare_all, inputs, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

LIN = CONFIGS["linear_bf16_B8_H12_L2048"]
LIN_LN = CONFIGS["linear_ln_bf16_B4_H16_L8192"]

# names of the tensor-core TTT-Linear kernels the library may pick for bf16, d = 64, b = 16
LINEAR_TC_KERNELS = ("ttt_linear_fused", "ttt_linear_chunked")


@pytest.mark.parametrize("name", ["linear_bf16_B8_H12_L2048", "linear_ln_bf16_B4_H16_L8192",
                                  "linear_ln_drift_bf16_B1_H32_L32768"])
def test_fused_kernel_is_selected(name):
    cfg = CONFIGS[name]
    q = torch.empty((cfg.B, cfg.H, cfg.L, cfg.d), dtype=torch.bfloat16, device="cuda")
    desc = ttt.make_desc(q, cfg.mini_batch, cfg.ln, cfg.eps)
    assert ttt.kernel_name(desc) in LINEAR_TC_KERNELS


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("L", [16, 32, 48, 64, 80, 144, 256, 400])
def test_fused_lengths(ln, L):
    """Lengths that end inside a 64-token pipeline stage, one to many stages."""
    cfg = (LIN_LN if ln else LIN).with_(name="len", B=2, H=3, L=L)
    x = inputs(cfg, seed=11 + L)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


@pytest.mark.parametrize("ln", [False, True])
def test_fused_more_ctas_than_sms(ln):
    """Several waves of CTAs (B*H > 148)."""
    cfg = (LIN_LN if ln else LIN).with_(name="waves", B=20, H=16, L=128)
    x = inputs(cfg, seed=13)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


@pytest.mark.parametrize("ln", [False, True])
def test_fused_large_state_values(ln):
    """Large eta: the state moves far from its start within a few mini-batches."""
    cfg = (LIN_LN if ln else LIN).with_(name="bigeta", B=1, H=4, L=512)
    x = inputs(cfg, seed=17)
    x["eta"] = uniform_eta(cfg.B, cfg.H, cfg.L, 0.0, 1.0, seed=17)   # eta up to ~1
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


@pytest.mark.parametrize("ln", [False, True])   # the chunked and the fused kernel
def test_bounded_wait_reports_timeout_and_context_survives(ln):
    cfg = (LIN_LN if ln else LIN).with_(name="timeout", B=1, H=2, L=256)
    x = inputs(cfg, seed=19)
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
    # the flag was cleared and the context still works
    ttt.ttt_sync_status()
    compare_all(cfg, run_gpu(cfg, dev), run_oracle(cfg, x))


@pytest.mark.parametrize("ln", [False, True])   # the chunked and the fused kernel
def test_per_call_status_word_takes_the_timeout(ln):
    """With a per-call status word in the descriptor, a bounded wait that runs out is reported
    in that word only: the device-wide flag (ttt_sync_status) stays clear, and a later call
    with its own word reports nothing."""
    import torch
    cfg = (LIN_LN if ln else LIN).with_(name="status_word", B=1, H=2, L=256)
    x = inputs(cfg, seed=23)
    dev = to_device(cfg, x)
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        ttt.set_wait_timeout_ns(5_000_000)     # 5 ms
        ttt.debug_withhold_loads(True)
        run_gpu(cfg, dev, status=word)         # syncs through ttt_sync_status: must not raise
    finally:
        ttt.debug_withhold_loads(False)
        ttt.set_wait_timeout_ns(0)
    assert int(word.item()) == 1
    word.zero_()
    compare_all(cfg, run_gpu(cfg, dev, status=word), run_oracle(cfg, x))
    assert int(word.item()) == 0
