"""The TTT-MLP tensor-core kernels for bf16 I/O, d = 64, d_hidden = 256, b = 16: the
warp-MMA kernel (the default) and the tcgen05 kernel with the fast weights in tensor memory
(TTT_MLP_KERNEL=tmem).  Each is the kernel the library picks when asked, matches the oracle
on edge shapes, and its bounded waits report a timeout instead of hanging."""
import numpy as np
import pytest
import torch

import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS, uniform_eta

from gpu_util import compare_all, compare_pairs, inputs, run_gpu, run_oracle, sample_pairs, to_device

pytestmark = pytest.mark.gpu

MLP = CONFIGS["mlp_ln_bf16_B4_H12_L4096"]
KERNELS = {"fused": "ttt_mlp_fused", "tmem": "ttt_mlp_tmem"}


@pytest.fixture(params=list(KERNELS))
def mlp_kernel(request, monkeypatch):
    monkeypatch.setenv("TTT_MLP_KERNEL", request.param)
    return request.param


def test_fused_mlp_is_selected(mlp_kernel):
    cfg = MLP
    q = torch.empty((cfg.B, cfg.H, cfg.L, cfg.d), dtype=torch.bfloat16, device="cuda")
    desc = ttt.make_desc(q, cfg.mini_batch, cfg.ln, cfg.eps, d_hidden=cfg.dh)
    assert ttt.kernel_name(desc, mlp=True) == KERNELS[mlp_kernel]


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("L", [16, 48, 64, 80, 272])
def test_fused_mlp_lengths(mlp_kernel, ln, L):
    """Lengths that end inside a 64-token pipeline stage, one to several ring turns."""
    cfg = MLP.with_(name="len", B=2, H=2, L=L, ln=ln)
    x = inputs(cfg, seed=23 + L)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_fused_mlp_more_ctas_than_sms(mlp_kernel):
    """Several waves of CTAs (B*H > 148)."""
    cfg = MLP.with_(name="waves", B=13, H=12, L=32)
    x = inputs(cfg, seed=29)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_fused_mlp_large_eta(mlp_kernel):
    """An eta large enough to move the state far from its start within a few mini-batches.
    (Per-(batch, head) initial state is covered by the state-carry test.)"""
    cfg = MLP.with_(name="bigeta", B=2, H=2, L=128)
    x = inputs(cfg, seed=31)
    x["eta"] = uniform_eta(cfg.B, cfg.H, cfg.L, 0.0, 0.25, seed=31)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_fused_mlp_bounded_wait_reports_timeout(mlp_kernel):
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


@pytest.mark.parametrize("ln", [False, True])
def test_tmem_mlp_inner_product_loss(monkeypatch, ln):
    """The tcgen05 kernel with the inner-product loss (zeroed LayerNorm-backward terms)."""
    monkeypatch.setenv("TTT_MLP_KERNEL", "tmem")
    cfg = MLP.with_(name="tmem_ip", B=2, H=2, L=96, ln=ln)
    x = inputs(cfg, seed=41)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x), loss="ip"), run_oracle(cfg, x, loss="ip"))


def test_tmem_mlp_offset_bias(monkeypatch):
    """The tcgen05 kernel with b2 around 4 (the LayerNorm pivot keeps the one-pass statistics
    free of cancellation)."""
    monkeypatch.setenv("TTT_MLP_KERNEL", "tmem")
    cfg = MLP.with_(name="tmem_offset", B=2, H=2, L=128)
    x = inputs(cfg, seed=43)
    rng = np.random.default_rng(43)
    x["b2"] = (x["b2"] + 4.0 + 0.1 * rng.standard_normal(x["b2"].shape)).astype(np.float32)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_tmem_mlp_full_size(monkeypatch):
    """The 4 x 12 x 4096 TTT-MLP workload on the tcgen05 kernel, sampled (batch, head)."""
    monkeypatch.setenv("TTT_MLP_KERNEL", "tmem")
    cfg = MLP
    x = inputs(cfg, seed=0)
    got = run_gpu(cfg, to_device(cfg, x))
    compare_pairs(cfg, got, run_oracle(cfg, x, sample_pairs(cfg, 2, seed=13)))
