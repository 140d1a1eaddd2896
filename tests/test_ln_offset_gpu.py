"""LayerNorm inputs with a large common offset.

With the residual LayerNorm the gradient and the output go through the mean and the
variance of every token's pre-normalisation row z = k W + c (TTT-MLP: the second
layer's output).  When z has a common offset much larger than its spread, a one-pass
variance (sum z^2 / d - mean^2) loses the spread to cancellation in fp32.  These cases
put that offset in the bias (b0, or b2 for TTT-MLP) and, separately, shift the keys and
values by a large constant, and compare every (batch, head) with the oracle."""
import numpy as np
import pytest

from test_sequence_layers_08_b300.inputs import CONFIGS, round_bf16

from gpu_util import compare_all, inputs, run_gpu, run_oracle, to_device, with_oracle_eta

pytestmark = pytest.mark.gpu

LIN_LN = CONFIGS["linear_ln_bf16_B4_H16_L8192"]
MLP = CONFIGS["mlp_ln_bf16_B4_H12_L4096"]


def offset_bias(x, key, offset, seed):
    rng = np.random.default_rng(seed)
    x[key] = (offset + 0.01 * rng.standard_normal(x[key].shape)).astype(np.float32)


def shift_keys_values(cfg, x, shift):
    for k in ("K", "V"):
        v = (x[k] + np.float32(shift)).astype(np.float32)
        x[k] = round_bf16(v) if cfg.io == "bf16" else v


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("offset", [4.0, -16.0])
def test_linear_bias_offset(io, offset):
    cfg = LIN_LN.with_(name="lin_b0_offset", B=2, H=3, L=1024, io=io)
    x = inputs(cfg, seed=51)
    offset_bias(x, "b0", offset, 52)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_linear_key_value_shift():
    cfg = LIN_LN.with_(name="lin_kv_shift", B=2, H=3, L=1024)
    x = inputs(cfg, seed=53)
    shift_keys_values(cfg, x, 2.0)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_linear_bias_offset_per_batch_state():
    """The offset carried in a per-(batch, head) initial state (init_per_batch)."""
    cfg = LIN_LN.with_(name="lin_b0_offset_pb", B=2, H=3, L=256)
    x = inputs(cfg, seed=54)
    rng = np.random.default_rng(55)
    x["W0"] = np.ascontiguousarray(np.broadcast_to(x["W0"], (cfg.B, cfg.H, cfg.d, cfg.d)))
    x["b0"] = (4.0 + 0.01 * rng.standard_normal((cfg.B, cfg.H, cfg.d))).astype(np.float32)
    got = run_gpu(cfg, to_device(cfg, x), init_per_batch=True)
    import oracle
    x = with_oracle_eta(x)
    ref = oracle.ttt_linear(x["Q"], x["K"], x["V"], x["eta"], x["W0"], x["b0"], x["gamma"],
                            x["beta"], mini_batch=cfg.mini_batch, ln=True, eps=cfg.eps,
                            init_per_batch=True)
    compare_all(cfg, got, ref)


@pytest.mark.parametrize("offset", [4.0, -16.0])
def test_mlp_bias_offset(offset):
    cfg = MLP.with_(name="mlp_b2_offset", B=2, H=2, L=256)
    x = inputs(cfg, seed=57)
    offset_bias(x, "b2", offset, 58)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))


def test_mlp_key_value_shift():
    cfg = MLP.with_(name="mlp_kv_shift", B=2, H=2, L=256)
    x = inputs(cfg, seed=59)
    shift_keys_values(cfg, x, 2.0)
    compare_all(cfg, run_gpu(cfg, to_device(cfg, x)), run_oracle(cfg, x))
