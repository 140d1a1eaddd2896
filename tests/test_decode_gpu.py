"""GPU parity of the decode step (`ttt_linear_step`): tokens one at a time from a state carried
in device memory, against the oracle's mini-batch-1 recurrence on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS
from gpu_util import TOL, compare_all, inputs, rel_l2, to_device, with_oracle_eta

pytestmark = pytest.mark.gpu


def problem(io, ln, B, H, L, d=64, seed=3):
    base = CONFIGS["linear_ln_bf16_B4_H16_L8192" if ln else "linear_bf16_B8_H12_L2048"]
    cfg = base.with_(B=B, H=H, L=L, d=d, io=io)
    x = inputs(cfg, seed)
    rng = np.random.default_rng(seed + 100)
    # a distinct starting state per (batch, head), as a cache carried from earlier tokens holds
    W = (x["W0"][None] + 0.01 * rng.standard_normal((B, H, d, d))).astype(np.float32)
    b = (np.broadcast_to(x["b0"], (B, H, d)) + 0.01 * rng.standard_normal((B, H, d))).astype(np.float32)
    return cfg, x, W, b


def to_dev(cfg, x, W, b):
    d = to_device(cfg, {k: v for k, v in x.items() if k not in ("W0", "b0")})
    d["W"] = torch.from_numpy(W.copy()).cuda()
    d["b"] = torch.from_numpy(b.copy()).cuda()
    return d


def step(cfg, d, sl=slice(None), out=None):
    Z = ttt.ttt_linear_step(d["Q"][:, :, sl].contiguous(), d["K"][:, :, sl].contiguous(),
                            d["V"][:, :, sl].contiguous(), d["eta"][:, :, sl].contiguous(),
                            d["W"], d["b"], d["gamma"], d["beta"], residual_ln=cfg.ln,
                            ln_eps=cfg.eps, out=out)
    ttt.ttt_sync_status()
    return Z


def oracle_ref(cfg, x, W, b):
    x = with_oracle_eta(x)
    return oracle.ttt_linear(x["Q"], x["K"], x["V"], x["eta"], W, b, x["gamma"], x["beta"],
                             mini_batch=1, ln=cfg.ln, eps=cfg.eps, init_per_batch=True)


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("L", [1, 17, 40])
def test_decode_matches_oracle(io, ln, L):
    # B H = 6: one full CTA of four heads and a partial one
    cfg, x, W, b = problem(io, ln, B=2, H=3, L=L)
    d = to_dev(cfg, x, W, b)
    Z = step(cfg, d)
    compare_all(cfg, [Z.float().cpu().numpy(), d["W"].cpu().numpy(), d["b"].cpu().numpy()],
                oracle_ref(cfg, x, W, b))


@pytest.mark.parametrize("ln", [False, True])
def test_one_token_per_call_equals_one_call(ln):
    """The state carried through T calls of one token each gives bit-identical outputs and
    state to one call with the T tokens."""
    cfg, x, W, b = problem("bf16", ln, B=2, H=5, L=12)
    d1 = to_dev(cfg, x, W, b)
    Z1 = step(cfg, d1)
    d2 = to_dev(cfg, x, W, b)
    parts = [step(cfg, d2, slice(t, t + 1)) for t in range(cfg.L)]
    Z2 = torch.cat(parts, dim=2)
    assert torch.equal(Z1, Z2)
    assert torch.equal(d1["W"], d2["W"]) and torch.equal(d1["b"], d2["b"])
    compare_all(cfg, [Z1.float().cpu().numpy(), d1["W"].cpu().numpy(), d1["b"].cpu().numpy()],
                oracle_ref(cfg, x, W, b))


def test_decode_other_width_uses_the_generic_kernel():
    cfg, x, W, b = problem("f32", True, B=1, H=2, L=9, d=32)
    d = to_dev(cfg, x, W, b)
    Z = step(cfg, d)
    compare_all(cfg, [Z.cpu().numpy(), d["W"].cpu().numpy(), d["b"].cpu().numpy()],
                oracle_ref(cfg, x, W, b))


def test_decode_many_heads_full_width():
    """A decode batch at the bench's head count (B = 8, H = 12): every (batch, head) checked
    against the oracle on a short token run."""
    cfg, x, W, b = problem("bf16", False, B=8, H=12, L=8)
    d = to_dev(cfg, x, W, b)
    Z = step(cfg, d)
    compare_all(cfg, [Z.float().cpu().numpy(), d["W"].cpu().numpy(), d["b"].cpu().numpy()],
                oracle_ref(cfg, x, W, b))


@pytest.mark.parametrize("spread", [0.0, 0.5])
@pytest.mark.parametrize("ln", [False, True])
def test_decode_large_bias_offset(ln, spread):
    """A state whose bias carries a large common offset (about 4 on every feature, exactly or
    with a per-feature spread): the LayerNorm statistics of k W + c must not lose the token's
    spread to cancellation."""
    cfg, x, W, b = problem("bf16", ln, B=2, H=3, L=24, seed=41)
    rng = np.random.default_rng(42)
    b = (b + 4.0 + spread * rng.standard_normal(b.shape)).astype(np.float32)
    d = to_dev(cfg, x, W, b)
    Z = step(cfg, d)
    compare_all(cfg, [Z.float().cpu().numpy(), d["W"].cpu().numpy(), d["b"].cpu().numpy()],
                oracle_ref(cfg, x, W, b))
