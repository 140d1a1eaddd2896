"""Seeded synthetic inputs for the TTT inner-loop forward.

This module draws random numbers and rounds them to the I/O precision; it
holds none of the method's arithmetic.  In particular it does not evaluate the
per-token learning-rate gate: for the gated workloads it hands over the gate's
inputs (the layer input x, the per-head gate vectors theta and eta_base), and
the CUDA path (ttt_eta_gate) and the CPU oracle (oracle.eta_gate) each compute
eta from them.  Both the CUDA path's tests/benchmark and the CPU oracle are fed
from here.

Recipe (numpy PCG64, one independent sub-stream per tensor, seed 0 unless
overridden; values drawn in float32, then rounded to bfloat16 with
round-to-nearest-even when the I/O type is bf16):
  * Q, K, V ~ N(0, 1/d) i.i.d.
  * W0 ~ N(0, 0.02^2) of shape [H, d, d] (TTT-Linear init of the
    damodev.csdn.net TTT article, section 4.3), b0 ~ N(0, b0_std^2) ([H, d]).
  * TTT-MLP: W1 [H, d, dh], W2 [H, dh, d] ~ N(0, 0.02^2), b1 = b2 = 0.
  * residual LayerNorm: gamma ~ 1 + N(0, 0.02^2), beta ~ N(0, 0.02^2), [H, d].
  * eta: either a constant, or the inputs of the per-token gate
    eta = eta_base * sigmoid(theta_h . x_t) (lryc.cn TTT article, section 2.2)
    with eta_base = 1/d, x ~ N(0, 1)^768 per (batch, position) (rounded to bf16
    for bf16 I/O: it is the layer's input) and theta_h ~ N(0, 0.02^2)^768 per head.
  * drift (long-context case): K and V get +0.1 * j / sqrt(d) added to every
    coordinate in segment j = floor(t / 4096).
"""
from __future__ import annotations

import dataclasses

import numpy as np

_STREAMS = ("Q", "K", "V", "W0", "b0", "x", "theta", "gamma", "beta", "W1", "b1", "W2",
            "b2")
D_MODEL = 768   # width of the layer input x that the learning-rate gate reads


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    kind: str            # "linear" | "mlp"
    B: int
    H: int
    L: int
    d: int = 64
    mini_batch: int = 16
    io: str = "bf16"     # "f32" | "bf16"
    ln: bool = False     # residual LayerNorm f(k) = k + LN(f_res(k))
    eta: str = "gate"    # "gate" | "const"
    eta_const: float = 0.1
    b0_std: float = 0.0
    dh: int = 256        # MLP hidden width (4d)
    drift: bool = False
    eps: float = 1e-6

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)

    @property
    def head_tokens(self) -> int:
        return self.B * self.H * self.L

    @property
    def tokens(self) -> int:
        return self.B * self.L


# The five workloads (TTT-Linear/TTT-MLP forward, d = 64, mini-batch 16).
CONFIGS = {
    "linear_f32_B1_H2_L256": Config("linear_f32_B1_H2_L256", "linear", B=1, H=2, L=256,
                                    io="f32", eta="const", eta_const=0.1, b0_std=0.0),
    "linear_bf16_B8_H12_L2048": Config("linear_bf16_B8_H12_L2048", "linear", B=8, H=12,
                                       L=2048, b0_std=0.01),
    "linear_ln_bf16_B4_H16_L8192": Config("linear_ln_bf16_B4_H16_L8192", "linear", B=4, H=16,
                                          L=8192, ln=True),
    "mlp_ln_bf16_B4_H12_L4096": Config("mlp_ln_bf16_B4_H12_L4096", "mlp", B=4, H=12, L=4096,
                                       ln=True),
    "linear_ln_drift_bf16_B1_H32_L32768": Config("linear_ln_drift_bf16_B1_H32_L32768",
                                                 "linear", B=1, H=32, L=32768, ln=True,
                                                 drift=True),
}
CONFIG_ORDER = list(CONFIGS)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); the result
    is float32 holding exactly representable bf16 values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are exact bf16 values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def uniform_eta(B: int, H: int, L: int, lo: float, hi: float, seed: int) -> np.ndarray:
    """A learning rate drawn uniformly from [lo, hi) per (batch, head, token), float32
    [B, H, L]: for cases that set eta directly instead of through the gate."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x37A])))
    return rng.uniform(lo, hi, (B, H, L)).astype(np.float32)


def make_inputs(cfg: Config, seed: int = 0) -> dict:
    """All inputs of one workload as float32 numpy arrays (bf16-exact for bf16
    I/O).  Keys: Q, K, V; eta (constant-rate workloads) or x [B, L, 768], theta
    [H, 768] and eta_base (gated workloads); W0, b0 (linear) or W1, b1, W2, b2
    (MLP); gamma, beta (None without LayerNorm)."""
    ss = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    rng = {name: np.random.Generator(np.random.PCG64(s)) for name, s in zip(_STREAMS, ss)}
    B, H, L, d = cfg.B, cfg.H, cfg.L, cfg.d
    sd = np.float32(1.0 / np.sqrt(d))

    def normal(name, shape, std, dtype=np.float32):
        return (rng[name].standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(dtype)

    Q = normal("Q", (B, H, L, d), sd)
    K = normal("K", (B, H, L, d), sd)
    V = normal("V", (B, H, L, d), sd)
    if cfg.drift:
        seg = (np.arange(L) // 4096).astype(np.float32) * np.float32(0.1) * sd
        K += seg[None, None, :, None]
        V += seg[None, None, :, None]
    if cfg.io == "bf16":
        Q, K, V = round_bf16(Q), round_bf16(K), round_bf16(V)

    out = {"Q": Q, "K": K, "V": V}
    if cfg.eta == "const":
        out["eta"] = np.full((B, H, L), cfg.eta_const, dtype=np.float32)
    else:
        x = rng["x"].standard_normal((B, L, D_MODEL), dtype=np.float32)
        out["x"] = round_bf16(x) if cfg.io == "bf16" else x
        out["theta"] = normal("theta", (H, D_MODEL), 0.02)
        out["eta_base"] = 1.0 / d
    if cfg.kind == "linear":
        out["W0"] = normal("W0", (H, d, d), 0.02)
        out["b0"] = (normal("b0", (H, d), cfg.b0_std) if cfg.b0_std > 0
                     else np.zeros((H, d), np.float32))
    else:
        out["W1"] = normal("W1", (H, d, cfg.dh), 0.02)
        out["b1"] = np.zeros((H, cfg.dh), np.float32)
        out["W2"] = normal("W2", (H, cfg.dh, d), 0.02)
        out["b2"] = np.zeros((H, d), np.float32)
    if cfg.ln:
        out["gamma"] = (1.0 + normal("gamma", (H, d), 0.02)).astype(np.float32)
        out["beta"] = normal("beta", (H, d), 0.02)
    else:
        out["gamma"] = None
        out["beta"] = None
    return out
