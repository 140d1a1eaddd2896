"""(batch, head) partition through the C ABI: calls on disjoint row ranges of the B*H grid
(row b*H + h), each given its rows and the whole head-indexed parameters, reproduce one call
on all rows bit for bit (the rows are independent scans and every kernel is deterministic),
and agree with the oracle.  Ranges cross batch boundaries, so row i of a call must use head
(bh_offset + i) mod H."""
import numpy as np
import pytest
import torch

import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import CONFIGS

from gpu_util import compare_all, inputs, run_oracle, to_device

pytestmark = pytest.mark.gpu

CASES = {
    "linear_ln_bf16": CONFIGS["linear_ln_bf16_B4_H16_L8192"].with_(B=3, H=5, L=128),
    "linear_bf16": CONFIGS["linear_bf16_B8_H12_L2048"].with_(B=3, H=5, L=96),
    "linear_f32": CONFIGS["linear_ln_bf16_B4_H16_L8192"].with_(B=3, H=5, L=64, io="f32"),
    "linear_f32_noln": CONFIGS["linear_f32_B1_H2_L256"].with_(B=3, H=5, L=64),   # column split
    "mlp_ln_bf16": CONFIGS["mlp_ln_bf16_B4_H12_L4096"].with_(B=3, H=5, L=64),
    # the tcgen05 TTT-MLP kernel (TTT_MLP_KERNEL=tmem)
    "mlp_ln_bf16_tmem": CONFIGS["mlp_ln_bf16_B4_H12_L4096"].with_(B=3, H=5, L=64),
}
RANGES = [(0, 4), (4, 11), (11, 15)]


def rows_of(t, r0, r1):
    """Rows r0..r1-1 of a [B, H, ...] tensor, as a contiguous [rows, ...] tensor."""
    return t.reshape((-1,) + tuple(t.shape[2:]))[r0:r1].contiguous()


def call(cfg, dev, r=None, init_per_batch=False):
    kw = dict(mini_batch=cfg.mini_batch, residual_ln=cfg.ln, ln_eps=cfg.eps,
              init_per_batch=init_per_batch)
    seq = {k: dev[k] for k in ("Q", "K", "V", "eta")}
    state = ["W0", "b0"] if cfg.kind == "linear" else ["W1", "b1", "W2", "b2"]
    st = {k: dev[k] for k in state}
    if r is not None:
        seq = {k: rows_of(v, *r) for k, v in seq.items()}
        if init_per_batch:
            st = {k: rows_of(v, *r) for k, v in st.items()}
        kw.update(heads=cfg.H, bh_offset=r[0])
    fn = ttt.ttt_linear_fwd if cfg.kind == "linear" else ttt.ttt_mlp_fwd
    out = fn(seq["Q"], seq["K"], seq["V"], seq["eta"], *[st[k] for k in state], dev["gamma"],
             dev["beta"], **kw)
    ttt.ttt_sync_status()
    return out


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("init_per_batch", [False, True])
def test_row_ranges_reproduce_one_call(name, init_per_batch, monkeypatch):
    cfg = CASES[name]
    if name.endswith("_tmem"):
        monkeypatch.setenv("TTT_MLP_KERNEL", "tmem")
    x = inputs(cfg, seed=61)
    dev = to_device(cfg, x)
    if init_per_batch:   # a distinct initial state per (batch, head)
        rng = np.random.default_rng(62)
        for k in (["W0", "b0"] if cfg.kind == "linear" else ["W1", "b1", "W2", "b2"]):
            per = np.broadcast_to(x[k], (cfg.B,) + x[k].shape).copy()
            per += (0.01 * rng.standard_normal(per.shape)).astype(np.float32)
            x[k] = per
            dev[k] = torch.from_numpy(per).cuda()
    full = call(cfg, dev, init_per_batch=init_per_batch)
    parts = [call(cfg, dev, r, init_per_batch) for r in RANGES]
    for i, f in enumerate(full):
        joined = torch.cat([p[i] for p in parts], dim=0)
        assert torch.equal(joined, f.reshape(joined.shape)), f"output {i} differs"
    if not init_per_batch:
        compare_all(cfg, [f.float().cpu().numpy() for f in full], run_oracle(cfg, x))


def test_decode_row_ranges():
    cfg = CASES["linear_ln_bf16"].with_(L=8, mini_batch=1)
    x = inputs(cfg, seed=63)
    dev = to_device(cfg, x)
    rng = np.random.default_rng(64)
    W = (np.broadcast_to(x["W0"], (cfg.B, cfg.H, 64, 64)) + 0.01 * rng.standard_normal((cfg.B, cfg.H, 64, 64))).astype(np.float32)
    b = (np.broadcast_to(x["b0"], (cfg.B, cfg.H, 64)) + 0.01 * rng.standard_normal((cfg.B, cfg.H, 64))).astype(np.float32)
    Wa, ba = torch.from_numpy(W.copy()).cuda(), torch.from_numpy(b.copy()).cuda()
    Za = ttt.ttt_linear_step(dev["Q"], dev["K"], dev["V"], dev["eta"], Wa, ba, dev["gamma"],
                             dev["beta"], residual_ln=True, ln_eps=cfg.eps)
    Wr = torch.from_numpy(W.copy()).cuda().reshape(-1, 64, 64)
    br = torch.from_numpy(b.copy()).cuda().reshape(-1, 64)
    Zs = []
    for r0, r1 in RANGES:
        Wv, bv = Wr[r0:r1].contiguous(), br[r0:r1].contiguous()
        Zs.append(ttt.ttt_linear_step(*(rows_of(dev[k], r0, r1) for k in ("Q", "K", "V", "eta")),
                                      Wv, bv, dev["gamma"], dev["beta"], residual_ln=True,
                                      ln_eps=cfg.eps, heads=cfg.H, bh_offset=r0))
        Wr[r0:r1], br[r0:r1] = Wv, bv
    ttt.ttt_sync_status()
    assert torch.equal(torch.cat(Zs, 0), Za.reshape(-1, cfg.L, 64))
    assert torch.equal(Wr, Wa.reshape(-1, 64, 64)) and torch.equal(br, ba.reshape(-1, 64))
