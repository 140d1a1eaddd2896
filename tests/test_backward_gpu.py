"""GPU parity of the TTT-Linear backward pass (ttt_linear_bwd) with the backward oracle:
every gradient of every (batch, head), with and without the residual LayerNorm (then also
dgamma, dbeta), for fp32 and bf16 I/O, both losses, head-shared and per-batch initial
states, several mini-batch sizes and head dims, a (batch, head) partition, and repeated
calls on one workspace."""
import numpy as np
import pytest
import torch

import test_sequence_layers_08_b300 as ttt
from oracle.backward import ttt_linear_grad
from test_sequence_layers_08_b300.inputs import round_bf16

from gpu_util import check_scan, current_case, rel_l2

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def problem(B, H, L, d, io, seed, init_per_batch=False, finals=True, ln=False):
    rng = np.random.default_rng(seed)
    f = (lambda a: round_bf16(a.astype(np.float32))) if io == "bf16" else (lambda a: a.astype(np.float32))
    x = dict(Q=f(rng.standard_normal((B, H, L, d)) / np.sqrt(d)),
             K=f(rng.standard_normal((B, H, L, d)) / np.sqrt(d)),
             V=f(rng.standard_normal((B, H, L, d)) / np.sqrt(d)),
             eta=rng.uniform(0.2, 1.0, (B, H, L)).astype(np.float32) / d * 8,
             dZ=f(rng.standard_normal((B, H, L, d))))
    shape0 = (B, H) if init_per_batch else (H,)
    x["W0"] = (0.05 * rng.standard_normal(shape0 + (d, d))).astype(np.float32)
    x["b0"] = (0.05 * rng.standard_normal(shape0 + (d,))).astype(np.float32)
    x["dW_final"] = rng.standard_normal((B, H, d, d)).astype(np.float32) if finals else None
    x["db_final"] = rng.standard_normal((B, H, d)).astype(np.float32) if finals else None
    x["gamma"] = (1.0 + 0.2 * rng.standard_normal((H, d))).astype(np.float32) if ln else None
    x["beta"] = (0.2 * rng.standard_normal((H, d))).astype(np.float32) if ln else None
    return x


def to_dev(x, io):
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    out = {}
    for k, v in x.items():
        if v is None:
            out[k] = None
        elif k in ("Q", "K", "V", "dZ"):
            out[k] = torch.from_numpy(v).cuda().to(dt)
        else:
            out[k] = torch.from_numpy(v).cuda()
    return out


def run(x, io, mb, loss="mse", init_per_batch=False, weight_decay=0.0, **kw):
    t = to_dev(x, io)
    ln = x.get("gamma") is not None
    res = ttt.ttt_linear_bwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], t["b0"], t["dZ"],
                             t["dW_final"], t["db_final"], t.get("gamma"), t.get("beta"),
                             mini_batch=mb, loss=loss, residual_ln=ln, init_per_batch=init_per_batch,
                             weight_decay=weight_decay, **kw)
    ttt.ttt_sync_status()
    return [r.float().cpu().numpy().astype(np.float64) for r in res]


def reference(x, mb, loss="mse", init_per_batch=False, weight_decay=0.0):
    ln = x.get("gamma") is not None
    g = ttt_linear_grad(x["Q"], x["K"], x["V"], x["eta"], x["W0"], x["b0"], x.get("gamma"),
                        x.get("beta"), x["dZ"], x["dW_final"], x["db_final"], mini_batch=mb, ln=ln,
                        eps=1e-6, loss=loss, weight_decay=weight_decay, init_per_batch=init_per_batch)
    names = ("dQ", "dK", "dV", "deta", "dW0", "db0") + (("dgamma", "dbeta") if ln else ())
    return [g[k] for k in names]


def compare(got, ref, io, init_per_batch=False, case=None):
    case = case or current_case("bwd")
    tol = TOL[io]
    names = ("dQ", "dK", "dV", "deta", "dW0", "db0", "dgamma", "dbeta")
    assert len(got) == len(ref)
    for name, g, r in zip(names, got, ref):
        if name in ("dgamma", "dbeta") or (name in ("dW0", "db0") and not init_per_batch):
            for hi in range(g.shape[0]):
                check_scan(case, name, g[hi], r[hi], tol)
            continue
        for bi in range(g.shape[0]):
            for hi in range(g.shape[1]):
                check_scan(case, name, g[bi, hi], r[bi, hi], tol, seq_axis=0 if name != "dW0" and name != "db0" else None)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("loss", ["mse", "ip"])
def test_backward_matches_oracle(io, loss):
    x = problem(B=2, H=3, L=96, d=64, io=io, seed=21)
    compare(run(x, io, 16, loss), reference(x, 16, loss), io)


@pytest.mark.parametrize("mb,d", [(4, 32), (8, 16), (16, 128), (32, 64)])
def test_backward_shapes(mb, d):
    x = problem(B=1, H=2, L=4 * mb + mb * 3, d=d, io="f32", seed=23 + mb + d)
    compare(run(x, "f32", mb), reference(x, mb), "f32")


def test_backward_per_batch_initial_state_and_no_final_gradients():
    x = problem(B=2, H=2, L=64, d=64, io="f32", seed=25, init_per_batch=True, finals=False)
    compare(run(x, "f32", 16, init_per_batch=True), reference(x, 16, init_per_batch=True), "f32",
            init_per_batch=True)


def test_backward_row_partition_sums_the_call_rows_per_head():
    """Rows 2..4 of a 2 x 3 grid: dW0/db0 hold, per head, the sum over the call's rows of that
    head (heads 2, 0, 1 here), the per-token gradients the rows' own."""
    B, H, L, d = 2, 3, 64, 64
    x = problem(B, H, L, d, "f32", seed=27)
    rows = slice(2, 5)
    flat = lambda a: None if a is None else a.reshape((B * H,) + a.shape[2:])[rows].copy()
    xr = dict(Q=flat(x["Q"]), K=flat(x["K"]), V=flat(x["V"]), eta=flat(x["eta"]), dZ=flat(x["dZ"]),
              W0=x["W0"], b0=x["b0"], dW_final=flat(x["dW_final"]), db_final=flat(x["db_final"]))
    got = run(xr, "f32", 16, heads=H, bh_offset=2)
    full = ttt_linear_grad(x["Q"], x["K"], x["V"], x["eta"], x["W0"], x["b0"], None, None, x["dZ"],
                           x["dW_final"], x["db_final"], mini_batch=16)
    for name, g in zip(("dQ", "dK", "dV", "deta"), got[:4]):
        ref = full[name].reshape((B * H,) + full[name].shape[2:])[rows]
        assert rel_l2(g, ref) <= TOL["f32"], name
    # per-head sums over the rows of the call, from the oracle's per-(batch, head) gradients
    per_row = []
    for r in range(B * H):
        b, h = divmod(r, H)
        sl = lambda a: a[b:b + 1, h:h + 1]
        g1 = ttt_linear_grad(sl(x["Q"]), sl(x["K"]), sl(x["V"]), sl(x["eta"]), x["W0"][h:h + 1],
                             x["b0"][h:h + 1], None, None, sl(x["dZ"]), sl(x["dW_final"]),
                             sl(x["db_final"]), mini_batch=16)
        per_row.append((g1["dW0"][0], g1["db0"][0]))
    for h in range(H):
        want_w = sum(per_row[r][0] for r in range(2, 5) if r % H == h)
        want_b = sum(per_row[r][1] for r in range(2, 5) if r % H == h)
        assert rel_l2(got[4][h], want_w) <= TOL["f32"]
        assert rel_l2(got[5][h], want_b) <= TOL["f32"]


def test_backward_two_calls_on_one_workspace_agree_bit_for_bit():
    x = problem(B=2, H=2, L=64, d=64, io="bf16", seed=29)
    t = to_dev(x, "bf16")
    need = ttt.ttt_linear_bwd_workspace_size(t["Q"], mini_batch=16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        r = ttt.ttt_linear_bwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], t["b0"], t["dZ"],
                               t["dW_final"], t["db_final"], mini_batch=16, workspace=ws)
        ttt.ttt_sync_status()
        outs.append([a.clone() for a in r])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("loss", ["mse", "ip"])
def test_backward_residual_ln_matches_oracle(io, loss):
    x = problem(B=2, H=3, L=96, d=64, io=io, seed=41, ln=True)
    compare(run(x, io, 16, loss), reference(x, 16, loss), io)


@pytest.mark.parametrize("mb,d", [(8, 32), (16, 128), (4, 64)])
def test_backward_residual_ln_shapes(mb, d):
    x = problem(B=1, H=2, L=4 * mb + mb * 3, d=d, io="f32", seed=43 + mb + d, ln=True)
    compare(run(x, "f32", mb), reference(x, mb), "f32")


def test_backward_residual_ln_per_batch_initial_state():
    x = problem(B=2, H=2, L=64, d=64, io="f32", seed=45, init_per_batch=True, ln=True)
    compare(run(x, "f32", 16, init_per_batch=True), reference(x, 16, init_per_batch=True), "f32",
            init_per_batch=True)


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("loss", ["mse", "ip"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_backward_weight_decay(io, loss, ln):
    """Weight decay (ai-feeds Modular TTT page): lambda = 0.5 on eta up to ~0.13 per token."""
    x = problem(B=2, H=2, L=80, d=64, io=io, seed=61 + ln, ln=ln)
    compare(run(x, io, 16, loss, weight_decay=0.5), reference(x, 16, loss, weight_decay=0.5), io)


def test_backward_weight_decay_small_shapes():
    x = problem(B=1, H=2, L=40, d=32, io="f32", seed=63, ln=True)
    compare(run(x, "f32", 8, weight_decay=0.3), reference(x, 8, weight_decay=0.3), "f32")


@pytest.mark.parametrize("B,H,L,ln", [(8, 12, 2048, False), (4, 16, 8192, True)],
                         ids=["B8_H12_L2048", "B4_H16_L8192_ln"])
def test_backward_full_size_sampled_rows(B, H, L, ln):
    """The backward at the full sizes the bench times (the 8 x 12 x 2048 workload without LN,
    the 4 x 16 x 8192 one with LN), one call over every row with a distinct initial state per
    (batch, head); three sampled rows' gradients against the oracle run on those rows alone,
    and with LN the dgamma, dbeta of one head against the oracle's sum over that head's rows."""
    from gpu_util import sample_pairs
    from test_sequence_layers_08_b300.inputs import CONFIGS
    x = problem(B, H, L, 64, "bf16", seed=47, init_per_batch=True, ln=ln)
    got = run(x, "bf16", 16, init_per_batch=True)
    cfg = CONFIGS["linear_bf16_B8_H12_L2048"].with_(B=B, H=H, L=L)
    names = ("dQ", "dK", "dV", "deta", "dW0", "db0")
    row = lambda a, b, h: None if a is None else a[b:b + 1, h:h + 1]

    def oracle_row(b, h):
        return ttt_linear_grad(row(x["Q"], b, h), row(x["K"], b, h), row(x["V"], b, h), row(x["eta"], b, h),
                               row(x["W0"], b, h), row(x["b0"], b, h),
                               None if not ln else x["gamma"][h:h + 1], None if not ln else x["beta"][h:h + 1],
                               row(x["dZ"], b, h), row(x["dW_final"], b, h), row(x["db_final"], b, h),
                               mini_batch=16, ln=ln, eps=1e-6, init_per_batch=True)
    case = current_case("bwd_full")
    for b, h in sample_pairs(cfg, 3, seed=9):
        ref = oracle_row(b, h)
        for name, g in zip(names, got[:6]):
            check_scan(case, name, g[b, h], ref[name][0, 0], TOL["bf16"],
                       seq_axis=0 if name not in ("dW0", "db0") else None)
    if ln:
        h = 5
        refs = [oracle_row(b, h) for b in range(B)]
        check_scan(case, "dgamma", got[6][h], sum(r["dgamma"][0] for r in refs), TOL["bf16"])
        check_scan(case, "dbeta", got[7][h], sum(r["dbeta"][0] for r in refs), TOL["bf16"])
