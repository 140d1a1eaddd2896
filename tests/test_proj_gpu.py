"""GPU parity of the input projections (ttt_qkv_proj, the tcgen05 GEMM): Q, K, V [B, H, L, d]
from the layer's tokens x [B, L, d_model] and the stacked projection matrices W [3 H d,
d_model] (lryc.cn TTT article, section 2.2), against the oracle's float64 product of the same
bf16 values; every (batch, head) within the bf16 tolerance, at small, ragged and full size."""
import numpy as np
import pytest
import torch

import oracle
import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import round_bf16

from gpu_util import check_scan, current_case

pytestmark = pytest.mark.gpu

TOL = 1e-2   # bf16 outputs (one rounding of an fp32 sum)


def problem(B, L, Dx, H, d, seed):
    rng = np.random.default_rng(seed)
    x = round_bf16(rng.standard_normal((B, L, Dx)).astype(np.float32))
    W = round_bf16((rng.standard_normal((3 * H * d, Dx)) / np.sqrt(Dx)).astype(np.float32))
    return x, W


def run(x, W, H, d, max_sms=0):
    xt = torch.from_numpy(x).cuda().to(torch.bfloat16)
    Wt = torch.from_numpy(W).cuda().to(torch.bfloat16)
    out = ttt.ttt_qkv_proj(xt, Wt, H, d, max_sms=max_sms)
    ttt.ttt_sync_status()
    return [o.float().cpu().numpy().astype(np.float64) for o in out]


@pytest.mark.parametrize("B,L,Dx,H", [(2, 256, 128, 4), (1, 200, 64, 4), (3, 128, 768, 8), (2, 384, 256, 12),
                                      (1, 96, 192, 4), (3, 20, 64, 4), (2, 1000, 128, 4)],
                         ids=["small", "ragged_tokens", "d_model768", "twelve_heads", "one_tile_short_k",
                              "short_sequences", "sequences_cross_groups"])
def test_projection_matches_oracle(B, L, Dx, H):
    d = 64
    x, W = problem(B, L, Dx, H, d, seed=B * L + Dx + H)
    got = run(x, W, H, d)
    ref = oracle.qkv_proj(x, W, H, d)
    case = current_case("proj")
    for name, g, r in zip("QKV", got, ref):
        for b in range(B):
            for h in range(H):
                check_scan(case, name, g[b, h], r[b, h], TOL, seq_axis=0)


@pytest.mark.parametrize("max_sms", [1, 3, 20])
def test_projection_sm_cap(max_sms):
    """A capped grid (one cluster of two for max_sms 1 and 3, ten for 20) covers every tile:
    same parity."""
    B, L, Dx, H, d = 2, 640, 192, 4, 64
    x, W = problem(B, L, Dx, H, d, seed=30 + max_sms)
    got = run(x, W, H, d, max_sms=max_sms)
    ref = oracle.qkv_proj(x, W, H, d)
    case = current_case("proj_cap")
    for name, g, r in zip("QKV", got, ref):
        for b in range(B):
            for h in range(H):
                check_scan(case, name, g[b, h], r[b, h], TOL, seq_axis=0)


def test_projection_full_size_sampled_tokens():
    """4 x 8192 tokens of 768 features into 3 x 16 heads of 64 (the input of the L = 8192
    residual-LN workload): 64 sampled tokens of every (batch, head) against the oracle."""
    B, L, Dx, H, d = 4, 8192, 768, 16, 64
    x, W = problem(B, L, Dx, H, d, seed=12)
    got = run(x, W, H, d)
    rng = np.random.default_rng(13)
    ts = np.sort(rng.choice(L, 64, replace=False))
    ref = oracle.qkv_proj(x[:, ts], W, H, d)
    case = current_case("proj_full")
    for name, g, r in zip("QKV", got, ref):
        for b in range(B):
            for h in range(H):
                check_scan(case, name, g[b, h][ts], r[b, h], TOL)
