"""ttt_linear_bwd_static: the backward pass on the library's static device scratch (no
allocation).  It must give what ttt_linear_bwd gives with a caller workspace, call after
call, and refuse a call that needs more scratch than it holds.  (This file is collected
last, so the GPU test also runs after every other test of the session.)"""
import ctypes

import numpy as np
import pytest

import test_sequence_layers_08_b300 as ttt


def test_static_scratch_refuses_calls_beyond_its_size():
    lib = ttt.load()
    cap = lib.ttt_linear_bwd_static_scratch_bytes()
    assert cap == 64 << 20
    # 8 x 12 rows of 16384 tokens: ~0.4 GB of state checkpoints
    desc = ttt.Desc(B=8, H=12, L=16384, d=64, d_hidden=0, mini_batch=16, io_dtype=1, residual_ln=0,
                    ln_eps=1e-6, init_per_batch=0)
    assert lib.ttt_linear_bwd_workspace_size(ctypes.byref(desc)) > cap
    fake = [ctypes.c_void_p((1 << 20) + i * (1 << 30)) for i in range(20)]
    st = lib.ttt_linear_bwd_static(ctypes.byref(desc), *fake, None)
    assert st == 1
    assert "static scratch" in lib.ttt_last_error().decode()


@pytest.mark.gpu
def test_static_scratch_matches_caller_workspace_two_calls_in_a_row():
    import torch
    rng = np.random.default_rng(31)
    B, H, L, d = 2, 3, 96, 64
    dev = torch.device("cuda")
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(dev).to(torch.bfloat16)
    f32 = lambda a: torch.from_numpy(a.astype(np.float32)).to(dev)
    Q, K, V = (bf(rng.standard_normal((B, H, L, d)) / 8) for _ in range(3))
    dZ = bf(rng.standard_normal((B, H, L, d)))
    eta = f32(rng.uniform(0.02, 0.12, (B, H, L)))
    W0, b0 = f32(0.05 * rng.standard_normal((H, d, d))), f32(0.05 * rng.standard_normal((H, d)))
    dWf, dbf = f32(rng.standard_normal((B, H, d, d))), f32(rng.standard_normal((B, H, d)))
    ref = [t.clone() for t in ttt.ttt_linear_bwd(Q, K, V, eta, W0, b0, dZ, dWf, dbf, mini_batch=16)]
    ttt.ttt_sync_status()
    out = (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V), torch.empty_like(eta),
           torch.empty_like(W0), torch.empty_like(b0))
    for _ in range(2):
        for t in out:
            t.fill_(float("nan"))
        ttt.ttt_linear_bwd_static(Q, K, V, eta, W0, b0, dZ, dWf, dbf, out=out, mini_batch=16)
        ttt.ttt_sync_status()
        for name, a, r in zip(("dQ", "dK", "dV", "deta", "dW0", "db0"), out, ref):
            assert torch.equal(a, r), name
