"""Pins of the backward oracle (oracle/backward.py) against things other than itself.

The backward oracle is torch autograd through a float64 PyTorch restatement of the
forward.  These tests tie it to the C oracle's forward (an independent program) by central
finite differences, for every input and every variant, and to the closed form at eta = 0
(the state never moves: Z = Q W0 + b0, or Q + LN(Q W0 + b0))."""
import numpy as np
import pytest

import oracle
from oracle.backward import ttt_linear_grad

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")

INPUTS = ["Q", "K", "V", "eta", "W0", "b0"]


def problem(rng, B=1, H=2, L=8, d=4, ln=False):
    p = dict(Q=rng.standard_normal((B, H, L, d)) / np.sqrt(d),
             K=rng.standard_normal((B, H, L, d)) / np.sqrt(d),
             V=rng.standard_normal((B, H, L, d)) / np.sqrt(d),
             eta=rng.uniform(0.1, 0.6, (B, H, L)),
             W0=rng.standard_normal((H, d, d)) * 0.3,
             b0=rng.standard_normal((H, d)) * 0.1,
             gamma=1.0 + 0.2 * rng.standard_normal((H, d)) if ln else None,
             beta=0.2 * rng.standard_normal((H, d)) if ln else None)
    cot = dict(dZ=rng.standard_normal((B, H, L, d)),
               dW_final=rng.standard_normal((B, H, d, d)),
               db_final=rng.standard_normal((B, H, d)))
    return p, cot


def outer_loss(p, cot, mb, ln, loss, wd):
    """F = <Z, dZ> + <W_final, dW_final> + <b_final, db_final> with the C oracle's forward."""
    Z, Wf, bf = oracle.ttt_linear(p["Q"], p["K"], p["V"], p["eta"], p["W0"], p["b0"],
                                  p["gamma"], p["beta"], mini_batch=mb, ln=ln, eps=1e-6,
                                  loss=loss, weight_decay=wd)
    return float((Z * cot["dZ"]).sum() + (Wf * cot["dW_final"]).sum()
                 + (bf * cot["db_final"]).sum())


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("loss,wd", [("mse", 0.0), ("ip", 0.0), ("mse", 0.3)])
def test_gradients_match_finite_differences_of_the_c_oracle(ln, loss, wd):
    rng = np.random.default_rng(7 + 2 * ln + (loss == "ip") + 5 * (wd > 0))
    p, cot = problem(rng, ln=ln)
    mb = 4   # two mini-batches of four tokens
    g = ttt_linear_grad(p["Q"], p["K"], p["V"], p["eta"], p["W0"], p["b0"], p["gamma"],
                        p["beta"], cot["dZ"], cot["dW_final"], cot["db_final"],
                        mini_batch=mb, ln=ln, eps=1e-6, loss=loss, weight_decay=wd)
    names = INPUTS + (["gamma", "beta"] if ln else [])
    h = 1e-5
    for name in names:
        for trial in range(2):
            delta = rng.standard_normal(np.shape(p[name]))
            plus = dict(p, **{name: p[name] + h * delta})
            minus = dict(p, **{name: p[name] - h * delta})
            fd = (outer_loss(plus, cot, mb, ln, loss, wd) - outer_loss(minus, cot, mb, ln, loss, wd)) / (2 * h)
            an = float((g["d" + name] * delta).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)


def test_eta_zero_closed_form():
    """eta = 0: Z = Q W0 + b0 and the state stays W0, so dQ = dZ W0^T, dK = dV = 0,
    dW0 = sum_b (Q^T dZ + dW_final), db0 = sum_b (1^T dZ + db_final)."""
    rng = np.random.default_rng(3)
    p, cot = problem(rng, B=2, H=2, L=8, d=4)
    p["eta"] = np.zeros_like(p["eta"])
    g = ttt_linear_grad(p["Q"], p["K"], p["V"], p["eta"], p["W0"], p["b0"], None, None,
                        cot["dZ"], cot["dW_final"], cot["db_final"], mini_batch=4)
    W0, Q, dZ = p["W0"], p["Q"], cot["dZ"]
    np.testing.assert_allclose(g["dQ"], np.einsum("bhtj,hij->bhti", dZ, W0), atol=1e-12)
    np.testing.assert_allclose(g["dK"], 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dV"], 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dW0"], np.einsum("bhti,bhtj->hij", Q, dZ) + cot["dW_final"].sum(0),
                               atol=1e-12)
    np.testing.assert_allclose(g["db0"], dZ.sum((0, 2)) + cot["db_final"].sum(0), atol=1e-12)


def test_per_batch_initial_state_gradient_is_per_batch():
    """With init_per_batch the initial state has its own gradient per (batch, head): it
    equals the head-shared gradient of that batch alone."""
    rng = np.random.default_rng(11)
    p, cot = problem(rng, B=2, H=1, L=8, d=4)
    W0b = np.broadcast_to(p["W0"], (2, 1, 4, 4)).copy()
    b0b = np.broadcast_to(p["b0"], (2, 1, 4)).copy()
    g = ttt_linear_grad(p["Q"], p["K"], p["V"], p["eta"], W0b, b0b, None, None, cot["dZ"],
                        cot["dW_final"], cot["db_final"], mini_batch=4, init_per_batch=True)
    for bi in range(2):
        sl = lambda a: a[bi:bi + 1]
        g1 = ttt_linear_grad(sl(p["Q"]), sl(p["K"]), sl(p["V"]), sl(p["eta"]), p["W0"], p["b0"],
                             None, None, sl(cot["dZ"]), sl(cot["dW_final"]), sl(cot["db_final"]),
                             mini_batch=4)
        np.testing.assert_allclose(g["dW0"][bi], g1["dW0"], atol=1e-12)
        np.testing.assert_allclose(g["db0"][bi], g1["db0"], atol=1e-12)
