"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- a library routine (torch autograd / layer_norm / gelu, numpy matmul),
a closed form, a hand-worked example, an invariant, or finite differences.

Sources of the definitions: the update/apply equation (section 3.1) and the
mini-batch / dual-form description (sections 4.1-4.2) of the damodev.csdn.net
TTT article; the TTT-MLP shape and residual LayerNorm of the lryc.cn TTT
article (section 2.1).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(autouse=True)
def _float64_default():
    """torch's default dtype is float64 inside this module's tests only."""
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


def rand_problem(rng, B=1, H=2, L=32, d=8, ln=False, mlp=False, dh=None, eta_scale=0.3,
                 b0_std=0.1):
    Q = rng.standard_normal((B, H, L, d)) / np.sqrt(d)
    K = rng.standard_normal((B, H, L, d)) / np.sqrt(d)
    V = rng.standard_normal((B, H, L, d)) / np.sqrt(d)
    eta = rng.uniform(0.05, 1.0, (B, H, L)) * eta_scale
    p = dict(Q=Q, K=K, V=V, eta=eta)
    if mlp:
        dh = dh or 4 * d
        p["W1"] = rng.standard_normal((H, d, dh)) * 0.3
        p["b1"] = rng.standard_normal((H, dh)) * 0.1
        p["W2"] = rng.standard_normal((H, dh, d)) * 0.3
        p["b2"] = rng.standard_normal((H, d)) * 0.1
    else:
        p["W0"] = rng.standard_normal((H, d, d)) * 0.3
        p["b0"] = rng.standard_normal((H, d)) * b0_std
    if ln:
        p["gamma"] = 1.0 + 0.2 * rng.standard_normal((H, d))
        p["beta"] = 0.2 * rng.standard_normal((H, d))
    else:
        p["gamma"] = p["beta"] = None
    return p


def run_linear(p, mb, ln, dual=False, eps=1e-6, **kw):
    return oracle.ttt_linear(p["Q"], p["K"], p["V"], p["eta"], p["W0"], p["b0"], p["gamma"],
                             p["beta"], mini_batch=mb, ln=ln, eps=eps, dual=dual, **kw)


def run_mlp(p, mb, ln, dual=False, eps=1e-6, **kw):
    return oracle.ttt_mlp(p["Q"], p["K"], p["V"], p["eta"], p["W1"], p["b1"], p["W2"], p["b2"],
                          p["gamma"], p["beta"], mini_batch=mb, ln=ln, eps=eps, dual=dual, **kw)


# ---------------------------------------------------------------------------
# Brute force from the definition with torch autograd (library differentiation
# of the forward definitions; no hand-derived gradient anywhere).
# ---------------------------------------------------------------------------

def _ln(z, g, b, eps):
    return torch.nn.functional.layer_norm(z, (z.shape[-1],), g, b, eps)


def torch_f_linear(x, W, c, ln, g, b, eps):
    z = x @ W + c
    return x + _ln(z, g, b, eps) if ln else z


def torch_f_mlp(x, W1, b1, W2, b2, ln, g, b, eps):
    z2 = torch.nn.functional.gelu(x @ W1 + b1, approximate="tanh") @ W2 + b2
    return x + _ln(z2, g, b, eps) if ln else z2


def brute_force(p, mb, ln, mlp, eps=1e-6, loss="mse", wd=0.0):
    """Mini-batch TTT from the definition: at each mini-batch start take every
    token's gradient of its loss (autograd) -- 1/2||f(k_s) - v_s||^2 or -<f(k_s), v_s>,
    plus 1/2 wd ||W||^2 over the weight matrices -- then apply the updates token by
    token and read the output with the updated weights."""
    T = lambda a: None if a is None else torch.tensor(a)
    Q, K, V, eta = T(p["Q"]), T(p["K"]), T(p["V"]), T(p["eta"])
    B, H, L, d = Q.shape
    Z = torch.zeros_like(Q)
    finals = []
    for bi in range(B):
        for hi in range(H):
            g = None if p["gamma"] is None else T(p["gamma"][hi])
            b = None if p["beta"] is None else T(p["beta"][hi])
            if mlp:
                params = [T(p["W1"][hi]), T(p["b1"][hi]), T(p["W2"][hi]), T(p["b2"][hi])]
                f = lambda x, ps: torch_f_mlp(x, *ps, ln, g, b, eps)
            else:
                params = [T(p["W0"][hi]), T(p["b0"][hi])]
                f = lambda x, ps: torch_f_linear(x, *ps, ln, g, b, eps)
            for n0 in range(0, L, mb):
                start = [w.clone().requires_grad_(True) for w in params]
                grads = []
                mats = [start[0], start[2]] if mlp else [start[0]]
                for s in range(mb):
                    k, v = K[bi, hi, n0 + s], V[bi, hi, n0 + s]
                    fk = f(k, start)
                    lo = 0.5 * ((fk - v) ** 2).sum() if loss == "mse" else -(fk * v).sum()
                    lo = lo + 0.5 * wd * sum((w ** 2).sum() for w in mats)
                    grads.append(torch.autograd.grad(lo, start))
                cur = [w.detach().clone() for w in start]
                for t in range(mb):
                    e = eta[bi, hi, n0 + t]
                    cur = [w - e * gr for w, gr in zip(cur, grads[t])]
                    with torch.no_grad():
                        Z[bi, hi, n0 + t] = f(Q[bi, hi, n0 + t], cur)
                params = cur
            finals.append([w.numpy() for w in params])
    return Z.numpy(), finals


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("mb", [1, 4, 8])
def test_linear_matches_autograd_brute_force(ln, mb):
    rng = np.random.default_rng(1 + mb + 10 * ln)
    p = rand_problem(rng, B=2, H=2, L=16, d=6, ln=ln)
    Z, Wf, bf = run_linear(p, mb, ln)
    Zr, fin = brute_force(p, mb, ln, mlp=False)
    np.testing.assert_allclose(Z, Zr, rtol=1e-10, atol=1e-11)
    for idx, (W, c) in enumerate(fin):
        bi, hi = divmod(idx, 2)
        np.testing.assert_allclose(Wf[bi, hi], W, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(bf[bi, hi], c, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("mb", [1, 4])
def test_mlp_matches_autograd_brute_force(ln, mb):
    rng = np.random.default_rng(7 + mb + 10 * ln)
    p = rand_problem(rng, B=1, H=2, L=8, d=4, ln=ln, mlp=True, dh=16)
    Z, W1f, b1f, W2f, b2f = run_mlp(p, mb, ln)
    Zr, fin = brute_force(p, mb, ln, mlp=True)
    np.testing.assert_allclose(Z, Zr, rtol=1e-10, atol=1e-11)
    for hi, (W1, b1, W2, b2) in enumerate(fin):
        np.testing.assert_allclose(W1f[0, hi], W1, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(b1f[0, hi], b1, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(W2f[0, hi], W2, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(b2f[0, hi], b2, rtol=1e-10, atol=1e-11)


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_linear_d1.json")))
    x = g["inputs"]
    p = dict(Q=np.array(x["q"]).reshape(1, 1, 2, 1), K=np.array(x["k"]).reshape(1, 1, 2, 1),
             V=np.array(x["v"]).reshape(1, 1, 2, 1), eta=np.array(x["eta"]).reshape(1, 1, 2),
             W0=np.array([[[x["W0"]]]]), b0=np.array([[x["b0"]]]), gamma=None, beta=None)
    for dual in (False, True):
        Z, Wf, bf = run_linear(p, 2, False, dual=dual)
        np.testing.assert_allclose(Z.ravel(), g["expected"]["Z"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(Wf.ravel(), [g["expected"]["W_final"]], rtol=0, atol=1e-14)
        np.testing.assert_allclose(bf.ravel(), [g["expected"]["b_final"]], rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# Closed forms and special cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ln", [False, True])
def test_eta_zero_is_plain_forward(ln):
    rng = np.random.default_rng(3)
    p = rand_problem(rng, B=1, H=2, L=32, d=8, ln=ln)
    p["eta"][:] = 0.0
    Z, Wf, bf = run_linear(p, 8, ln)
    for hi in range(2):
        z = p["Q"][0, hi] @ p["W0"][hi] + p["b0"][hi]
        if ln:
            z = p["Q"][0, hi] + torch.nn.functional.layer_norm(
                torch.tensor(z), (8,), torch.tensor(p["gamma"][hi]), torch.tensor(p["beta"][hi]),
                1e-6).numpy()
        np.testing.assert_allclose(Z[0, hi], z, rtol=1e-12, atol=1e-13)
        np.testing.assert_array_equal(Wf[0, hi], p["W0"][hi])
        np.testing.assert_array_equal(bf[0, hi], p["b0"][hi])


def test_single_minibatch_closed_form():
    """L = b: W_final = W0 - K^T diag(eta) (K W0 + b0 - V)."""
    rng = np.random.default_rng(4)
    p = rand_problem(rng, B=1, H=1, L=16, d=8)
    Z, Wf, bf = run_linear(p, 16, False)
    K, V, e = p["K"][0, 0], p["V"][0, 0], p["eta"][0, 0]
    G = K @ p["W0"][0] + p["b0"][0] - V
    np.testing.assert_allclose(Wf[0, 0], p["W0"][0] - K.T @ (e[:, None] * G), rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose(bf[0, 0], p["b0"][0] - e @ G, rtol=1e-12, atol=1e-13)


def test_single_minibatch_closed_form_ln():
    """L = b with residual LN: W_final = W0 - K^T diag(eta) G, G the autograd
    gradient of 1/2||LN(K W0 + b0) - (V - K)||^2 w.r.t. the pre-LN rows."""
    rng = np.random.default_rng(5)
    p = rand_problem(rng, B=1, H=1, L=16, d=8, ln=True)
    Z, Wf, bf = run_linear(p, 16, True)
    K, V, e = p["K"][0, 0], p["V"][0, 0], p["eta"][0, 0]
    z = torch.tensor(K @ p["W0"][0] + p["b0"][0], requires_grad=True)
    loss = 0.5 * ((_ln(z, torch.tensor(p["gamma"][0]), torch.tensor(p["beta"][0]), 1e-6)
                   - torch.tensor(V - K)) ** 2).sum()
    G = torch.autograd.grad(loss, z)[0].numpy()
    np.testing.assert_allclose(Wf[0, 0], p["W0"][0] - K.T @ (e[:, None] * G), rtol=1e-11,
                               atol=1e-12)
    np.testing.assert_allclose(bf[0, 0], p["b0"][0] - e @ G, rtol=1e-11, atol=1e-12)


def test_zero_init_is_causal_linear_attention():
    """W0 = 0, b0 = 0, no LN, one mini-batch: G = -V, so
    z_t = sum_{s<=t} eta_s (q_t . k_s + 1) v_s (un-normalised causal linear
    attention with a constant-1 feature)."""
    rng = np.random.default_rng(6)
    p = rand_problem(rng, B=1, H=1, L=24, d=8)
    p["W0"][:] = 0.0
    p["b0"][:] = 0.0
    Z, _, _ = run_linear(p, 24, False)
    Q, K, V, e = p["Q"][0, 0], p["K"][0, 0], p["V"][0, 0], p["eta"][0, 0]
    A = np.tril(Q @ K.T + 1.0) * e[None, :]
    np.testing.assert_allclose(Z[0, 0], A @ V, rtol=1e-12, atol=1e-13)


def test_ln_d2_eps0_has_zero_gradient():
    """With d = 2 and eps = 0, LN(z) only depends on sign(z1 - z2), so every
    gradient vanishes: the weights never move and z = q + LN(q W0 + b0)."""
    rng = np.random.default_rng(8)
    p = rand_problem(rng, B=1, H=1, L=16, d=2, ln=True)
    Z, Wf, bf = run_linear(p, 4, True, eps=0.0)
    np.testing.assert_allclose(Wf[0, 0], p["W0"][0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(bf[0, 0], p["b0"][0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("ln", [False, True])
def test_minibatch_differs_from_online(ln):
    """b = 16 is not b = 1 (the mini-batch reading is really exercised)."""
    rng = np.random.default_rng(9)
    p = rand_problem(rng, B=1, H=1, L=32, d=8, ln=ln)
    Z1, _, _ = run_linear(p, 1, ln)
    Z16, _, _ = run_linear(p, 16, ln)
    assert np.abs(Z1 - Z16).max() > 1e-3


# ---------------------------------------------------------------------------
# Primal == dual (the dual form only reorders the arithmetic)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("mb", [1, 4, 16])
def test_linear_primal_equals_dual(ln, mb):
    rng = np.random.default_rng(11 + mb)
    p = rand_problem(rng, B=2, H=2, L=64, d=16, ln=ln)
    a = run_linear(p, mb, ln)
    b = run_linear(p, mb, ln, dual=True)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("mb", [1, 4])
def test_mlp_primal_equals_dual(ln, mb):
    rng = np.random.default_rng(21 + mb)
    p = rand_problem(rng, B=1, H=2, L=16, d=8, ln=ln, mlp=True)
    a = run_mlp(p, mb, ln)
    b = run_mlp(p, mb, ln, dual=True)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# Carry, structure
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mlp", [False, True])
def test_state_carry(mlp):
    """forward(L1) then forward(L2) started from the final state == forward(L1+L2)."""
    rng = np.random.default_rng(31)
    p = rand_problem(rng, B=2, H=2, L=32, d=8, ln=True, mlp=mlp)
    run = run_mlp if mlp else run_linear
    full = run(p, 8, True)
    cut = 16
    p1 = dict(p, Q=p["Q"][:, :, :cut], K=p["K"][:, :, :cut], V=p["V"][:, :, :cut],
              eta=p["eta"][:, :, :cut])
    first = run(p1, 8, True)
    sl = lambda a: np.ascontiguousarray(a[:, :, cut:])
    if mlp:
        Z2, *fin2 = oracle.ttt_mlp(sl(p["Q"]), sl(p["K"]), sl(p["V"]), sl(p["eta"]), *first[1:],
                                   p["gamma"], p["beta"], mini_batch=8, ln=True,
                                   init_per_batch=True)
    else:
        Z2, *fin2 = oracle.ttt_linear(sl(p["Q"]), sl(p["K"]), sl(p["V"]), sl(p["eta"]), first[1],
                                      first[2], p["gamma"], p["beta"], mini_batch=8, ln=True,
                                      init_per_batch=True)
    np.testing.assert_allclose(np.concatenate([first[0], Z2], axis=2), full[0], rtol=1e-12,
                               atol=1e-13)
    for x, y in zip(fin2, full[1:]):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13)


def test_linear_column_permutation():
    """Without LN the output columns are independent: permuting the columns of
    W0, b0 and V permutes the columns of Z and W_final."""
    rng = np.random.default_rng(41)
    p = rand_problem(rng, B=1, H=1, L=32, d=8)
    perm = rng.permutation(8)
    Z, Wf, bf = run_linear(p, 8, False)
    pp = dict(p, W0=p["W0"][:, :, perm], b0=p["b0"][:, perm], V=p["V"][..., perm])
    Zp, Wfp, bfp = run_linear(pp, 8, False)
    np.testing.assert_allclose(Zp, Z[..., perm], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Wfp, Wf[..., perm], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(bfp, bf[..., perm], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Hand-derived gradients against library routines and finite differences
# ---------------------------------------------------------------------------

def test_gelu_matches_torch_tanh_gelu():
    xs = np.linspace(-6, 6, 97)
    ref = torch.nn.functional.gelu(torch.tensor(xs), approximate="tanh").numpy()
    np.testing.assert_allclose([oracle.gelu(x) for x in xs], ref, rtol=1e-13, atol=1e-15)


def test_gelu_prime_matches_autograd():
    xs = torch.tensor(np.linspace(-6, 6, 97), requires_grad=True)
    torch.nn.functional.gelu(xs, approximate="tanh").sum().backward()
    np.testing.assert_allclose([oracle.gelu_prime(x) for x in xs.detach().numpy()],
                               xs.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_ln_fwd_matches_torch():
    rng = np.random.default_rng(51)
    z, g, b = rng.standard_normal(16), rng.standard_normal(16), rng.standard_normal(16)
    ref = torch.nn.functional.layer_norm(torch.tensor(z), (16,), torch.tensor(g), torch.tensor(b),
                                         1e-6).numpy()
    np.testing.assert_allclose(oracle.ln_fwd(z, g, b, 1e-6), ref, rtol=1e-13, atol=1e-14)


def test_ln_bwd_matches_autograd():
    rng = np.random.default_rng(52)
    z, y = rng.standard_normal(16), rng.standard_normal(16)
    g, b = 1 + 0.3 * rng.standard_normal(16), 0.3 * rng.standard_normal(16)
    zt = torch.tensor(z, requires_grad=True)
    loss = 0.5 * ((_ln(zt, torch.tensor(g), torch.tensor(b), 1e-6) - torch.tensor(y)) ** 2).sum()
    ref = torch.autograd.grad(loss, zt)[0].numpy()
    np.testing.assert_allclose(oracle.ln_l2_bwd(z, y, g, b, 1e-6), ref, rtol=1e-11, atol=1e-13)


def _fd(f, x, h=1e-6):
    out = np.empty_like(x)
    flat = x.reshape(-1)
    o = out.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + h
        fp = f()
        flat[i] = old - h
        fm = f()
        flat[i] = old
        o[i] = (fp - fm) / (2 * h)
    return out


@pytest.mark.parametrize("ln", [False, True])
def test_linear_token_grad_finite_differences(ln):
    rng = np.random.default_rng(61 + ln)
    d = 6
    k, v = rng.standard_normal(d), rng.standard_normal(d)
    W, c = rng.standard_normal((d, d)) * 0.5, rng.standard_normal(d) * 0.3
    g, b = (1 + 0.3 * rng.standard_normal(d), 0.3 * rng.standard_normal(d)) if ln else (None, None)
    gW, gc = oracle.linear_token_grad(k, v, W, c, ln, g, b)
    loss = lambda: oracle.linear_token_loss(k, v, W, c, ln, g, b)
    fW, fc = _fd(loss, W), _fd(loss, c)
    assert np.abs(gW - fW).max() <= 1e-6 * max(1.0, np.abs(fW).max())
    assert np.abs(gc - fc).max() <= 1e-6 * max(1.0, np.abs(fc).max())


@pytest.mark.parametrize("ln", [False, True])
def test_mlp_token_grad_finite_differences(ln):
    rng = np.random.default_rng(71 + ln)
    d, dh = 4, 12
    k, v = rng.standard_normal(d), rng.standard_normal(d)
    W1, b1 = rng.standard_normal((d, dh)) * 0.5, rng.standard_normal(dh) * 0.3
    W2, b2 = rng.standard_normal((dh, d)) * 0.5, rng.standard_normal(d) * 0.3
    g, b = (1 + 0.3 * rng.standard_normal(d), 0.3 * rng.standard_normal(d)) if ln else (None, None)
    grads = oracle.mlp_token_grad(k, v, W1, b1, W2, b2, ln, g, b)
    loss = lambda: oracle.mlp_token_loss(k, v, W1, b1, W2, b2, ln, g, b)
    for got, x in zip(grads, (W1, b1, W2, b2)):
        fd = _fd(loss, x)
        assert np.abs(got - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max())


def test_bad_arguments_rejected():
    rng = np.random.default_rng(81)
    p = rand_problem(rng, B=1, H=1, L=20, d=4)
    with pytest.raises(ValueError):
        run_linear(p, 16, False)   # L % b != 0


# --------------------------------------------------------------------------
# the per-token learning-rate gate (lryc.cn TTT article, section 2.2)
# --------------------------------------------------------------------------

def test_gate_zero_theta_is_half_the_base_rate():
    rng = np.random.default_rng(71)
    x = rng.standard_normal((2, 5, 12))
    eta = oracle.eta_gate(x, np.zeros((3, 12)), 0.3)
    np.testing.assert_array_equal(eta, np.full((2, 3, 5), 0.15))


def test_gate_hand_value():
    """sigmoid(ln 3) = 3/4 exactly: one feature, theta = 1, x = ln 3."""
    eta = oracle.eta_gate(np.array([[[np.log(3.0)], [-np.log(3.0)]]]), np.array([[1.0]]), 2.0)
    np.testing.assert_allclose(eta[0, 0], [1.5, 0.5], rtol=1e-15)


def test_gate_matches_library_sigmoid():
    """Against scipy's expit of a numpy contraction, with every dimension distinct so that a
    transposed index fails."""
    from scipy.special import expit
    rng = np.random.default_rng(72)
    B, L, Dx, H = 2, 7, 33, 5
    x = rng.standard_normal((B, L, Dx))
    theta = rng.standard_normal((H, Dx)) * 0.3
    ref = 0.125 * expit(np.einsum("blk,hk->bhl", x, theta))
    np.testing.assert_allclose(oracle.eta_gate(x, theta, 0.125), ref, rtol=1e-13, atol=0)


def test_gate_symmetry_and_saturation():
    """sigmoid(u) + sigmoid(-u) = 1, and large |u| saturates without overflow."""
    rng = np.random.default_rng(73)
    x = rng.standard_normal((1, 9, 16))
    theta = rng.standard_normal((2, 16))
    s = oracle.eta_gate(x, theta, 1.0) + oracle.eta_gate(-x, theta, 1.0)
    np.testing.assert_allclose(s, 1.0, rtol=1e-15)
    big = oracle.eta_gate(np.full((1, 2, 1), 800.0) * np.array([1.0, -1.0])[None, :, None],
                          np.ones((1, 1)), 0.5)
    assert np.isfinite(big).all()
    np.testing.assert_allclose(big[0, 0], [0.5, 0.0], atol=1e-300)



# --------------------------------------------------------------------------
# inner-learner variants (ai-feeds "Modular TTT" page, method overview): the loss
# (1/2 ||f(k) - v||^2 or the inner product -<f(k), v>) and weight decay
# --------------------------------------------------------------------------

VARIANTS = [("ip", 0.0), ("mse", 0.3), ("ip", 0.3)]


@pytest.mark.parametrize("loss,wd", VARIANTS)
@pytest.mark.parametrize("ln", [False, True])
@pytest.mark.parametrize("mb", [1, 4])
def test_linear_variants_match_autograd_brute_force(loss, wd, ln, mb):
    rng = np.random.default_rng(81 + mb + 10 * ln + 100 * (loss == "ip"))
    p = rand_problem(rng, B=1, H=2, L=16, d=6, ln=ln)
    Z, Wf, bf = run_linear(p, mb, ln, loss=loss, weight_decay=wd)
    Zr, fin = brute_force(p, mb, ln, mlp=False, loss=loss, wd=wd)
    np.testing.assert_allclose(Z, Zr, rtol=1e-10, atol=1e-11)
    for idx, (W, c) in enumerate(fin):
        np.testing.assert_allclose(Wf[0, idx], W, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(bf[0, idx], c, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("loss,wd", VARIANTS)
@pytest.mark.parametrize("ln", [False, True])
def test_mlp_variants_match_autograd_brute_force(loss, wd, ln):
    rng = np.random.default_rng(91 + 10 * ln + 100 * (loss == "ip"))
    p = rand_problem(rng, B=1, H=2, L=8, d=4, ln=ln, mlp=True, dh=16)
    Z, W1f, b1f, W2f, b2f = run_mlp(p, 4, ln, loss=loss, weight_decay=wd)
    Zr, fin = brute_force(p, 4, ln, mlp=True, loss=loss, wd=wd)
    np.testing.assert_allclose(Z, Zr, rtol=1e-9, atol=1e-11)
    for idx, (W1, b1, W2, b2) in enumerate(fin):
        np.testing.assert_allclose(W1f[0, idx], W1, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(W2f[0, idx], W2, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(b1f[0, idx], b1, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(b2f[0, idx], b2, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("loss,wd", VARIANTS)
@pytest.mark.parametrize("ln", [False, True])
def test_variants_primal_equals_dual(loss, wd, ln):
    rng = np.random.default_rng(101 + 10 * ln)
    p = rand_problem(rng, B=1, H=2, L=32, d=8, ln=ln)
    for a, b in zip(run_linear(p, 8, ln, loss=loss, weight_decay=wd),
                    run_linear(p, 8, ln, dual=True, loss=loss, weight_decay=wd)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)
    q = rand_problem(rng, B=1, H=1, L=16, d=4, ln=ln, mlp=True, dh=8)
    for a, b in zip(run_mlp(q, 4, ln, loss=loss, weight_decay=wd),
                    run_mlp(q, 4, ln, dual=True, loss=loss, weight_decay=wd)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("mb", [1, 4, 16])
def test_inner_product_loss_is_causal_linear_attention(mb):
    """With the inner-product loss and no LayerNorm the gradient is -v whatever the
    weights, so from W0 = 0, b0 = 0 every mini-batch size gives
    z_t = sum_{s <= t} eta_s (q_t . k_s + 1) v_s over the whole sequence."""
    rng = np.random.default_rng(111)
    p = rand_problem(rng, B=1, H=2, L=32, d=5)
    p["W0"] = np.zeros_like(p["W0"])
    p["b0"] = np.zeros_like(p["b0"])
    Z, Wf, bf = run_linear(p, mb, False, loss="ip")
    for h in range(2):
        Q, K, V, e = p["Q"][0, h], p["K"][0, h], p["V"][0, h], p["eta"][0, h]
        A = np.tril((Q @ K.T + 1.0) * e[None, :])
        np.testing.assert_allclose(Z[0, h], A @ V, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(Wf[0, h], K.T @ (e[:, None] * V), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(bf[0, h], e @ V, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mb", [1, 4])
def test_weight_decay_with_zero_keys(mb):
    """With all keys zero the gradient part of the weight update vanishes, so weight decay
    alone shrinks W by 1 - lambda * (sum of the mini-batch's eta) per mini-batch."""
    rng = np.random.default_rng(121)
    p = rand_problem(rng, B=1, H=1, L=16, d=4)
    p["K"] = np.zeros_like(p["K"])
    lam = 0.7
    _, Wf, _ = run_linear(p, mb, False, weight_decay=lam)
    e = p["eta"][0, 0]
    factor = np.prod([1.0 - lam * e[n:n + mb].sum() for n in range(0, 16, mb)])
    np.testing.assert_allclose(Wf[0, 0], factor * p["W0"][0], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("ln", [False, True])
def test_inner_product_gradients_by_finite_differences(ln):
    rng = np.random.default_rng(131 + ln)
    d, dh, h = 5, 7, 1e-6
    k, v = rng.standard_normal(d), rng.standard_normal(d)
    W, c = rng.standard_normal((d, d)) * 0.4, rng.standard_normal(d) * 0.1
    gm, bt = 1.0 + 0.2 * rng.standard_normal(d), 0.1 * rng.standard_normal(d)
    kw = dict(ln=ln, gamma=gm, beta=bt, loss="ip")
    gW, gc = oracle.linear_token_grad(k, v, W, c, **kw)
    for (i, j) in [(0, 0), (2, 3), (4, 1)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[i, j] += h
        Wm[i, j] -= h
        fd = (oracle.linear_token_loss(k, v, Wp, c, **kw) - oracle.linear_token_loss(k, v, Wm, c, **kw)) / (2 * h)
        assert abs(fd - gW[i, j]) <= 1e-6 * max(1.0, abs(fd))
    W1, b1 = rng.standard_normal((d, dh)) * 0.4, rng.standard_normal(dh) * 0.1
    W2, b2 = rng.standard_normal((dh, d)) * 0.4, rng.standard_normal(d) * 0.1
    g1, _, g2, _ = oracle.mlp_token_grad(k, v, W1, b1, W2, b2, **kw)
    for (M, G, ij) in [(W1, g1, (1, 2)), (W2, g2, (3, 4))]:
        Mp, Mm = M.copy(), M.copy()
        Mp[ij] += h
        Mm[ij] -= h
        args_p = (W1 if M is not W1 else Mp, b1, W2 if M is not W2 else Mp, b2)
        args_m = (W1 if M is not W1 else Mm, b1, W2 if M is not W2 else Mm, b2)
        fd = (oracle.mlp_token_loss(k, v, *args_p, **kw) - oracle.mlp_token_loss(k, v, *args_m, **kw)) / (2 * h)
        assert abs(fd - G[ij]) <= 1e-6 * max(1.0, abs(fd))


def test_qkv_projection_against_a_triple_loop():
    """The input projections (lryc.cn TTT article, section 2.2: Q, K, V as views of the
    layer's input tokens) against a plain triple loop on a tiny case with every dimension
    distinct (a transposed weight or a swapped Q/K/V slice fails it)."""
    rng = np.random.default_rng(3)
    B, L, Dx, H, d = 2, 3, 5, 2, 3
    x = rng.standard_normal((B, L, Dx))
    W = rng.standard_normal((3 * H * d, Dx))
    got = oracle.qkv_proj(x, W, H, d)
    for k in range(3):
        want = np.zeros((B, H, L, d))
        for b in range(B):
            for h in range(H):
                for t in range(L):
                    for j in range(d):
                        n = k * H * d + h * d + j
                        want[b, h, t, j] = sum(x[b, t, i] * W[n, i] for i in range(Dx))
        np.testing.assert_allclose(got[k], want, rtol=1e-12, atol=1e-12)


def test_qkv_projection_selection_matrix_copies_features():
    """W selecting input features (row n picks feature n mod Dx) makes Q, K, V copies of x."""
    rng = np.random.default_rng(4)
    B, L, H, d = 1, 4, 2, 4
    Dx = 3 * H * d
    x = rng.standard_normal((B, L, Dx))
    W = np.eye(3 * H * d, Dx)
    Q, K, V = oracle.qkv_proj(x, W, H, d)
    for k, out in enumerate((Q, K, V)):
        for h in range(H):
            np.testing.assert_array_equal(out[0, h], x[0, :, k * H * d + h * d:k * H * d + (h + 1) * d])
