"""CPU oracle for the backward pass of the TTT-Linear inner loop (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import
this module.  It shares no code with the CUDA path.

What it computes: the gradients of a scalar outer loss
    F = <Z, dZ> + <W_final, dW_final> + <b_final, db_final>
with respect to every input of the TTT-Linear forward (Q, K, V, eta, W0, b0, gamma,
beta), i.e. the vector-Jacobian product that training through the inner loop needs (the
meta-learning gradient of the damodev.csdn.net TTT article, section 6.1, taken through
the mini-batch inner loop of sections 4.1-4.2; residual LayerNorm of the lryc.cn TTT
article, section 2.1; inner-learner variants of the ai-feeds Modular TTT page).

How: the forward is restated here in float64 PyTorch ops, token by token, exactly as the
C oracle's primal form defines it (every gradient of a mini-batch at the mini-batch's
starting state, each output read from the state after its own token's update), and the
outer gradient is taken by torch autograd, a library primitive.  The inner gradient of
the reconstruction loss is itself taken by autograd with the graph kept
(``create_graph=True``), so no hand-derived derivative enters: the result is the
gradient of the definition.  Pinned in ``tests/test_backward_pins.py`` by central finite
differences of the C oracle's forward and by the eta = 0 closed form.
"""
from __future__ import annotations

import numpy as np
import torch


def _ln(z, gamma, beta, eps):
    mu = z.mean(-1, keepdim=True)
    var = ((z - mu) ** 2).mean(-1, keepdim=True)
    return (z - mu) / torch.sqrt(var + eps) * gamma + beta


def _f(x, W, c, ln, gamma, beta, eps):
    """The inner model on rows x: x W + c, or x + LN(x W + c) (residual form)."""
    z = x @ W + c
    return x + _ln(z, gamma, beta, eps) if ln else z


def _scan_one(q, k, v, eta, W, c, gamma, beta, mb, ln, eps, loss, wd):
    """One (batch, head): Z [L, d], W_final, c_final, all float64 torch with autograd."""
    L = q.shape[0]
    outs = []
    for n0 in range(0, L, mb):
        kb, vb, qb, eb = k[n0:n0 + mb], v[n0:n0 + mb], q[n0:n0 + mb], eta[n0:n0 + mb]
        # per-token loss at the mini-batch's starting state; its gradient w.r.t. z = k W + c
        z = kb @ W + c
        out = kb + _ln(z, gamma, beta, eps) if ln else z
        if loss == "ip":
            ell = -(out * vb).sum()
        else:
            ell = 0.5 * ((out - vb) ** 2).sum()
        g, = torch.autograd.grad(ell, z, create_graph=True)   # [mb, d], row s = dl_s/dz_s
        # token by token: W_t = (1 - wd cum_t) W_start - sum_{s<=t} eta_s k_s^T g_s
        cum_eta = torch.cumsum(eb, 0)
        gw = torch.cumsum(eb[:, None, None] * kb[:, :, None] * g[:, None, :], 0)   # [mb, d, d]
        gc = torch.cumsum(eb[:, None] * g, 0)                                       # [mb, d]
        Wt = (1.0 - wd * cum_eta)[:, None, None] * W[None] - gw
        ct = c[None] - gc
        zq = torch.einsum("ti,tij->tj", qb, Wt) + ct
        outs.append(qb + _ln(zq, gamma, beta, eps) if ln else zq)
        W, c = Wt[-1], ct[-1]
    return torch.cat(outs, 0), W, c


def ttt_linear_grad(Q, K, V, eta, W0, b0, gamma, beta, dZ, dW_final=None, db_final=None, *,
                    mini_batch: int, ln: bool = False, eps: float = 1e-6, loss: str = "mse",
                    weight_decay: float = 0.0, init_per_batch: bool = False):
    """Gradients of F = <Z, dZ> + <W_final, dW_final> + <b_final, db_final>.

    Shapes as the forward: Q, K, V, dZ [B, H, L, d]; eta [B, H, L]; W0 [H, d, d] (or
    [B, H, d, d] with init_per_batch); b0 [H, d] (or [B, H, d]); gamma, beta [H, d] (used
    iff ln); dW_final [B, H, d, d], db_final [B, H, d] (None = 0).  Returns a dict of
    float64 numpy arrays: dQ, dK, dV, deta, dW0, db0 (shaped like W0, b0: summed over the
    batch when the initial state is shared by the head) and, with ln, dgamma, dbeta [H, d].
    """
    B, H, L, d = np.shape(Q)
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    Qt, Kt, Vt, Et = t(Q), t(K), t(V), t(eta)
    W0t, b0t = t(W0), t(b0)
    gt = t(gamma) if ln else None
    bt = t(beta) if ln else None
    F = torch.zeros((), dtype=torch.float64)
    dZt = torch.tensor(np.asarray(dZ, np.float64))
    for bi in range(B):
        for hi in range(H):
            W = W0t[bi, hi] if init_per_batch else W0t[hi]
            c = b0t[bi, hi] if init_per_batch else b0t[hi]
            Z, Wf, cf = _scan_one(Qt[bi, hi], Kt[bi, hi], Vt[bi, hi], Et[bi, hi], W, c,
                                  gt[hi] if ln else None, bt[hi] if ln else None,
                                  mini_batch, ln, eps, loss, weight_decay)
            F = F + (Z * dZt[bi, hi]).sum()
            if dW_final is not None:
                F = F + (Wf * torch.tensor(np.asarray(dW_final[bi, hi], np.float64))).sum()
            if db_final is not None:
                F = F + (cf * torch.tensor(np.asarray(db_final[bi, hi], np.float64))).sum()
    wrt = [Qt, Kt, Vt, Et, W0t, b0t] + ([gt, bt] if ln else [])
    grads = torch.autograd.grad(F, wrt, allow_unused=True)
    names = ["dQ", "dK", "dV", "deta", "dW0", "db0"] + (["dgamma", "dbeta"] if ln else [])
    return {n: (np.zeros(w.shape) if g is None else g.detach().numpy())
            for n, g, w in zip(names, grads, wrt)}
