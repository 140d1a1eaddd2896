"""CPU oracle for the TTT layer's inner loop (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls it, and shares no code with
it.  The oracle is ``ttt_oracle.c`` (plain C, IEEE double, single-threaded),
compiled with gcc into ``liboracle.so`` beside this file; this module only
marshals numpy arrays into it.

What it computes, and where the pages say so, is stated in the header of
``ttt_oracle.c``.  ``parity unpinned``: the choice of LayerNorm eps and of the
synthetic eta-gate distribution are spec choices, not computed results; every
computed function is pinned by the CPU tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ttt_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ttt_oracle.c into liboracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
             "-D_DEFAULT_SOURCE", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_gelu.restype = d
            lib.oracle_gelu.argtypes = [d]
            lib.oracle_gelu_prime.restype = d
            lib.oracle_gelu_prime.argtypes = [d]
            lib.oracle_ln_fwd.restype = None
            lib.oracle_ln_fwd.argtypes = [dp, i, dp, dp, d, dp]
            lib.oracle_ln_l2_bwd.restype = None
            lib.oracle_ln_l2_bwd.argtypes = [dp, dp, i, dp, dp, d, dp]
            lib.oracle_linear_token_loss_v.restype = d
            lib.oracle_linear_token_loss_v.argtypes = [dp, dp, dp, dp, i, i, i, dp, dp, d]
            lib.oracle_linear_token_grad_v.restype = None
            lib.oracle_linear_token_grad_v.argtypes = [dp, dp, dp, dp, i, i, i, dp, dp, d, dp, dp]
            lib.oracle_mlp_token_loss_v.restype = d
            lib.oracle_mlp_token_loss_v.argtypes = [dp, dp, dp, dp, dp, dp, i, i, i, i, dp, dp, d]
            lib.oracle_mlp_token_grad_v.restype = None
            lib.oracle_mlp_token_grad_v.argtypes = [dp, dp, dp, dp, dp, dp, i, i, i, i, dp, dp, d,
                                                    dp, dp, dp, dp]
            lib.oracle_eta_gate.restype = i
            lib.oracle_eta_gate.argtypes = [i, i, i, i, d, dp, dp, dp]
            for name in ("oracle_ttt_linear_v", "oracle_ttt_linear_dual_v"):
                fn = getattr(lib, name)
                fn.restype = i
                fn.argtypes = [i, i, i, i, i, i, d, i, i, d] + [dp] * 11
            for name in ("oracle_ttt_mlp_v", "oracle_ttt_mlp_dual_v"):
                fn = getattr(lib, name)
                fn.restype = i
                fn.argtypes = [i, i, i, i, i, i, i, d, i, i, d] + [dp] * 15
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


# --------------------------------------------------------------------------
# per-token learning rate
# --------------------------------------------------------------------------

def eta_gate(x, theta, eta_base: float):
    """eta [B, H, L] = eta_base * sigmoid(theta[h] . x[b, t]) for the layer input
    x [B, L, Dx] and the per-head gate vectors theta [H, Dx] (float64)."""
    x, theta = _f64(x), _f64(theta)
    B, L, Dx = x.shape
    H = theta.shape[0]
    if theta.shape != (H, Dx):
        raise ValueError("theta must be [H, Dx]")
    eta = np.empty((B, H, L))
    rc = _load().oracle_eta_gate(B, H, L, Dx, float(eta_base), _p(x), _p(theta), _p(eta))
    if rc != 0:
        raise ValueError(f"oracle_eta_gate returned {rc}")
    return eta


def qkv_proj(x, W, H: int, d: int):
    """The layer's input projections (the views theta_Q x, theta_K x, theta_V x of the lryc.cn
    TTT article, section 2.2): for tokens x [B, L, Dx] and the stacked projection matrices
    W [3 H d, Dx] (row n = one output unit), Q[b, h, t, j] = sum_i x[b, t, i] W[h d + j, i],
    K from rows H d + h d + j, V from rows 2 H d + h d + j; each [B, H, L, d], float64.
    (A library matrix product; pinned against a plain triple loop.)"""
    x, W = _f64(x), _f64(W)
    B, L, Dx = x.shape
    if W.shape != (3 * H * d, Dx):
        raise ValueError("W must be [3 H d, Dx]")
    Y = np.matmul(x, W.T)                                   # [B, L, 3 H d]
    return tuple(Y[..., k * H * d:(k + 1) * H * d].reshape(B, L, H, d).transpose(0, 2, 1, 3).copy()
                 for k in range(3))


# --------------------------------------------------------------------------
# elementwise pieces and per-token losses/gradients (for the FD pins)
# --------------------------------------------------------------------------

def gelu(x: float) -> float:
    return _load().oracle_gelu(float(x))


def gelu_prime(x: float) -> float:
    return _load().oracle_gelu_prime(float(x))


def ln_fwd(z, gamma=None, beta=None, eps=1e-6):
    z = _f64(z)
    out = np.empty_like(z)
    g = None if gamma is None else _f64(gamma)
    b = None if beta is None else _f64(beta)
    _load().oracle_ln_fwd(_p(z), z.size, _p(g), _p(b), eps, _p(out))
    return out


def ln_l2_bwd(z, y, gamma=None, beta=None, eps=1e-6):
    z, y = _f64(z), _f64(y)
    out = np.empty_like(z)
    g = None if gamma is None else _f64(gamma)
    b = None if beta is None else _f64(beta)
    _load().oracle_ln_l2_bwd(_p(z), _p(y), z.size, _p(g), _p(b), eps, _p(out))
    return out


LOSSES = {"mse": 0, "ip": 1}   # 1/2 ||f(k) - v||^2, or the inner product -<f(k), v>


def _loss_id(loss: str) -> int:
    if loss not in LOSSES:
        raise ValueError(f"loss must be one of {sorted(LOSSES)}")
    return LOSSES[loss]


def linear_token_loss(k, v, W, c, ln=False, gamma=None, beta=None, eps=1e-6, loss="mse"):
    k, v, W, c = _f64(k), _f64(v), _f64(W), _f64(c)
    g = None if gamma is None else _f64(gamma)
    b = None if beta is None else _f64(beta)
    return _load().oracle_linear_token_loss_v(_p(k), _p(v), _p(W), _p(c), k.size, int(ln),
                                              _loss_id(loss), _p(g), _p(b), eps)


def linear_token_grad(k, v, W, c, ln=False, gamma=None, beta=None, eps=1e-6, loss="mse"):
    k, v, W, c = _f64(k), _f64(v), _f64(W), _f64(c)
    g = None if gamma is None else _f64(gamma)
    b = None if beta is None else _f64(beta)
    gW, gc = np.empty_like(W), np.empty_like(c)
    _load().oracle_linear_token_grad_v(_p(k), _p(v), _p(W), _p(c), k.size, int(ln),
                                       _loss_id(loss), _p(g), _p(b), eps, _p(gW), _p(gc))
    return gW, gc


def mlp_token_loss(k, v, W1, b1, W2, b2, ln=False, gamma=None, beta=None, eps=1e-6, loss="mse"):
    k, v, W1, b1, W2, b2 = map(_f64, (k, v, W1, b1, W2, b2))
    g = None if gamma is None else _f64(gamma)
    b = None if beta is None else _f64(beta)
    return _load().oracle_mlp_token_loss_v(_p(k), _p(v), _p(W1), _p(b1), _p(W2), _p(b2),
                                           k.size, b1.size, int(ln), _loss_id(loss), _p(g),
                                           _p(b), eps)


def mlp_token_grad(k, v, W1, b1, W2, b2, ln=False, gamma=None, beta=None, eps=1e-6, loss="mse"):
    k, v, W1, b1, W2, b2 = map(_f64, (k, v, W1, b1, W2, b2))
    g = None if gamma is None else _f64(gamma)
    b = None if beta is None else _f64(beta)
    gW1, gb1, gW2, gb2 = (np.empty_like(a) for a in (W1, b1, W2, b2))
    _load().oracle_mlp_token_grad_v(_p(k), _p(v), _p(W1), _p(b1), _p(W2), _p(b2), k.size,
                                    b1.size, int(ln), _loss_id(loss), _p(g), _p(b), eps,
                                    _p(gW1), _p(gb1), _p(gW2), _p(gb2))
    return gW1, gb1, gW2, gb2


# --------------------------------------------------------------------------
# full forward passes
# --------------------------------------------------------------------------

def ttt_linear(Q, K, V, eta, W0, b0, gamma=None, beta=None, *, mini_batch: int,
               ln: bool, eps: float = 1e-6, init_per_batch: bool = False,
               dual: bool = False, loss: str = "mse", weight_decay: float = 0.0):
    """TTT-Linear forward.  Q,K,V: [B,H,L,d]; eta: [B,H,L]; W0: [H,d,d] (or
    [B,H,d,d] if init_per_batch); b0: [H,d] (or [B,H,d]); gamma/beta: [H,d].
    loss: "mse" (1/2 ||f(k) - v||^2) or "ip" (-<f(k), v>); weight_decay lambda on W.
    Returns (Z [B,H,L,d], W_final [B,H,d,d], b_final [B,H,d]) in float64."""
    Q, K, V, eta, W0, b0 = map(_f64, (Q, K, V, eta, W0, b0))
    B, H, L, d = Q.shape
    g = _f64(gamma) if ln else None
    b = _f64(beta) if ln else None
    Z = np.empty((B, H, L, d))
    Wf = np.empty((B, H, d, d))
    bf = np.empty((B, H, d))
    fn = _load().oracle_ttt_linear_dual_v if dual else _load().oracle_ttt_linear_v
    rc = fn(B, H, L, d, int(mini_batch), int(ln), float(eps), int(init_per_batch),
            _loss_id(loss), float(weight_decay),
            _p(Q), _p(K), _p(V), _p(eta), _p(W0), _p(b0), _p(g), _p(b), _p(Z), _p(Wf), _p(bf))
    if rc != 0:
        raise ValueError(f"oracle_ttt_linear returned {rc}")
    return Z, Wf, bf


def ttt_mlp(Q, K, V, eta, W1, b1, W2, b2, gamma=None, beta=None, *, mini_batch: int,
            ln: bool, eps: float = 1e-6, init_per_batch: bool = False, dual: bool = False,
            loss: str = "mse", weight_decay: float = 0.0):
    """TTT-MLP forward.  W1: [H,d,dh], b1: [H,dh], W2: [H,dh,d], b2: [H,d] (or with
    a leading B if init_per_batch); loss and weight_decay as for ttt_linear.
    Returns (Z, W1_f, b1_f, W2_f, b2_f)."""
    Q, K, V, eta, W1, b1, W2, b2 = map(_f64, (Q, K, V, eta, W1, b1, W2, b2))
    B, H, L, d = Q.shape
    dh = b1.shape[-1]
    g = _f64(gamma) if ln else None
    b = _f64(beta) if ln else None
    Z = np.empty((B, H, L, d))
    W1f = np.empty((B, H, d, dh))
    b1f = np.empty((B, H, dh))
    W2f = np.empty((B, H, dh, d))
    b2f = np.empty((B, H, d))
    fn = _load().oracle_ttt_mlp_dual_v if dual else _load().oracle_ttt_mlp_v
    rc = fn(B, H, L, d, dh, int(mini_batch), int(ln), float(eps), int(init_per_batch),
            _loss_id(loss), float(weight_decay),
            _p(Q), _p(K), _p(V), _p(eta), _p(W1), _p(b1), _p(W2), _p(b2), _p(g), _p(b),
            _p(Z), _p(W1f), _p(b1f), _p(W2f), _p(b2f))
    if rc != 0:
        raise ValueError(f"oracle_ttt_mlp returned {rc}")
    return Z, W1f, b1f, W2f, b2f


def _pick_init(a, bi, hi, per_batch):
    return a[bi, hi][None, None] if per_batch else a[hi][None]


def run_pairs(kind: str, inputs: dict, pairs, threads: int = 1, **kw):
    """Run the oracle on a subset of (batch, head) pairs, one pair per call,
    spread over ``threads`` Python threads (ctypes releases the GIL, so the
    calls run on separate cores).  Returns {(bi, hi): outputs-tuple}.  The
    initial state must be head-shared (not per batch)."""
    def one(pair):
        bi, hi = pair
        sl = lambda a: a[bi:bi + 1, hi:hi + 1]
        if kind == "linear":
            out = ttt_linear(sl(inputs["Q"]), sl(inputs["K"]), sl(inputs["V"]),
                             sl(inputs["eta"]), inputs["W0"][hi:hi + 1],
                             inputs["b0"][hi:hi + 1],
                             None if inputs.get("gamma") is None else inputs["gamma"][hi:hi + 1],
                             None if inputs.get("beta") is None else inputs["beta"][hi:hi + 1],
                             **kw)
        else:
            out = ttt_mlp(sl(inputs["Q"]), sl(inputs["K"]), sl(inputs["V"]),
                          sl(inputs["eta"]), inputs["W1"][hi:hi + 1], inputs["b1"][hi:hi + 1],
                          inputs["W2"][hi:hi + 1], inputs["b2"][hi:hi + 1],
                          None if inputs.get("gamma") is None else inputs["gamma"][hi:hi + 1],
                          None if inputs.get("beta") is None else inputs["beta"][hi:hi + 1],
                          **kw)
        return pair, out

    pairs = list(pairs)
    if threads <= 1:
        return dict(one(p) for p in pairs)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return dict(ex.map(one, pairs))
