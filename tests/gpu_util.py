"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
CUDA path through the C ABI, run the oracle on the same inputs, compare."""
import os

import numpy as np
import torch

import oracle
import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300.inputs import make_inputs

TOL = {"f32": 1e-5, "bf16": 2e-2}   # relative L2 error bounds


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def to_device(cfg, x, device="cuda:0"):
    io = torch.bfloat16 if cfg.io == "bf16" else torch.float32
    dev = {}
    for k, v in x.items():
        if v is None:
            dev[k] = None
        elif k in ("Q", "K", "V"):
            dev[k] = torch.from_numpy(v).to(device).to(io).contiguous()
        else:
            dev[k] = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(device)
    return dev


def run_gpu(cfg, dev, stream=None, out=None, init_per_batch=False):
    kw = dict(mini_batch=cfg.mini_batch, residual_ln=cfg.ln, ln_eps=cfg.eps,
              init_per_batch=init_per_batch, stream=stream, out=out)
    if cfg.kind == "linear":
        res = ttt.ttt_linear_fwd(dev["Q"], dev["K"], dev["V"], dev["eta"], dev["W0"], dev["b0"],
                                 dev["gamma"], dev["beta"], **kw)
    else:
        res = ttt.ttt_mlp_fwd(dev["Q"], dev["K"], dev["V"], dev["eta"], dev["W1"], dev["b1"],
                              dev["W2"], dev["b2"], dev["gamma"], dev["beta"], **kw)
    ttt.ttt_sync_status(stream)
    return [r.float().cpu().numpy().astype(np.float64) for r in res]


def run_oracle(cfg, x, pairs=None, threads=None):
    """Oracle outputs, either for everything or for a list of (batch, head)."""
    kw = dict(mini_batch=cfg.mini_batch, ln=cfg.ln, eps=cfg.eps)
    if pairs is None:
        if cfg.kind == "linear":
            return oracle.ttt_linear(x["Q"], x["K"], x["V"], x["eta"], x["W0"], x["b0"],
                                     x["gamma"], x["beta"], **kw)
        return oracle.ttt_mlp(x["Q"], x["K"], x["V"], x["eta"], x["W1"], x["b1"], x["W2"],
                              x["b2"], x["gamma"], x["beta"], **kw)
    threads = threads or max(1, min(len(pairs), os.cpu_count() or 1))
    return oracle.run_pairs(cfg.kind, x, pairs, threads=threads, **kw)


def compare_all(cfg, got, ref, tol=None):
    tol = TOL[cfg.io] if tol is None else tol
    errs = [rel_l2(g, r) for g, r in zip(got, ref)]
    assert all(np.isfinite(g).all() for g in got)
    assert max(errs) <= tol, f"{cfg.name}: rel-L2 errors {errs} > {tol}"
    return errs


def compare_pairs(cfg, got, ref_pairs, tol=None):
    tol = TOL[cfg.io] if tol is None else tol
    errs = []
    for (bi, hi), ref in ref_pairs.items():
        for g, r in zip(got, ref):
            errs.append(rel_l2(g[bi, hi], r[0, 0]))
    assert all(np.isfinite(g).all() for g in got)
    assert max(errs) <= tol, f"{cfg.name}: rel-L2 errors {max(errs)} > {tol}"
    return errs


def sample_pairs(cfg, n, seed=0):
    rng = np.random.default_rng(seed)
    allp = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    if n >= len(allp):
        return allp
    idx = rng.choice(len(allp), n, replace=False)
    return sorted(allp[i] for i in idx)


def inputs(cfg, seed=0):
    return make_inputs(cfg, seed)
