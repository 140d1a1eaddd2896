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
    """The inputs on the GPU.  When the workload gives the gate's inputs (x, theta,
    eta_base) instead of eta, eta is computed on the GPU by the library's gate."""
    io = torch.bfloat16 if cfg.io == "bf16" else torch.float32
    dev = {}
    for k, v in x.items():
        if v is None or k == "eta_base":
            dev[k] = v
        elif k in ("Q", "K", "V", "x"):
            dev[k] = torch.from_numpy(np.ascontiguousarray(v)).to(device).to(io).contiguous()
        else:
            dev[k] = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(device)
    if "eta" not in dev:
        dev["eta"] = ttt.ttt_eta_gate(dev["x"], dev["theta"], dev["eta_base"])
    return dev


def with_oracle_eta(x):
    """The inputs with eta for the oracle: given, or computed by the oracle's own gate."""
    if "eta" in x:
        return x
    y = dict(x)
    y["eta"] = oracle.eta_gate(x["x"], x["theta"], x["eta_base"])
    return y


def run_gpu(cfg, dev, stream=None, out=None, init_per_batch=False, **variant):
    """The CUDA path; ``variant`` is the inner learner's loss= and weight_decay=."""
    kw = dict(mini_batch=cfg.mini_batch, residual_ln=cfg.ln, ln_eps=cfg.eps,
              init_per_batch=init_per_batch, stream=stream, out=out, **variant)
    if cfg.kind == "linear":
        res = ttt.ttt_linear_fwd(dev["Q"], dev["K"], dev["V"], dev["eta"], dev["W0"], dev["b0"],
                                 dev["gamma"], dev["beta"], **kw)
    else:
        res = ttt.ttt_mlp_fwd(dev["Q"], dev["K"], dev["V"], dev["eta"], dev["W1"], dev["b1"],
                              dev["W2"], dev["b2"], dev["gamma"], dev["beta"], **kw)
    ttt.ttt_sync_status(stream)
    return [r.float().cpu().numpy().astype(np.float64) for r in res]


def run_oracle(cfg, x, pairs=None, threads=None, **variant):
    """Oracle outputs, either for everything or for a list of (batch, head)."""
    x = with_oracle_eta(x)
    kw = dict(mini_batch=cfg.mini_batch, ln=cfg.ln, eps=cfg.eps, **variant)
    if pairs is None:
        if cfg.kind == "linear":
            return oracle.ttt_linear(x["Q"], x["K"], x["V"], x["eta"], x["W0"], x["b0"],
                                     x["gamma"], x["beta"], **kw)
        return oracle.ttt_mlp(x["Q"], x["K"], x["V"], x["eta"], x["W1"], x["b1"], x["W2"],
                              x["b2"], x["gamma"], x["beta"], **kw)
    threads = threads or max(1, min(len(pairs), os.cpu_count() or 1))
    return oracle.run_pairs(cfg.kind, x, pairs, threads=threads, **kw)


# worst relative L2 error seen per (case, output), printed at the end of the session
# (conftest.py) and written to $TTT_PARITY_LOG when that is set
WORST = {}
TAIL_TOKENS = 64   # the last four mini-batches of a scan are checked on their own


def _record(case, what, err):
    key = (case, what)
    WORST[key] = max(WORST.get(key, 0.0), err)


def check_scan(case, what, got, ref, tol, seq_axis=None):
    """Relative L2 error of one (batch, head) slice, and of the last TAIL_TOKENS tokens along
    ``seq_axis`` on their own; both must be within ``tol``.  Returns the larger."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{case} {what}: non-finite values"
    errs = [rel_l2(got, ref)]
    if seq_axis is not None and got.shape[seq_axis] > TAIL_TOKENS:
        tail = [slice(None)] * got.ndim
        tail[seq_axis] = slice(-TAIL_TOKENS, None)
        errs.append(rel_l2(got[tuple(tail)], ref[tuple(tail)]))
        _record(case, what + " tail", errs[-1])
    _record(case, what, errs[0])
    assert max(errs) <= tol, f"{case} {what}: rel-L2 {errs} > {tol}"
    return max(errs)


OUT_NAMES = {"linear": ["Z", "W_final", "b_final"],
             "mlp": ["Z", "W1_final", "b1_final", "W2_final", "b2_final"]}


def current_case(default):
    """The running test's node id (pytest sets it in the environment)."""
    cur = os.environ.get("PYTEST_CURRENT_TEST")
    return cur.split(" ")[0].split("::", 1)[-1] if cur else default


def compare_all(cfg, got, ref, tol=None, case=None):
    """Every output of every (batch, head) within ``tol`` (Z also over its last
    TAIL_TOKENS tokens alone); outputs are [B, H, ...]."""
    tol = TOL[cfg.io] if tol is None else tol
    case = case or current_case(cfg.name)
    names = OUT_NAMES[cfg.kind]
    worst = 0.0
    for name, g, r in zip(names, got, ref):
        g = np.asarray(g)
        r = np.broadcast_to(np.asarray(r), g.shape)
        for bi in range(g.shape[0]):
            for hi in range(g.shape[1]):
                worst = max(worst, check_scan(case, name, g[bi, hi], r[bi, hi], tol,
                                              seq_axis=0 if name == "Z" else None))
    return worst


def compare_pairs(cfg, got, ref_pairs, tol=None, case=None):
    """Sampled (batch, head) scans of a full-size run against the oracle's scans."""
    tol = TOL[cfg.io] if tol is None else tol
    case = case or current_case(cfg.name)
    names = OUT_NAMES[cfg.kind]
    worst = 0.0
    for (bi, hi), ref in ref_pairs.items():
        for name, g, r in zip(names, got, ref):
            worst = max(worst, check_scan(case, name, g[bi, hi], r[0, 0], tol,
                                          seq_axis=0 if name == "Z" else None))
    return worst


def sample_pairs(cfg, n, seed=0):
    rng = np.random.default_rng(seed)
    allp = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    if n >= len(allp):
        return allp
    idx = rng.choice(len(allp), n, replace=False)
    return sorted(allp[i] for i in idx)


def inputs(cfg, seed=0):
    return make_inputs(cfg, seed)
