"""Python binding of libttt.so: the TTT inner loop on B300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/ttt.h``.  Torch tensors are
used for device memory and streams.  There is no CPU fallback: if the
library has not been built, or the GPU is missing, calls raise.

Functions mirror the C entry points:
    ttt_eta_gate(x, theta, eta_base) -> eta
    ttt_linear_fwd(Q, K, V, eta, W0, b0, gamma, beta, ...) -> (Z, W_final, b_final)
      (every entry point takes loss="mse"|"ip" and weight_decay=lambda)
    ttt_mlp_fwd(Q, K, V, eta, W1, b1, W2, b2, gamma, beta, ...) -> (Z, W1_f, b1_f, W2_f, b2_f)
    ttt_linear_step(Q, K, V, eta, W, b, gamma, beta, ...) -> Z   (decode, state in place)
    ttt_linear_bwd(Q, K, V, eta, W0, b0, dZ, dW_final, db_final, ...)
        -> (dQ, dK, dV, deta, dW0, db0)
    ttt_sync_status(stream=None)
    kernel_name(...)
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["TTTError", "Desc", "load", "library_path", "partition_rows", "ttt_eta_gate", "ttt_linear_fwd", "ttt_mlp_fwd", "ttt_linear_step",
           "ttt_linear_bwd", "ttt_linear_bwd_workspace_size", "ttt_linear_bwd_static",
           "ttt_qkv_proj", "ttt_sync_status", "kernel_name", "version", "STATUS", "set_wait_timeout_ns",
           "debug_withhold_loads"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libttt.so")
_lock = threading.Lock()
_lib = None

TTT_F32, TTT_BF16 = 0, 1
STATUS = {0: "TTT_OK", 1: "TTT_ERR_INVALID_ARG", 2: "TTT_ERR_UNSUPPORTED", 3: "TTT_ERR_CUDA",
          4: "TTT_ERR_TIMEOUT"}


class TTTError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int),
                ("d", ctypes.c_int), ("d_hidden", ctypes.c_int), ("mini_batch", ctypes.c_int),
                ("io_dtype", ctypes.c_int), ("residual_ln", ctypes.c_int),
                ("ln_eps", ctypes.c_float), ("init_per_batch", ctypes.c_int),
                ("bh_offset", ctypes.c_int), ("bh_count", ctypes.c_int),
                ("loss", ctypes.c_int), ("weight_decay", ctypes.c_float),
                ("status", ctypes.c_void_p)]   # optional per-call failure word (device pointer)

LOSSES = {"mse": 0, "ip": 1}   # 1/2 ||f(k) - v||^2, or the inner product -<f(k), v>


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libttt.so (built in place by ``build.py``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(f"libttt.so not built ({_LIB_PATH}); run "
                                  "`python -m test_sequence_layers_08_b300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, dp = ctypes.c_void_p, ctypes.POINTER(Desc)
            lib.ttt_linear_fwd.restype = ctypes.c_int
            lib.ttt_linear_fwd.argtypes = [dp] + [vp] * 12
            lib.ttt_linear_step.restype = ctypes.c_int
            lib.ttt_linear_step.argtypes = [dp] + [vp] * 10
            lib.ttt_mlp_fwd.restype = ctypes.c_int
            lib.ttt_mlp_fwd.argtypes = [dp] + [vp] * 16
            lib.ttt_linear_bwd.restype = ctypes.c_int
            lib.ttt_linear_bwd.argtypes = [dp] + [vp] * 20 + [ctypes.c_size_t, vp]
            lib.ttt_linear_bwd_static.restype = ctypes.c_int
            lib.ttt_linear_bwd_static.argtypes = [dp] + [vp] * 20
            lib.ttt_linear_bwd_static_scratch_bytes.restype = ctypes.c_size_t
            lib.ttt_linear_bwd_static_scratch_bytes.argtypes = []
            lib.ttt_linear_bwd_workspace_size.restype = ctypes.c_size_t
            lib.ttt_linear_bwd_workspace_size.argtypes = [dp]
            lib.ttt_eta_gate.restype = ctypes.c_int
            lib.ttt_eta_gate.argtypes = [ctypes.c_int] * 5 + [ctypes.c_float] + [vp] * 3 + [ctypes.c_int, vp]
            lib.ttt_qkv_proj.restype = ctypes.c_int
            lib.ttt_qkv_proj.argtypes = [ctypes.c_int] * 5 + [vp] * 5 + [ctypes.c_int, vp]
            lib.ttt_sync_status.restype = ctypes.c_int
            lib.ttt_sync_status.argtypes = [vp]
            lib.ttt_status_string.restype = ctypes.c_char_p
            lib.ttt_status_string.argtypes = [ctypes.c_int]
            lib.ttt_last_error.restype = ctypes.c_char_p
            lib.ttt_last_error.argtypes = []
            lib.ttt_kernel_name.restype = ctypes.c_char_p
            lib.ttt_kernel_name.argtypes = [dp, ctypes.c_int]
            lib.ttt_version.restype = ctypes.c_int
            lib.ttt_version.argtypes = []
            lib.ttt_set_wait_timeout_ns.restype = None
            lib.ttt_set_wait_timeout_ns.argtypes = [ctypes.c_longlong]
            lib.ttt_debug_withhold_loads.restype = None
            lib.ttt_debug_withhold_loads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def version() -> int:
    return load().ttt_version()


def _check(status: int):
    if status != 0:
        raise TTTError(status, load().ttt_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(Q, mini_batch: int, residual_ln: bool, ln_eps: float = 1e-6,
              init_per_batch: bool = False, d_hidden: int = 0, heads=None, bh_offset: int = 0,
              loss: str = "mse", weight_decay: float = 0.0, status=None) -> Desc:
    """Descriptor of a call on Q [B, H, L, d], or on the row form Q [rows, L, d] covering rows
    bh_offset .. bh_offset + rows - 1 of a (batch, head) grid with `heads` heads.  loss: "mse"
    or "ip" (inner product); weight_decay: lambda on the weight matrices; status: an int32
    CUDA tensor whose first element is the call's own failure word (None: the device-wide
    flag that ttt_sync_status reads)."""
    import torch
    io = {torch.float32: TTT_F32, torch.bfloat16: TTT_BF16}.get(Q.dtype)
    if io is None:
        raise TypeError(f"unsupported I/O dtype {Q.dtype}")
    lead, H, L, d, B, off, cnt = _geometry(Q, heads, bh_offset)
    if loss not in LOSSES:
        raise ValueError(f"loss must be one of {sorted(LOSSES)}")
    if status is not None:
        if not (isinstance(status, torch.Tensor) and status.dtype == torch.int32 and status.is_cuda
                and status.numel() >= 1 and status.device == Q.device):
            raise ValueError("status must be an int32 CUDA tensor on Q's device with >= 1 element")
    return Desc(B, H, L, d, d_hidden, mini_batch, io, int(residual_ln), float(ln_eps),
                int(init_per_batch), off, cnt, LOSSES[loss], float(weight_decay),
                None if status is None else status.data_ptr())


def partition_rows(total_rows: int, world: int, rank: int):
    """The contiguous range [r0, r1) of (batch, head) rows that rank `rank` of `world` owns:
    balanced (sizes differ by at most one), in rank order, covering 0 .. total_rows - 1."""
    if world <= 0 or not 0 <= rank < world or total_rows < 0:
        raise ValueError("need world > 0, 0 <= rank < world and total_rows >= 0")
    base, extra = divmod(total_rows, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def _geometry(Q, heads, bh_offset):
    """(row-indexed leading shape, H, L, d, descriptor B, bh_offset, bh_count) of a call:
    Q [B, H, L, d] (heads None), or the row form Q [rows, L, d] with `heads` = H."""
    import torch
    if not isinstance(Q, torch.Tensor):
        raise TypeError("Q must be a torch.Tensor")
    if heads is None:
        if Q.dim() != 4:
            raise ValueError("Q must be [B, H, L, d], or the row form [rows, L, d] with heads=H")
        if bh_offset:
            raise ValueError("bh_offset needs the row form Q [rows, L, d] with heads=H")
        B, H, L, d = Q.shape
        return (B, H), H, L, d, B, 0, 0
    if Q.dim() != 3:
        raise ValueError("with heads=H, Q must be the row form [rows, L, d]")
    rows, L, d = Q.shape
    H = int(heads)
    if H <= 0 or bh_offset < 0 or rows <= 0:
        raise ValueError("need heads > 0, bh_offset >= 0 and at least one row")
    B = -(-(bh_offset + rows) // H)
    return (rows,), H, L, d, B, int(bh_offset), rows


def kernel_name(desc: Desc, mlp: bool = False):
    n = load().ttt_kernel_name(ctypes.byref(desc), int(mlp))
    return None if n is None else n.decode()


def _expect(name, t, shape, dtype, device):
    """Raise unless ``t`` is a contiguous tensor of exactly ``shape``, ``dtype`` and ``device``.
    Shape is checked first, so a wrong shape is reported even for host tensors."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise TypeError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_sequence(Q, K, V, eta, gamma, beta, residual_ln, heads=None, bh_offset=0):
    """Shapes, dtypes, device and contiguity of the per-token inputs and the LayerNorm
    parameters; returns (row-indexed leading shape, H, L, d, device)."""
    import torch
    lead, H, L, d, _, _, _ = _geometry(Q, heads, bh_offset)
    if Q.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"unsupported I/O dtype {Q.dtype}")
    dev = Q.device
    _expect("Q", Q, lead + (L, d), Q.dtype, dev)
    _expect("K", K, lead + (L, d), Q.dtype, dev)
    _expect("V", V, lead + (L, d), Q.dtype, dev)
    _expect("eta", eta, lead + (L,), torch.float32, dev)
    if residual_ln:
        _expect("gamma", gamma, (H, d), torch.float32, dev)
        _expect("beta", beta, (H, d), torch.float32, dev)
    return lead, H, L, d, dev


def _require_cuda(dev):
    if dev.type != "cuda":
        raise TypeError(f"tensors must be on a CUDA device, got {dev}")


def ttt_linear_fwd(Q, K, V, eta, W0, b0, gamma=None, beta=None, *, mini_batch: int = 16,
                   residual_ln: bool = False, ln_eps: float = 1e-6, init_per_batch: bool = False,
                   out=None, stream=None, heads=None, bh_offset: int = 0, loss: str = "mse",
                   weight_decay: float = 0.0, status=None):
    """TTT-Linear forward on the GPU.  Q,K,V: [B,H,L,d] (float32 or bfloat16);
    eta [B,H,L] float32; W0 [H,d,d] (or [B,H,d,d] with init_per_batch); b0 [H,d]
    (or [B,H,d]); gamma, beta [H,d] float32 (residual LayerNorm only).  Returns
    (Z, W_final, b_final); pass ``out=(Z, W_final, b_final)`` to reuse buffers.
    Row form (a (batch, head) partition): with ``heads=H``, Q, K, V are [rows, L, d], eta
    [rows, L], the outputs [rows, ...], W0/b0 [H, ...] (or [rows, ...] with init_per_batch),
    and the rows are rows bh_offset .. bh_offset + rows - 1 of the B*H grid (row b*H + h).
    Every operand is checked (shape, dtype, device, contiguity) before the C call.
    ``status``: an int32 CUDA tensor; its first element receives this call's timeout flag
    instead of the device-wide one (clear it before, read it after synchronising).
    The call is asynchronous on ``stream`` (default: torch's current stream)."""
    import torch
    lead, H, L, d, dev = _check_sequence(Q, K, V, eta, gamma, beta, residual_ln, heads, bh_offset)
    init = lead if init_per_batch else (H,)
    _expect("W0", W0, init + (d, d), torch.float32, dev)
    _expect("b0", b0, init + (d,), torch.float32, dev)
    if out is not None:
        Z, Wf, bf = out
        _expect("out Z", Z, lead + (L, d), Q.dtype, dev)
        _expect("out W_final", Wf, lead + (d, d), torch.float32, dev)
        _expect("out b_final", bf, lead + (d,), torch.float32, dev)
    _require_cuda(dev)
    lib = load()
    desc = make_desc(Q, mini_batch, residual_ln, ln_eps, init_per_batch, heads=heads,
                     bh_offset=bh_offset, loss=loss, weight_decay=weight_decay, status=status)
    if out is None:
        out = (torch.empty_like(Q), torch.empty(lead + (d, d), device=dev, dtype=torch.float32),
               torch.empty(lead + (d,), device=dev, dtype=torch.float32))
    Z, Wf, bf = out
    _check(lib.ttt_linear_fwd(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(eta),
                              _ptr(W0), _ptr(b0), _ptr(gamma if residual_ln else None),
                              _ptr(beta if residual_ln else None), _ptr(Z), _ptr(Wf), _ptr(bf),
                              _stream_handle(stream)))
    return Z, Wf, bf


def ttt_linear_bwd_workspace_size(Q, *, mini_batch: int = 16, init_per_batch: bool = False,
                                  heads=None, bh_offset: int = 0, loss: str = "mse",
                                  residual_ln: bool = False, ln_eps: float = 1e-6,
                                  weight_decay: float = 0.0) -> int:
    """Bytes of device workspace ttt_linear_bwd needs for inputs shaped like Q (0 when the
    shape is not supported)."""
    desc = make_desc(Q, mini_batch, residual_ln, ln_eps, init_per_batch, heads=heads,
                     bh_offset=bh_offset, loss=loss, weight_decay=weight_decay)
    return int(load().ttt_linear_bwd_workspace_size(ctypes.byref(desc)))


def _bwd_outputs(Q, K, V, eta, W0, b0, gamma, residual_ln):
    import torch
    o = (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V), torch.empty_like(eta),
         torch.empty_like(W0), torch.empty_like(b0))
    return o + ((torch.empty_like(gamma), torch.empty_like(gamma)) if residual_ln else ())


def _bwd_check(Q, K, V, eta, W0, b0, gamma, beta, dZ, dW_final, db_final, out, residual_ln,
               init_per_batch, heads, bh_offset):
    import torch
    lead, H, L, d, dev = _check_sequence(Q, K, V, eta, gamma, beta, residual_ln, heads, bh_offset)
    init = lead if init_per_batch else (H,)
    _expect("W0", W0, init + (d, d), torch.float32, dev)
    _expect("b0", b0, init + (d,), torch.float32, dev)
    _expect("dZ", dZ, lead + (L, d), Q.dtype, dev)
    if dW_final is not None:
        _expect("dW_final", dW_final, lead + (d, d), torch.float32, dev)
    if db_final is not None:
        _expect("db_final", db_final, lead + (d,), torch.float32, dev)
    if out is not None:
        refs = (Q, K, V, eta, W0, b0) + ((gamma, beta) if residual_ln else ())
        names = ("dQ", "dK", "dV", "deta", "dW0", "db0", "dgamma", "dbeta")
        if len(out) != len(refs):
            raise ValueError(f"out must hold {len(refs)} tensors")
        for name, t, ref in zip(names, out, refs):
            _expect("out " + name, t, tuple(ref.shape), ref.dtype, dev)
    _require_cuda(dev)
    return dev


def ttt_linear_bwd(Q, K, V, eta, W0, b0, dZ, dW_final=None, db_final=None, gamma=None, beta=None,
                   *, mini_batch: int = 16, residual_ln: bool = False, ln_eps: float = 1e-6,
                   init_per_batch: bool = False, loss: str = "mse", weight_decay: float = 0.0,
                   out=None, workspace=None, stream=None, heads=None, bh_offset: int = 0):
    """TTT-Linear backward on the GPU: the gradients of
    F = <Z, dZ> + <W_final, dW_final> + <b_final, db_final> for the forward
    ttt_linear_fwd(Q, K, V, eta, W0, b0, gamma, beta, ...).  Returns (dQ, dK, dV, deta, dW0,
    db0), plus (dgamma, dbeta) with the residual LayerNorm; dW0, db0 are shaped like W0, b0.
    ``workspace``: a uint8 CUDA tensor of at least ttt_linear_bwd_workspace_size(...) bytes
    (allocated here when None).  ``out`` reuses output buffers.  Row form as for
    ttt_linear_fwd.  Asynchronous on ``stream``."""
    import torch
    dev = _bwd_check(Q, K, V, eta, W0, b0, gamma, beta, dZ, dW_final, db_final, out, residual_ln,
                     init_per_batch, heads, bh_offset)
    lib = load()
    desc = make_desc(Q, mini_batch, residual_ln, ln_eps, init_per_batch, heads=heads,
                     bh_offset=bh_offset, loss=loss, weight_decay=weight_decay)
    need = int(lib.ttt_linear_bwd_workspace_size(ctypes.byref(desc)))
    if need == 0:
        raise TTTError(2, "ttt_linear_bwd: shape not supported")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _expect("workspace", workspace, (workspace.numel(),), torch.uint8, dev)
    if out is None:
        out = _bwd_outputs(Q, K, V, eta, W0, b0, gamma, residual_ln)
    dgam, dbet = (out[6], out[7]) if residual_ln else (None, None)
    _check(lib.ttt_linear_bwd(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(eta), _ptr(W0),
                              _ptr(b0), _ptr(gamma if residual_ln else None),
                              _ptr(beta if residual_ln else None), _ptr(dZ), _ptr(dW_final),
                              _ptr(db_final), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), _ptr(out[3]),
                              _ptr(out[4]), _ptr(out[5]), _ptr(dgam), _ptr(dbet), _ptr(workspace),
                              ctypes.c_size_t(workspace.numel()), _stream_handle(stream)))
    return tuple(out)


def ttt_linear_bwd_static(Q, K, V, eta, W0, b0, dZ, dW_final=None, db_final=None, gamma=None,
                          beta=None, *, out, mini_batch: int = 16, residual_ln: bool = False,
                          ln_eps: float = 1e-6, init_per_batch: bool = False, loss: str = "mse",
                          weight_decay: float = 0.0, stream=None, heads=None, bh_offset: int = 0):
    """ttt_linear_bwd on the library's static device scratch: allocates nothing, so the
    output buffers ``out=(dQ, dK, dV, deta, dW0, db0[, dgamma, dbeta])`` are required.  Calls
    on one device share the scratch and must not overlap in time.  Returns ``out``."""
    _bwd_check(Q, K, V, eta, W0, b0, gamma, beta, dZ, dW_final, db_final, out, residual_ln,
               init_per_batch, heads, bh_offset)
    lib = load()
    desc = make_desc(Q, mini_batch, residual_ln, ln_eps, init_per_batch, heads=heads,
                     bh_offset=bh_offset, loss=loss, weight_decay=weight_decay)
    dgam, dbet = (out[6], out[7]) if residual_ln else (None, None)
    _check(lib.ttt_linear_bwd_static(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(eta),
                                     _ptr(W0), _ptr(b0), _ptr(gamma if residual_ln else None),
                                     _ptr(beta if residual_ln else None), _ptr(dZ), _ptr(dW_final),
                                     _ptr(db_final), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                     _ptr(out[3]), _ptr(out[4]), _ptr(out[5]), _ptr(dgam), _ptr(dbet),
                                     _stream_handle(stream)))
    return out


def ttt_linear_step(Q, K, V, eta, W, b, gamma=None, beta=None, *, residual_ln: bool = False,
                    ln_eps: float = 1e-6, out=None, stream=None, heads=None, bh_offset: int = 0,
                    loss: str = "mse", weight_decay: float = 0.0):
    """TTT-Linear decode on the GPU: the L tokens of Q, K, V [B,H,L,d] one at a time from
    the state W [B,H,d,d], b [B,H,d] (float32), which is updated in place.  Returns Z
    [B,H,L,d]; pass ``out=Z`` to reuse a buffer.  Row form as for ttt_linear_fwd (the state
    is then [rows, d, d] and [rows, d]).  Asynchronous on ``stream``."""
    import torch
    lead, H, L, d, dev = _check_sequence(Q, K, V, eta, gamma, beta, residual_ln, heads, bh_offset)
    _expect("W", W, lead + (d, d), torch.float32, dev)
    _expect("b", b, lead + (d,), torch.float32, dev)
    if out is not None:
        _expect("out Z", out, lead + (L, d), Q.dtype, dev)
    _require_cuda(dev)
    lib = load()
    desc = make_desc(Q, 1, residual_ln, ln_eps, True, heads=heads, bh_offset=bh_offset, loss=loss,
                     weight_decay=weight_decay)
    Z = torch.empty_like(Q) if out is None else out
    _check(lib.ttt_linear_step(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(eta), _ptr(W),
                               _ptr(b), _ptr(gamma if residual_ln else None),
                               _ptr(beta if residual_ln else None), _ptr(Z), _stream_handle(stream)))
    return Z


def ttt_mlp_fwd(Q, K, V, eta, W1, b1, W2, b2, gamma=None, beta=None, *, mini_batch: int = 16,
                residual_ln: bool = False, ln_eps: float = 1e-6, init_per_batch: bool = False,
                out=None, stream=None, heads=None, bh_offset: int = 0, loss: str = "mse",
                weight_decay: float = 0.0, status=None):
    """TTT-MLP forward on the GPU.  W1 [H,d,dh], b1 [H,dh], W2 [H,dh,d], b2 [H,d]
    (leading B when init_per_batch).  Returns (Z, W1_f, b1_f, W2_f, b2_f).  Row form and
    ``status`` as for ttt_linear_fwd.  Every operand is checked before the C call."""
    import torch
    lead, H, L, d, dev = _check_sequence(Q, K, V, eta, gamma, beta, residual_ln, heads, bh_offset)
    if not isinstance(b1, torch.Tensor) or b1.dim() < 1:
        raise ValueError("b1 must be a [H, dh] (or [B, H, dh]) tensor")
    dh = b1.shape[-1]
    init = lead if init_per_batch else (H,)
    _expect("W1", W1, init + (d, dh), torch.float32, dev)
    _expect("b1", b1, init + (dh,), torch.float32, dev)
    _expect("W2", W2, init + (dh, d), torch.float32, dev)
    _expect("b2", b2, init + (d,), torch.float32, dev)
    if out is not None:
        Z, W1f, b1f, W2f, b2f = out
        _expect("out Z", Z, lead + (L, d), Q.dtype, dev)
        _expect("out W1_f", W1f, lead + (d, dh), torch.float32, dev)
        _expect("out b1_f", b1f, lead + (dh,), torch.float32, dev)
        _expect("out W2_f", W2f, lead + (dh, d), torch.float32, dev)
        _expect("out b2_f", b2f, lead + (d,), torch.float32, dev)
    _require_cuda(dev)
    lib = load()
    desc = make_desc(Q, mini_batch, residual_ln, ln_eps, init_per_batch, d_hidden=dh, heads=heads,
                     bh_offset=bh_offset, loss=loss, weight_decay=weight_decay, status=status)
    if out is None:
        f32 = dict(device=dev, dtype=torch.float32)
        out = (torch.empty_like(Q), torch.empty(lead + (d, dh), **f32), torch.empty(lead + (dh,), **f32),
               torch.empty(lead + (dh, d), **f32), torch.empty(lead + (d,), **f32))
    Z, W1f, b1f, W2f, b2f = out
    _check(lib.ttt_mlp_fwd(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(eta), _ptr(W1),
                           _ptr(b1), _ptr(W2), _ptr(b2), _ptr(gamma if residual_ln else None),
                           _ptr(beta if residual_ln else None), _ptr(Z), _ptr(W1f), _ptr(b1f),
                           _ptr(W2f), _ptr(b2f), _stream_handle(stream)))
    return Z, W1f, b1f, W2f, b2f


def ttt_eta_gate(x, theta, eta_base: float, *, out=None, stream=None, max_sms: int = 0):
    """Per-token learning rate on the GPU: eta [B,H,L] = eta_base * sigmoid(theta[h] . x[b,t])
    for the layer input x [B,L,d_model] (float32 or bfloat16) and theta [H,d_model] float32.
    Pass ``out=eta`` to reuse a buffer.  Asynchronous on ``stream``; ``max_sms`` > 0 caps the
    grid at that many SMs (for a call beside a scan that holds the others)."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dim() != 3:
        raise ValueError("x must be a [B, L, d_model] tensor")
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"unsupported token dtype {x.dtype}")
    B, L, Dx = x.shape
    dev = x.device
    _expect("x", x, (B, L, Dx), x.dtype, dev)
    if not isinstance(theta, torch.Tensor) or theta.dim() != 2:
        raise ValueError("theta must be a [H, d_model] tensor")
    H = theta.shape[0]
    _expect("theta", theta, (H, Dx), torch.float32, dev)
    if out is not None:
        _expect("out eta", out, (B, H, L), torch.float32, dev)
    _require_cuda(dev)
    lib = load()
    eta = torch.empty((B, H, L), device=dev, dtype=torch.float32) if out is None else out
    io = TTT_BF16 if x.dtype == torch.bfloat16 else TTT_F32
    _check(lib.ttt_eta_gate(B, H, L, Dx, io, float(eta_base), _ptr(x), _ptr(theta), _ptr(eta),
                            int(max_sms), _stream_handle(stream)))
    return eta


def ttt_qkv_proj(x, W, heads: int, d: int = 64, *, out=None, stream=None, max_sms: int = 0):
    """The layer's input projections on the GPU (tcgen05): x [B, L, d_model] bfloat16 and the
    stacked projection matrices W [3 heads d, d_model] bfloat16 (one row per output unit, as
    a linear layer stores its weight) give (Q, K, V), each [B, heads, L, d] bfloat16, the
    layout the scan reads.  Pass ``out=(Q, K, V)`` to reuse buffers.  Asynchronous on
    ``stream``; ``max_sms`` > 0 caps the persistent grid at that many SMs."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dim() != 3:
        raise ValueError("x must be a [B, L, d_model] tensor")
    B, L, Dx = x.shape
    dev = x.device
    _expect("x", x, (B, L, Dx), torch.bfloat16, dev)
    _expect("W", W, (3 * heads * d, Dx), torch.bfloat16, dev)
    shape = (B, heads, L, d)
    if out is not None:
        if len(out) != 3:
            raise ValueError("out must hold (Q, K, V)")
        for name, t in zip("QKV", out):
            _expect("out " + name, t, shape, torch.bfloat16, dev)
    _require_cuda(dev)
    lib = load()
    Q, K, V = out if out is not None else tuple(torch.empty(shape, device=dev, dtype=torch.bfloat16)
                                                for _ in range(3))
    _check(lib.ttt_qkv_proj(B, heads, L, Dx, d, _ptr(x), _ptr(W), _ptr(Q), _ptr(K), _ptr(V),
                            int(max_sms), _stream_handle(stream)))
    return Q, K, V


def set_wait_timeout_ns(ns: int):
    """Bound (ns) of every mbarrier wait in the fused kernels; <= 0 restores 1 s."""
    load().ttt_set_wait_timeout_ns(int(ns))


def debug_withhold_loads(on: bool):
    """Test hook: the fused kernels issue no stage copies, so their waits run out
    and the next ttt_sync_status reports TTT_ERR_TIMEOUT."""
    load().ttt_debug_withhold_loads(int(bool(on)))


def ttt_sync_status(stream=None):
    """Synchronise the stream; raise TTTError on a pending CUDA error or a
    device-side bounded-wait timeout."""
    _check(load().ttt_sync_status(_stream_handle(stream)))
