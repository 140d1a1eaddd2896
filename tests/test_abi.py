"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, names its status codes, and rejects bad arguments before any
CUDA call is made."""
import ctypes
import os
import re

import pytest

import test_sequence_layers_08_b300 as ttt
from test_sequence_layers_08_b300 import build as ttt_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# names of the tensor-core TTT-Linear kernels the library may pick for bf16, d = 64, b = 16
LINEAR_TC_KERNELS = ("ttt_linear_fused", "ttt_linear_chunked")


@pytest.fixture(scope="module")
def lib():
    ttt_build.build()
    return ttt.load()


def header_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^TTT_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("ttt_linear_fwd", "ttt_mlp_fwd", "ttt_sync_status", "ttt_status_string",
              "ttt_last_error", "ttt_kernel_name", "ttt_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in header_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in ttt.STATUS.items():
        assert lib.ttt_status_string(code).decode() == name
    assert lib.ttt_version() >= 100


def desc(**kw):
    base = dict(B=2, H=3, L=64, d=64, d_hidden=0, mini_batch=16, io_dtype=1, residual_ln=0,
                ln_eps=1e-6, init_per_batch=0)
    base.update(kw)
    return ttt.Desc(**base)


FAKE = 1 << 20   # an aligned address; validation never dereferences pointers


def call_linear(lib, dsc, ptrs=None):
    p = [FAKE + i * (1 << 30) for i in range(11)] if ptrs is None else ptrs
    return lib.ttt_linear_fwd(ctypes.byref(dsc), *[ctypes.c_void_p(x) if x else None for x in p],
                              None)


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=-1), dict(L=0), dict(d=0), dict(mini_batch=0),
                                dict(L=40), dict(io_dtype=7), dict(residual_ln=2),
                                dict(init_per_batch=3), dict(residual_ln=1, ln_eps=-1.0),
                                dict(residual_ln=1, ln_eps=0.0), dict(residual_ln=1, ln_eps=float('nan')),
                                dict(bh_offset=-1, bh_count=2), dict(bh_count=-3),
                                dict(bh_offset=2), dict(bh_offset=4, bh_count=3),
                                dict(B=1, H=3, bh_offset=0, bh_count=4),
                                dict(loss=2), dict(loss=-1), dict(weight_decay=-0.5),
                                dict(weight_decay=float('nan')), dict(weight_decay=float('inf'))])
def test_bad_descriptor_is_invalid_arg(lib, kw):
    assert call_linear(lib, desc(**kw)) == 1
    assert lib.ttt_last_error().decode() != ""
    assert lib.ttt_kernel_name(ctypes.byref(desc(**kw)), 0) is None


def test_null_and_misaligned_pointers(lib):
    base = [FAKE + i * (1 << 30) for i in range(11)]
    for i in (0, 1, 2, 3, 4, 5, 8, 9, 10):
        p = list(base)
        p[i] = 0
        assert call_linear(lib, desc(), p) == 1
        p[i] = base[i] + 4
        assert call_linear(lib, desc(), p) == 1
    # gamma / beta only required with the residual LayerNorm
    p = list(base)
    p[6] = 0
    assert call_linear(lib, desc(residual_ln=1), p) == 1


def test_aliasing_rules(lib):
    base = [FAKE + i * (1 << 30) for i in range(11)]
    p = list(base)
    p[8] = p[0]          # Z on top of Q
    assert call_linear(lib, desc(), p) == 1
    p = list(base)
    p[9] = p[4]          # W_final on W0 with a head-shared W0: shapes differ
    assert call_linear(lib, desc(), p) == 1
    assert "W_final" in lib.ttt_last_error().decode()


def test_kernel_choice(lib):
    k = lambda **kw: (lambda n: n and n.decode())(lib.ttt_kernel_name(ctypes.byref(desc(**kw)), 0))
    assert k() in LINEAR_TC_KERNELS
    assert k(residual_ln=1) in LINEAR_TC_KERNELS
    # without LN, few (batch, head) rows: split by output column; with LN, or with more rows
    # than two CTAs per SM hold at 16 columns each: one CTA per row
    assert k(io_dtype=0) == "ttt_linear_cols"
    assert k(d=32) == "ttt_linear_cols"
    assert k(io_dtype=0, residual_ln=1) == "ttt_linear_generic"
    assert k(io_dtype=0, B=8, H=12) == "ttt_linear_generic"
    assert k(io_dtype=0, B=2, H=12) == "ttt_linear_cols"
    assert k(d=256) is None
    assert k(d=6, io_dtype=0) is None   # the generic kernel takes d a multiple of 4
    m = lambda **kw: (lambda n: n and n.decode())(lib.ttt_kernel_name(ctypes.byref(desc(**kw)), 1))
    assert m() == "ttt_mlp_fused"                    # d_hidden 0 -> 4 d = 256
    assert m(residual_ln=1, d_hidden=256) == "ttt_mlp_fused"
    assert m(io_dtype=0) == "ttt_mlp_generic"
    assert m(d_hidden=128) == "ttt_mlp_generic"
    assert m(d_hidden=4096) is None


def call_step(lib, dsc, ptrs=None):
    p = [FAKE + i * (1 << 30) for i in range(9)] if ptrs is None else ptrs
    return lib.ttt_linear_step(ctypes.byref(dsc), *[ctypes.c_void_p(x) if x else None for x in p],
                               None)


def test_step_declared_and_checked(lib):
    assert "ttt_linear_step" in header_functions()
    # the decode step is the mini-batch-1 recurrence: any other mini_batch is rejected
    assert call_step(lib, desc(mini_batch=16)) == 1
    assert "mini_batch" in lib.ttt_last_error().decode()
    assert call_step(lib, desc(mini_batch=1, L=0)) == 1
    base = [FAKE + i * (1 << 30) for i in range(9)]
    for i in (0, 1, 2, 3, 4, 5, 8):            # Q K V eta W b Z
        p = list(base)
        p[i] = 0
        assert call_step(lib, desc(mini_batch=1), p) == 1
        p[i] = base[i] + 8
        assert call_step(lib, desc(mini_batch=1), p) == 1
    p = list(base)
    p[6] = 0                                   # gamma needed with the residual LayerNorm
    assert call_step(lib, desc(mini_batch=1, residual_ln=1), p) == 1


def test_step_aliasing_rules(lib):
    base = [FAKE + i * (1 << 30) for i in range(9)]
    for i, j in ((8, 0), (4, 2), (5, 4), (4, 8)):   # Z on Q, W on V, b on W, W on Z
        p = list(base)
        p[i] = p[j]
        assert call_step(lib, desc(mini_batch=1), p) == 1, (i, j)
    assert call_step(lib, desc(mini_batch=1, d=256)) == 2   # no kernel for that width



def call_gate(lib, B=2, H=3, L=64, Dx=768, io=1, eta_base=0.5, ptrs=None, max_sms=0):
    p = [FAKE + i * (1 << 30) for i in range(3)] if ptrs is None else ptrs
    return lib.ttt_eta_gate(B, H, L, Dx, io, eta_base,
                            *[ctypes.c_void_p(x) if x else None for x in p], max_sms, None)


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(L=-1), dict(Dx=0), dict(io=5),
                                dict(Dx=20), dict(eta_base=float("inf")), dict(max_sms=-1)])
def test_gate_bad_arguments(lib, kw):
    assert call_gate(lib, **kw) == 1
    assert lib.ttt_last_error().decode() != ""


def test_gate_null_misaligned_and_overlap(lib):
    base = [FAKE + i * (1 << 30) for i in range(3)]
    for i in range(3):
        p = list(base)
        p[i] = 0
        assert call_gate(lib, ptrs=p) == 1
        p[i] = base[i] + 8
        assert call_gate(lib, ptrs=p) == 1
    p = list(base)
    p[2] = base[0] + 4096            # eta inside x
    assert call_gate(lib, ptrs=p) == 1
    assert "overlap" in lib.ttt_last_error().decode()


def test_descriptor_matches_the_header_struct():
    """The binding's Desc has the header's ttt_desc fields in order, ending with the per-call
    status pointer (8-byte aligned after the fourteen 4-byte fields)."""
    import re
    text = open(os.path.join(ROOT, "include", "ttt.h")).read()
    body = re.search(r"typedef struct \{(.*?)\} ttt_desc;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"(\w+);", body)
    assert names == [f[0] for f in ttt.Desc._fields_]
    assert ctypes.sizeof(ttt.Desc) == 64 and ttt.Desc.status.offset == 56


def test_status_word_must_be_aligned(lib):
    assert call_linear(lib, desc(status=FAKE + 2)) == 1
    assert "status" in lib.ttt_last_error().decode()
    assert lib.ttt_kernel_name(ctypes.byref(desc(status=FAKE)), 0) is not None


def test_partition_fields_accepted(lib):
    """A call on rows [2, 6) of a 2 x 3 grid passes the descriptor checks (the kernel choice
    does not depend on the partition)."""
    d = desc(bh_offset=2, bh_count=4)
    assert lib.ttt_kernel_name(ctypes.byref(d), 0) is not None


def test_variant_kernel_choice(lib):
    """The tensor-core kernels run both inner-learner variants: for TTT-Linear the chunked
    kernel without the residual LayerNorm and the fused one with it; for TTT-MLP the tcgen05
    kernel (on request) the inner-product loss, the warp-MMA kernel both."""
    k = lambda mlp, **kw: (lambda n: n and n.decode())(lib.ttt_kernel_name(ctypes.byref(desc(**kw)), mlp))
    for var in (dict(loss=1), dict(weight_decay=0.1), dict(loss=1, weight_decay=0.1)):
        assert k(0, **var) == "ttt_linear_chunked"
        assert k(0, residual_ln=1, **var) == "ttt_linear_fused"
        assert k(1, **var) == "ttt_mlp_fused"
        assert k(1, residual_ln=1, d_hidden=256, **var) == "ttt_mlp_fused"


# ttt_linear_bwd pointer slots: Q K V eta W0 b0 gamma beta dZ dW_final db_final dQ dK dV deta
# dW0 db0 dgamma dbeta workspace
BWD_SLOTS = 20
BWD_WS, BWD_DQ = 19, 11
BWD_OPTIONAL = (9, 10)               # dW_final, db_final: NULL means zero
BWD_LN_ONLY = (6, 7, 17, 18)         # gamma, beta, dgamma, dbeta: NULL allowed without LN


def bwd_ptrs():
    return [FAKE + i * (1 << 30) for i in range(BWD_SLOTS)]


def call_bwd(lib, dsc, ptrs=None, ws_bytes=1 << 30):
    """Every call here must fail the host checks: the pointers are fake."""
    p = bwd_ptrs() if ptrs is None else ptrs
    args = [ctypes.c_void_p(x) if x else None for x in p]
    return lib.ttt_linear_bwd(ctypes.byref(dsc), *args, ctypes.c_size_t(ws_bytes),
                              ctypes.c_void_p(FAKE + 31 * (1 << 30)))


def test_backward_declared_and_checked(lib):
    """ttt_linear_bwd: supported shapes report a workspace size; a head dim that is no multiple
    of 4 is unsupported; a short or misaligned workspace, a NULL or overlapping buffer are
    invalid arguments (all rejected before any launch)."""
    assert "ttt_linear_bwd" in header_functions()
    assert "ttt_linear_bwd_workspace_size" in header_functions()
    ws = lib.ttt_linear_bwd_workspace_size
    assert ws(ctypes.byref(desc())) > 0 and ws(ctypes.byref(desc())) % 256 == 0
    assert ws(ctypes.byref(desc(residual_ln=1))) > ws(ctypes.byref(desc()))   # + dgamma/dbeta partials
    assert ws(ctypes.byref(desc(weight_decay=0.1))) > 0
    assert ws(ctypes.byref(desc(d=6))) == 0
    assert ws(ctypes.byref(desc(L=40))) == 0      # invalid descriptor
    # per-batch initial state needs no per-row partials: a smaller workspace
    assert ws(ctypes.byref(desc(init_per_batch=1))) < ws(ctypes.byref(desc()))
    assert call_bwd(lib, desc(d=6, io_dtype=0)) == 2   # d not a multiple of 4: no kernel
    need = ws(ctypes.byref(desc()))
    assert call_bwd(lib, desc(), ws_bytes=need - 256) == 1
    p = bwd_ptrs()
    p[BWD_WS] += 16                               # workspace not 256-byte aligned
    assert call_bwd(lib, desc(), p) == 1
    for i in range(BWD_SLOTS):                    # every required pointer
        if i in BWD_OPTIONAL or i in BWD_LN_ONLY:
            continue
        q = bwd_ptrs()
        q[i] = 0
        assert call_bwd(lib, desc(), q) == 1, i
    for i in BWD_LN_ONLY:                         # required with the residual LayerNorm
        q = bwd_ptrs()
        q[i] = 0
        assert call_bwd(lib, desc(residual_ln=1), q) == 1, i
    q = bwd_ptrs()
    q[BWD_DQ] = q[0]                              # dQ on top of Q
    assert call_bwd(lib, desc(), q) == 1
    q = bwd_ptrs()
    q[BWD_WS] = q[BWD_DQ]                         # workspace on top of dQ
    assert call_bwd(lib, desc(), q) == 1
    q = bwd_ptrs()
    q[17] = q[6]                                  # dgamma on top of gamma
    assert call_bwd(lib, desc(residual_ln=1), q) == 1


def test_projection_declared_and_checked(lib):
    """ttt_qkv_proj: unsupported shapes, NULL, misaligned or overlapping buffers are rejected
    before any launch."""
    assert "ttt_qkv_proj" in header_functions()
    p = [FAKE + i * (1 << 30) for i in range(5)]   # x W Q K V
    call = lambda B=2, H=4, L=256, Dx=128, d=64, q=None, max_sms=0: lib.ttt_qkv_proj(
        B, H, L, Dx, d, *[ctypes.c_void_p(v) if v else None for v in (q or p)], max_sms, None)
    assert call(max_sms=-1) == 1                    # a negative SM cap
    assert call(d=32) == 2                          # d = 64 only
    assert call(Dx=96) == 2                         # d_model a multiple of 64
    assert call(H=3) == 2                           # 3 H d = 576: no multiple of 256
    assert call(B=0) == 1
    for i in range(5):
        q = list(p)
        q[i] = 0
        assert call(q=q) == 1, i
    q = list(p)
    q[2] += 8                                       # Q misaligned
    assert call(q=q) == 1
    q = list(p)
    q[3] = q[2]                                     # K on top of Q
    assert call(q=q) == 1
    q = list(p)
    q[4] = q[0]                                     # V on top of x
    assert call(q=q) == 1


def test_mlp_tmem_kernel_on_request(lib, monkeypatch):
    """TTT_MLP_KERNEL=tmem selects the tcgen05 TTT-MLP kernel where it applies (bf16, d = 64,
    d_hidden = 256, b = 16, no weight decay); anything else keeps the default choice."""
    m = lambda **kw: (lambda n: n and n.decode())(lib.ttt_kernel_name(ctypes.byref(desc(**kw)), 1))
    monkeypatch.setenv("TTT_MLP_KERNEL", "tmem")
    assert m() == "ttt_mlp_tmem"
    assert m(residual_ln=1, d_hidden=256) == "ttt_mlp_tmem"
    assert m(loss=1) == "ttt_mlp_tmem"
    assert m(weight_decay=0.1) == "ttt_mlp_fused"
    assert m(io_dtype=0) == "ttt_mlp_generic"
    monkeypatch.setenv("TTT_MLP_KERNEL", "fused")
    assert m() == "ttt_mlp_fused"
