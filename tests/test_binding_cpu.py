"""The Python binding checks every operand (shape, dtype, device, contiguity) before it
calls into the C library, so a short eta, a smaller output buffer or K with another
length is an exception on the host, never an out-of-bounds access on the GPU.  These
checks run on host tensors: each case breaks one operand of an otherwise valid call."""
import pytest
import torch

import test_sequence_layers_08_b300 as ttt

B, H, L, d, dh = 2, 3, 32, 64, 256


def linear_args(dtype=torch.bfloat16, per_batch=False):
    lead = (B, H) if per_batch else (H,)
    f32 = torch.float32
    return dict(Q=torch.zeros(B, H, L, d, dtype=dtype), K=torch.zeros(B, H, L, d, dtype=dtype),
                V=torch.zeros(B, H, L, d, dtype=dtype), eta=torch.zeros(B, H, L, dtype=f32),
                W0=torch.zeros(*lead, d, d, dtype=f32), b0=torch.zeros(*lead, d, dtype=f32),
                gamma=torch.ones(H, d, dtype=f32), beta=torch.zeros(H, d, dtype=f32))


def mlp_args():
    f32 = torch.float32
    a = linear_args()
    del a["W0"], a["b0"]
    a.update(W1=torch.zeros(H, d, dh, dtype=f32), b1=torch.zeros(H, dh, dtype=f32),
             W2=torch.zeros(H, dh, d, dtype=f32), b2=torch.zeros(H, d, dtype=f32))
    return a


def call_linear(a, **kw):
    return ttt.ttt_linear_fwd(a["Q"], a["K"], a["V"], a["eta"], a["W0"], a["b0"], a["gamma"],
                              a["beta"], residual_ln=True, **kw)


def call_mlp(a, **kw):
    return ttt.ttt_mlp_fwd(a["Q"], a["K"], a["V"], a["eta"], a["W1"], a["b1"], a["W2"], a["b2"],
                           a["gamma"], a["beta"], residual_ln=True, **kw)


def test_valid_host_call_is_refused_for_its_device():
    with pytest.raises(TypeError, match="CUDA device"):
        call_linear(linear_args())
    with pytest.raises(TypeError, match="CUDA device"):
        call_mlp(mlp_args())


@pytest.mark.parametrize("name,bad", [
    ("K", torch.zeros(B, H, L - 16, d, dtype=torch.bfloat16)),
    ("V", torch.zeros(B, H, L, d, dtype=torch.float32)),
    ("eta", torch.zeros(B, H, L - 1)),
    ("eta", torch.zeros(B, H, L, dtype=torch.float64)),
    ("W0", torch.zeros(H, d, d + 1)),
    ("W0", torch.zeros(B, H, d, d)),          # per-batch shape without init_per_batch
    ("b0", torch.zeros(H + 1, d)),
    ("gamma", torch.ones(H, d - 1)),
    ("beta", torch.zeros(1, d)),
    ("K", torch.zeros(B, H, d, L, dtype=torch.bfloat16).transpose(2, 3)),   # not contiguous
])
def test_linear_operand_mismatch(name, bad):
    a = linear_args()
    a[name] = bad
    with pytest.raises((ValueError, TypeError), match=name):
        call_linear(a)


def test_linear_noncontiguous_q():
    a = linear_args()
    a["Q"] = torch.zeros(B, H, d, L, dtype=torch.bfloat16).transpose(2, 3)
    with pytest.raises(ValueError, match="Q"):
        call_linear(a)


@pytest.mark.parametrize("which,shape,dtype", [
    (0, (B, H, L - 16, d), torch.bfloat16),
    (0, (B, H, L, d), torch.float32),
    (1, (H, d, d), torch.float32),
    (2, (B, H, d + 1), torch.float32),
])
def test_linear_output_mismatch(which, shape, dtype):
    a = linear_args()
    out = [torch.empty(B, H, L, d, dtype=torch.bfloat16), torch.empty(B, H, d, d),
           torch.empty(B, H, d)]
    out[which] = torch.empty(shape, dtype=dtype)
    with pytest.raises((ValueError, TypeError), match="out"):
        call_linear(a, out=tuple(out))


def test_linear_per_batch_state_shapes():
    a = linear_args(per_batch=True)
    with pytest.raises(TypeError, match="CUDA device"):   # shapes accepted
        call_linear(a, init_per_batch=True)
    with pytest.raises(ValueError, match="W0"):
        call_linear(a, init_per_batch=False)


@pytest.mark.parametrize("name,bad", [
    ("W1", torch.zeros(H, d, dh // 2)),
    ("W2", torch.zeros(H, dh, d - 8)),
    ("b2", torch.zeros(H, dh)),
    ("eta", torch.zeros(B, H + 1, L)),
])
def test_mlp_operand_mismatch(name, bad):
    a = mlp_args()
    a[name] = bad
    with pytest.raises((ValueError, TypeError), match=name):
        call_mlp(a)


def test_step_state_shapes():
    a = linear_args()
    W = torch.zeros(B, H, d, d)
    b = torch.zeros(B, H, d)
    with pytest.raises(TypeError, match="CUDA device"):
        ttt.ttt_linear_step(a["Q"], a["K"], a["V"], a["eta"], W, b)
    with pytest.raises(ValueError, match="W"):
        ttt.ttt_linear_step(a["Q"], a["K"], a["V"], a["eta"], W[:, :1].contiguous(), b)
    with pytest.raises(ValueError, match="out Z"):
        ttt.ttt_linear_step(a["Q"], a["K"], a["V"], a["eta"], W, b,
                            out=torch.empty(B, H, L - 1, d, dtype=torch.bfloat16))


def test_partition_rows_is_balanced_and_covers_every_row():
    for total in (0, 1, 7, 64, 96, 1000):
        for world in (1, 2, 3, 8):
            ranges = [ttt.partition_rows(total, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == total
            for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
                assert a1 == b0
            sizes = [r1 - r0 for r0, r1 in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        ttt.partition_rows(10, 0, 0)
    with pytest.raises(ValueError):
        ttt.partition_rows(10, 2, 2)


def test_row_form_shapes():
    """Row form: Q [rows, L, d] with heads=H; row-indexed tensors carry [rows, ...], the
    head-shared initial state and LayerNorm parameters stay [H, ...]."""
    rows, f32, bf = 4, torch.float32, torch.bfloat16
    a = dict(Q=torch.zeros(rows, L, d, dtype=bf), K=torch.zeros(rows, L, d, dtype=bf),
             V=torch.zeros(rows, L, d, dtype=bf), eta=torch.zeros(rows, L),
             W0=torch.zeros(H, d, d), b0=torch.zeros(H, d), gamma=torch.ones(H, d),
             beta=torch.zeros(H, d))
    with pytest.raises(TypeError, match="CUDA device"):
        call_linear(a, heads=H, bh_offset=2)
    bad = dict(a, eta=torch.zeros(rows + 1, L))
    with pytest.raises(ValueError, match="eta"):
        call_linear(bad, heads=H, bh_offset=2)
    with pytest.raises(ValueError, match="row form"):
        call_linear(a)                       # 3-D Q needs heads=
    with pytest.raises(ValueError, match="bh_offset"):
        call_linear(linear_args(), bh_offset=1)
    desc = ttt.make_desc(a["Q"], 16, True, heads=H, bh_offset=2)
    assert (desc.B, desc.H, desc.bh_offset, desc.bh_count) == (2, H, 2, rows)
