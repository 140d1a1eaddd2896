"""CPU checks of bench.py's bookkeeping: the algorithmic FLOP and byte counts behind the
roofline fraction, the flat copy buffers of the end-to-end steps, and the rule that a
measured DRAM-traffic figure is only reported for the kernel source it was taken of."""
import hashlib
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from test_sequence_layers_08_b300.inputs import CONFIGS  # noqa: E402


def test_flops_per_head_token():
    # linear: three d x d products per token plus the two 16-wide blocks
    assert bench.flops_per_head_token(CONFIGS["linear_bf16_B8_H12_L2048"]) == 28672.0
    # MLP 64 -> 256 -> 64: seven d x dh products plus the blocks
    assert bench.flops_per_head_token(CONFIGS["mlp_ln_bf16_B4_H12_L4096"]) == 249856.0


@pytest.mark.parametrize("name,per_token", [("linear_bf16_B8_H12_L2048", 516),
                                            ("linear_f32_B1_H2_L256", 1028)])
def test_algorithmic_bytes(name, per_token):
    cfg = CONFIGS[name]
    d = cfg.d
    state = (d * d + d) * 4
    expect = cfg.B * cfg.H * cfg.L * per_token + state * cfg.H + state * cfg.B * cfg.H
    assert bench.algorithmic_bytes(cfg) == float(expect)


def test_packed_buffers_are_aligned_views():
    specs = [((2, 3, 5), torch.bfloat16), ((7,), torch.float32), ((4, 4), torch.float32)]
    flat, views = bench.packed(specs, "cpu")
    base = flat.data_ptr()
    for (shape, dt), v in zip(specs, views):
        assert tuple(v.shape) == shape and v.dtype == dt and v.is_contiguous()
        assert (v.data_ptr() - base) % 256 == 0
    views[1].fill_(3.0)
    assert torch.equal(flat[256:256 + 28].view(torch.float32), torch.full((7,), 3.0))
    assert flat.numel() == 3 * 256


def test_measured_traffic_needs_the_same_source(tmp_path, monkeypatch):
    csrc = tmp_path / "test_sequence_layers_08_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "ttt_linear_tc.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles" / "ttt_linear_fused_ncu_w.md").write_text(
        f"# summary\n\ntraffic_bytes_per_launch: 12345\nkernel_source_sha256: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("ttt_linear_fused", "w") == 12345.0
    assert bench.measured_traffic("ttt_linear_fused", "other") is None
    assert bench.measured_traffic("no_such_kernel", "w") is None
    src.write_text("// kernel v2\n")          # the kernel changed since the capture
    assert bench.measured_traffic("ttt_linear_fused", "w") is None
