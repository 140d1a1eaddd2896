"""Host-side checks of the seeded input generator (no method arithmetic)."""
import numpy as np

from test_sequence_layers_08_b300.inputs import CONFIGS, bf16_bits, make_inputs, round_bf16


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, 1.0 + 3 * 2 ** -8, -2.5],
                 dtype=np.float32)
    r = round_bf16(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins
    assert r[0] == 1.0 and r[1] == 1.0
    assert r[2] == np.float32(1.0 + 2 ** -7)
    assert r[3] == np.float32(1.0 + 2 ** -6)   # tie, rounds to even
    assert r[4] == -2.5
    assert np.all(bf16_bits(r).astype(np.uint32) << 16 == r.view(np.uint32))


def test_inputs_are_deterministic_and_bf16_exact():
    cfg = CONFIGS["linear_ln_bf16_B4_H16_L8192"].with_(B=1, H=2, L=64)
    a, b = make_inputs(cfg, 0), make_inputs(cfg, 0)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(np.asarray(a[k]), np.asarray(b[k]))
    for k in ("Q", "K", "V"):
        assert np.array_equal(round_bf16(a[k]), a[k])
    c = make_inputs(cfg, 1)
    assert not np.array_equal(a["Q"], c["Q"])


def test_input_statistics():
    cfg = CONFIGS["linear_bf16_B8_H12_L2048"].with_(B=2, H=4, L=1024)
    x = make_inputs(cfg, 0)
    assert x["Q"].shape == (2, 4, 1024, 64)
    assert abs(x["Q"].std() - 1 / 8) < 0.01
    assert abs(x["W0"].std() - 0.02) < 0.002
    assert abs(x["b0"].std() - 0.01) < 0.002
    # the gate's inputs, not eta itself: x ~ N(0, 1) (bf16-exact), theta ~ N(0, 0.02^2)
    assert "eta" not in x
    assert x["x"].shape == (2, 1024, 768) and x["theta"].shape == (4, 768)
    assert np.array_equal(round_bf16(x["x"]), x["x"])
    assert abs(x["x"].std() - 1.0) < 0.01
    assert abs(x["theta"].std() - 0.02) < 0.001
    assert x["eta_base"] == 1 / 64
    assert x["gamma"] is None


def test_uniform_eta_range_and_determinism():
    from test_sequence_layers_08_b300.inputs import uniform_eta
    a = uniform_eta(2, 3, 50, 0.2, 0.5, seed=4)
    assert a.shape == (2, 3, 50) and a.dtype == np.float32
    assert a.min() >= 0.2 and a.max() < 0.5
    np.testing.assert_array_equal(a, uniform_eta(2, 3, 50, 0.2, 0.5, seed=4))


def test_drift_shifts_k_and_v_only():
    cfg = CONFIGS["linear_ln_drift_bf16_B1_H32_L32768"].with_(H=2, L=3 * 4096)
    x = make_inputs(cfg, 0)
    seg = lambda a, j: a[:, :, j * 4096:(j + 1) * 4096].mean()
    for k in ("K", "V"):
        assert abs(seg(x[k], 2) - seg(x[k], 0) - 0.2 / 8) < 3e-3
    assert abs(seg(x["Q"], 2) - seg(x["Q"], 0)) < 3e-3


def test_const_eta_and_zero_bias():
    x = make_inputs(CONFIGS["linear_f32_B1_H2_L256"], 0)
    assert np.all(x["eta"] == np.float32(0.1))
    assert np.all(x["b0"] == 0)
    assert x["Q"].dtype == np.float32
