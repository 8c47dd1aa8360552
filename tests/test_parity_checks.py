"""The parity checks themselves, on the CPU: they accept the oracle's own
results and reject plausible kernel mistakes planted in oracle-derived data
(round-toward-zero conversions, a one-ulp error, an unrounded g, swapped
gate/up, a dropped scale)."""
import numpy as np
import pytest

import oracle
from nvfp4_weight_only_gb300 import synth

import parity_checks as pc


def _ffn_inputs(H=256, I=512, M=3, outliers=0.0, seed=0):
    gate = oracle.quantize(synth.weights_f32(I, H, seed=synth.layer_seed(seed, synth.GATE)).numpy())
    up = oracle.quantize(synth.weights_f32(I, H, seed=synth.layer_seed(seed, synth.UP)).numpy())
    down = oracle.quantize(synth.weights_f32(H, I, seed=synth.layer_seed(seed, synth.DOWN)).numpy())
    x = synth.bf16_bits(synth.activations_bf16(M, H, seed=seed, outlier_frac=outliers))
    return x, gate, up, down


@pytest.mark.parametrize("act", [oracle.ACT_SILU, oracle.ACT_GELU_TANH])
def test_oracle_hidden_passes_and_is_mostly_determined(act):
    x, gate, up, _ = _ffn_inputs()
    h = oracle.ffn_hidden(x, 512, gate, up, act)
    st = pc.check_hidden(h, x, gate, up, act)
    assert st["differs"] == 0
    # the check has teeth only where the rounding is determined: most elements
    assert st["determined"] > 0.6 * st["n"]


def _hidden_parts(x, gate, up, act):
    I = gate[0].shape[0]
    g = pc.bf16_round(oracle.gemv_f64(x, gate[0], gate[1], gate[2], I))
    u = pc.bf16_round(oracle.gemv_f64(x, up[0], up[1], up[2], I))
    return g, u, oracle.act_array(g, act) * u


@pytest.mark.parametrize("act", [oracle.ACT_SILU, oracle.ACT_GELU_TANH])
def test_hidden_check_rejects_round_toward_zero(act):
    x, gate, up, _ = _ffn_inputs()
    _, _, p = _hidden_parts(x, gate, up, act)
    with pytest.raises(AssertionError):
        pc.check_hidden(pc.round_toward_zero_bf16(p), x, gate, up, act)


def test_hidden_check_rejects_truncated_g():
    """g and u rounded toward zero (a truncating bf16 conversion), h correct."""
    x, gate, up, _ = _ffn_inputs()
    I = 512
    g = oracle.bf16_bits_to_f64(pc.round_toward_zero_bf16(
        oracle.gemv_f64(x, gate[0], gate[1], gate[2], I)))
    u = oracle.bf16_bits_to_f64(pc.round_toward_zero_bf16(
        oracle.gemv_f64(x, up[0], up[1], up[2], I)))
    h = oracle.bf16_from_double_array(oracle.act_array(g, 0) * u)
    with pytest.raises(AssertionError):
        pc.check_hidden(h, x, gate, up, oracle.ACT_SILU)


def test_hidden_check_rejects_unrounded_g_and_swapped_projections():
    x, gate, up, _ = _ffn_inputs()
    I = 512
    g = oracle.gemv_f64(x, gate[0], gate[1], gate[2], I)  # not rounded to bf16
    u = pc.bf16_round(oracle.gemv_f64(x, up[0], up[1], up[2], I))
    with pytest.raises(AssertionError):
        pc.check_hidden(oracle.bf16_from_double_array(oracle.act_array(g, 0) * u), x, gate, up, 0)
    with pytest.raises(AssertionError):  # act applied to up instead of gate
        pc.check_hidden(oracle.ffn_hidden(x, I, up, gate, 0), x, gate, up, 0)


def test_hidden_check_rejects_one_ulp_at_a_determined_element():
    x, gate, up, _ = _ffn_inputs()
    h = oracle.ffn_hidden(x, 512, gate, up, 0)
    lo, hi = pc.hidden_interval(x, gate, up, 0)
    idx = np.argwhere((lo == hi) & (lo != 0))[7]
    h2 = h.copy()
    h2[tuple(idx)] += 1  # one bf16 ulp away from zero
    with pytest.raises(AssertionError):
        pc.check_hidden(h2, x, gate, up, 0)


def test_gemv_check_rejects_round_toward_zero_and_dropped_scale():
    x, gate, _, _ = _ffn_inputs(M=5, outliers=0.01)
    N = 512
    y = oracle.gemv(x, gate[0], gate[1], gate[2], N)
    assert pc.check_gemv(y, x, gate, N)["differs"] == 0
    v = oracle.gemv_f64(x, gate[0], gate[1], gate[2], N)
    with pytest.raises(AssertionError):
        pc.check_gemv(pc.round_toward_zero_bf16(v), x, gate, N)
    with pytest.raises(AssertionError):  # scale2 applied twice
        pc.check_gemv(oracle.bf16_from_double_array(v * gate[2]), x, gate, N)


def test_output_check_rejects_round_toward_zero():
    x, gate, up, down = _ffn_inputs(M=2)
    h = oracle.ffn_hidden(x, 512, gate, up, 0)
    o = oracle.gemv_f64(h, down[0], down[1], down[2], 256)
    with pytest.raises(AssertionError):
        pc.check_gemv(pc.round_toward_zero_bf16(o), h, down, 256, "out")


def test_round_toward_zero_helper():
    # bf16 spacing is 2^-7 on [1, 2); bf16 keeps fp32's subnormals (2^-133 apart)
    v = np.array([1.0 + 2.0 ** -8, -(1.0 + 3 * 2.0 ** -8), 3.0, -0.0, 1.5 * 2.0 ** -133])
    got = oracle.bf16_bits_to_f64(pc.round_toward_zero_bf16(v))
    np.testing.assert_array_equal(got, [1.0, -(1.0 + 2.0 ** -7), 3.0, -0.0, 2.0 ** -133])
