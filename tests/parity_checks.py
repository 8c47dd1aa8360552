"""Element-wise parity checks of GPU results against the oracle.

The specification fixes the roundings (g = bf16(gate sum), u = bf16(up sum),
h = bf16(act(g) * u), out = bf16(down sum)) but leaves the accumulation order
free.  A GPU sum therefore differs from the exact one by at most its
accumulation error, bounded here by ACC_EPS * sum_k |x_k w_k|.  Because bf16
round-to-nearest-even is monotone, every rounding of a value within that
window of the exact sum lies in [bf16(v - w), bf16(v + w)]; where those two
ends coincide the rounded result is determined and the GPU must match the
oracle bit for bit.  Only where the window straddles a rounding boundary may
the GPU pick the neighbouring value, and then only inside the interval.

The helpers call the oracle for every value they compare against; they hold
none of the method's arithmetic themselves beyond interval bookkeeping.
"""
import numpy as np

import oracle

# Bound on the GPU's fp32 accumulation error, relative to sum_k |x_k w_k|:
# exact block products, fp32 block sums and FFMA scaling folded every 8
# chunks into an error-free hi/lo pair, then a few cross-range adds -- about
# 4e-6 in the worst case; twice that here.
ACC_EPS = 8e-6
# SiLU and the tanh GeLU each have one interior minimum (t*, act(t*)).
ACT_MIN_T = {oracle.ACT_SILU: -1.2784645427610738, oracle.ACT_GELU_TANH: -0.7524614257653106}


def bf16_round(v):
    """bf16 round-to-nearest-even of float64 values (through the oracle), widened back."""
    return oracle.bf16_bits_to_f64(oracle.bf16_from_double_array(v))


def rounding_interval(v, window):
    """[lo, hi] holding every bf16 rounding of a real number within `window` of v."""
    return bf16_round(v - window), bf16_round(v + window)


def abs_sum(x_bits, q, N):
    """scale2 * sum_k |x_k| |w_k| of every output (oracle GEMV of the magnitudes)."""
    codes = (q[0] & 0x77).astype(np.uint8)  # clear both nibbles' sign bits
    return oracle.gemv_f64((x_bits & 0x7FFF).astype(np.uint16), codes, q[1], q[2], N)


def gemv_interval(x_bits, q, N, acc_eps=ACC_EPS):
    """Interval of valid bf16 GEMV outputs [M, N] for x (bf16 bits) and q = (codes, scales, s2)."""
    v = oracle.gemv_f64(x_bits, q[0], q[1], q[2], N)
    return rounding_interval(v, acc_eps * abs_sum(x_bits, q, N))


def _stats(got, lo, hi, ref, what):
    """Assert lo <= got <= hi everywhere (so got == ref wherever lo == hi) and
    that the oracle's own value lies in its interval; return the counts."""
    assert np.all((lo <= ref) & (ref <= hi)), f"{what}: oracle value outside its own interval"
    bad = np.argwhere((got < lo) | (got > hi))
    determined = lo == hi
    wrong_det = np.argwhere(determined & (got != ref))
    assert wrong_det.size == 0, (f"{what}: {len(wrong_det)} determined elements differ from the "
                                 f"oracle, first {wrong_det[:5].tolist()}")
    assert bad.size == 0, (f"{what}: {len(bad)} elements outside their valid rounding interval, "
                           f"first {bad[:5].tolist()}")
    return {"n": int(got.size), "determined": int(determined.sum()),
            "differs": int(np.count_nonzero(got != ref))}


def check_gemv(y_bits, x_bits, q, N, what="gemv", acc_eps=ACC_EPS):
    """y (bf16 bits [M, N]) against the oracle GEMV: inside the rounding interval
    everywhere, bit-exact wherever the rounding is determined."""
    lo, hi = gemv_interval(x_bits, q, N, acc_eps)
    ref = oracle.bf16_bits_to_f64(oracle.gemv(x_bits, q[0], q[1], q[2], N))
    return _stats(oracle.bf16_bits_to_f64(y_bits), lo, hi, ref, what)


def hidden_interval(x_bits, gate, up, act, acc_eps=ACC_EPS):
    """Interval of valid h = bf16(act(g) * u) [M, I] for g and u the rounded
    gate and up projections of x (gemv_interval each)."""
    I = gate[0].shape[0]
    g_lo, g_hi = gemv_interval(x_bits, gate, I, acc_eps)
    u_lo, u_hi = gemv_interval(x_bits, up, I, acc_eps)
    return hidden_interval_from(g_lo, g_hi, u_lo, u_hi, act)


def hidden_interval_from(g_lo, g_hi, u_lo, u_hi, act):
    """Interval of valid h = bf16(act(g) * u) for g in [g_lo, g_hi] and u in
    [u_lo, u_hi] (bf16 values): act over its range on the g interval (monotone
    pieces plus the interior minimum), the product over the box corners,
    widened by the kernel's fp32 activation error."""
    a1, a2 = oracle.act_array(g_lo, act), oracle.act_array(g_hi, act)
    a_lo, a_hi = np.minimum(a1, a2), np.maximum(a1, a2)
    t_min = ACT_MIN_T[act]
    inside = (g_lo <= t_min) & (t_min <= g_hi)
    a_lo = np.where(inside, np.minimum(a_lo, oracle.act(t_min, act)), a_lo)
    corners = np.stack([a_lo * u_lo, a_lo * u_hi, a_hi * u_lo, a_hi * u_hi])
    p_lo, p_hi = corners.min(axis=0), corners.max(axis=0)
    # the kernel's fp32 activation: its relative error grows with the exponent
    # argument in the negative tails (act(t) ~ t e^-|arg|), measured below
    # 2.6 * |arg| * 6e-8 for GeLU-tanh and 1.2 * |t| * 6e-8 for SiLU
    g_far = np.maximum(np.abs(g_lo), np.abs(g_hi))
    arg = g_far if act == oracle.ACT_SILU else 1.5957691216057308 * (g_far + 0.044715 * g_far ** 3)
    rel = 4e-7 * (1.0 + arg)
    return bf16_round(p_lo - np.abs(p_lo) * rel), bf16_round(p_hi + np.abs(p_hi) * rel)


def check_hidden(h_bits, x_bits, gate, up, act, what="h", acc_eps=ACC_EPS):
    """GPU h against the oracle: inside the valid interval everywhere,
    bit-exact wherever it is determined."""
    lo, hi = hidden_interval(x_bits, gate, up, act, acc_eps)
    I = gate[0].shape[0]
    ref = oracle.bf16_bits_to_f64(oracle.ffn_hidden(x_bits, I, gate, up, act))
    return _stats(oracle.bf16_bits_to_f64(h_bits), lo, hi, ref, what)


def count_beyond_tolerance(got_bits, ref_bits, tol=1e-2):
    """Elements with |got - ref| > tol * max(1, |ref|)."""
    g = oracle.bf16_bits_to_f64(got_bits)
    r = oracle.bf16_bits_to_f64(ref_bits)
    return int(np.count_nonzero(np.abs(g - r) > tol * np.maximum(1.0, np.abs(r))))


def round_toward_zero_bf16(v):
    """bf16 rounding toward zero of float64 values (a deliberately wrong
    rounding, used to show the checks reject it)."""
    r = bf16_round(v)
    bits = oracle.bf16_from_double_array(v).astype(np.int32)
    away = np.abs(r) > np.abs(v)
    mag = np.where(away & ((bits & 0x7FFF) > 0), (bits & 0x7FFF) - 1, bits & 0x7FFF)
    return ((bits & 0x8000) | mag).astype(np.uint16)


def bf16_f64(bits):
    return oracle.bf16_bits_to_f64(np.asarray(bits, np.uint16))


def lora_delta_interval(v_lo, v_hi, A_bits, B_bits, acc_eps=ACC_EPS):
    """Interval of the adapter delta d = bf16(B bf16(A v)) [M, N] for v in the
    box [v_lo, v_hi] (float64 arrays [M, K] of bf16 values): A v over the box
    (interval arithmetic), its bf16 rounding interval with the fp32
    accumulation window, then B xa over the xa box likewise."""
    A = bf16_f64(A_bits)
    B = bf16_f64(B_bits)

    def box_matmul(lo, hi, W):  # [lo, hi] @ W.T elementwise-exact bounds
        Wp, Wn = np.maximum(W, 0.0), np.minimum(W, 0.0)
        return lo @ Wp.T + hi @ Wn.T, hi @ Wp.T + lo @ Wn.T

    mag = np.maximum(np.abs(v_lo), np.abs(v_hi))
    s_lo, s_hi = box_matmul(v_lo, v_hi, A)
    w = acc_eps * (mag @ np.abs(A).T)
    xa_lo, xa_hi = bf16_round(s_lo - w), bf16_round(s_hi + w)
    d_lo, d_hi = box_matmul(xa_lo, xa_hi, B)
    wd = acc_eps * (np.maximum(np.abs(xa_lo), np.abs(xa_hi)) @ np.abs(B).T)
    return bf16_round(d_lo - wd), bf16_round(d_hi + wd)


def check_interval(got_bits, lo, hi, ref_bits, what):
    """got inside [lo, hi] everywhere, equal to ref wherever lo == hi."""
    return _stats(bf16_f64(got_bits), lo, hi, bf16_f64(ref_bits), what)


# ------------------------------------------------------------ block-scaled FP8

def abs_sum_fp8(x_bits, q):
    """sum_k |x_k| |W[n][k]| for an FP8 projection q = (codes, grid)."""
    return oracle.gemv_fp8_f64((np.asarray(x_bits, np.uint16) & 0x7FFF).astype(np.uint16),
                               (np.asarray(q[0], np.uint8) & 0x7F).astype(np.uint8),
                               np.abs(np.asarray(q[1], np.float32)))


def gemv_interval_fp8(x_bits, q, acc_eps=ACC_EPS):
    v = oracle.gemv_fp8_f64(x_bits, q[0], q[1])
    return rounding_interval(v, acc_eps * abs_sum_fp8(x_bits, q))


def check_gemv_fp8(y_bits, x_bits, q, what="w8a16 gemv", acc_eps=ACC_EPS):
    lo, hi = gemv_interval_fp8(x_bits, q, acc_eps)
    ref = oracle.bf16_bits_to_f64(oracle.gemv_fp8(x_bits, q[0], q[1]))
    return _stats(oracle.bf16_bits_to_f64(y_bits), lo, hi, ref, what)


def check_hidden_fp8(h_bits, x_bits, gate, up, act, what="w8a16 h", acc_eps=ACC_EPS):
    g_lo, g_hi = gemv_interval_fp8(x_bits, gate, acc_eps)
    u_lo, u_hi = gemv_interval_fp8(x_bits, up, acc_eps)
    lo, hi = hidden_interval_from(g_lo, g_hi, u_lo, u_hi, act)
    ref = oracle.bf16_bits_to_f64(oracle.ffn_fp8_hidden(x_bits, gate, up, act))
    return _stats(oracle.bf16_bits_to_f64(h_bits), lo, hi, ref, what)
