"""Pins of the oracle's LoRA overlay (the dense-FFN page's apply_lora_gate_up /
apply_lora_down): exact rational arithmetic with an independent bf16 rounding
for the three steps xa = bf16(A v), delta = bf16(B xa), base = bf16(base +
delta); and the composition (gate/up deltas before the activation, the down
delta after the down projection and contracted over h, not over x)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

from test_oracle_pins import representable_weight


def bf16_rne(q: Fraction) -> Fraction:
    """Nearest bf16 value to an exact rational (ties to an even significand);
    normal and subnormal range only (no overflow in these pins)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)  # subnormals share the smallest normal exponent's spacing
    step = Fraction(2) ** (e - 7)
    n = a / step
    lo = n.numerator // n.denominator
    frac = n - lo
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * lo * step


def bits_to_fr(b):
    return Fraction(float(oracle.bf16_bits_to_f64(np.uint16(b))))


def fr_to_bits(q):
    return int(oracle.bf16_from_double(float(q)))  # q is bf16-exact here


def test_independent_bf16_rounding_agrees_with_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                           [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(257.0), 2 ** -130 * 1.5]])
    t = torch.tensor(vals.astype(np.float32)).to(torch.bfloat16).float().double().numpy()
    for v, ref in zip(vals.astype(np.float32), t):
        assert float(bf16_rne(Fraction(float(v)))) == ref


def _bf16_grid(rng, shape, lo=-8, hi=8, halves=True):
    """bf16-exact small values (integers or halves)."""
    v = rng.integers(lo * 2, hi * 2 + 1, size=shape) / (2.0 if halves else 1.0)
    return torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def test_lora_xa_exact():
    rng = np.random.default_rng(1)
    M, K, r = 3, 48, 5
    v = _bf16_grid(rng, (M, K))
    A = _bf16_grid(rng, (r, K))
    got = oracle.lora_xa(v, A)
    for m in range(M):
        for j in range(r):
            exact = sum(bits_to_fr(A[j, k]) * bits_to_fr(v[m, k]) for k in range(K))
            assert bits_to_fr(got[m, j]) == bf16_rne(exact), (m, j)
    # sums that must round, including a tie (257 = 256 + 1: spacing 2 at 256)
    v = _bf16_grid(rng, (1, 2), 0, 0)
    v[0, 0] = fr_to_bits(Fraction(257 - 1))  # 256
    v[0, 1] = fr_to_bits(Fraction(1))
    A = np.array([[fr_to_bits(1), fr_to_bits(1)], [fr_to_bits(1), fr_to_bits(3)]], np.uint16)
    got = oracle.lora_xa(v, A)
    assert bits_to_fr(got[0, 0]) == 256          # 257 ties to the even 256
    assert bits_to_fr(got[0, 1]) == 260          # 259 rounds up to 260


def test_lora_delta_and_add_exact():
    rng = np.random.default_rng(2)
    M, r, N = 2, 7, 33
    xa = _bf16_grid(rng, (M, r), -40, 40)
    B = _bf16_grid(rng, (N, r))
    d = oracle.lora_delta(xa, B)
    for m in range(M):
        for n in range(N):
            exact = sum(bits_to_fr(B[n, j]) * bits_to_fr(xa[m, j]) for j in range(r))
            assert bits_to_fr(d[m, n]) == bf16_rne(exact)
    base = _bf16_grid(rng, (M, N), -300, 300)
    out = oracle.lora_add(base, d)
    for i in range(M * N):
        exact = bits_to_fr(base.flat[i]) + bits_to_fr(d.flat[i])
        assert bits_to_fr(out.flat[i]) == bf16_rne(exact)
    # lora_apply is the three steps in order
    v = _bf16_grid(rng, (M, 11))
    A = _bf16_grid(rng, (r, 11))
    assert np.array_equal(oracle.lora_apply(v, A, B, base),
                          oracle.lora_add(base, oracle.lora_delta(oracle.lora_xa(v, A), B)))


def _ffn_case(H=32, I=48, M=2, r=3, seed=5):
    rng = np.random.default_rng(seed)
    q = [representable_weight(n, k, -8, rng)[0] for n, k in ((I, H), (I, H), (H, I))]
    q = [oracle.quantize(w) for w in q]
    x = _bf16_grid(rng, (M, H), -3, 3)
    mk = lambda n, k: _bf16_grid(rng, (n, k), -2, 2)  # noqa: E731
    lora = dict(rank=r, gate=(mk(r, H), mk(I, r)), up=(mk(r, H), mk(I, r)),
                down=(mk(r, I), mk(H, r)))
    return x, q, lora


@pytest.mark.parametrize("act", [oracle.ACT_SILU, oracle.ACT_GELU_TANH])
def test_ffn_lora_composition(act):
    """g and u take their deltas (of x) before the activation; out takes the
    down delta, contracted over h, after the down projection."""
    x, (gq, uq, dq), lora = _ffn_case()
    I = gq[0].shape[0]
    H = x.shape[1]
    out, h = oracle.ffn_lora(x, I, gq, uq, dq, act, lora)
    g = oracle.lora_apply(x, *lora["gate"], oracle.gemv(x, *gq, I))
    u = oracle.lora_apply(x, *lora["up"], oracle.gemv(x, *uq, I))
    gv, uv = oracle.bf16_bits_to_f64(g), oracle.bf16_bits_to_f64(u)
    h_ref = oracle.bf16_from_double_array(oracle.act_array(gv, act) * uv)
    assert np.array_equal(h, h_ref)
    out_ref = oracle.lora_apply(h, *lora["down"], oracle.gemv(h, *dq, H))
    assert np.array_equal(out, out_ref)
    # each delta matters here, so a misplaced one is visible
    assert not np.array_equal(out, oracle.ffn(x, I, gq, uq, dq, act))
    assert not np.array_equal(h, oracle.ffn_hidden(x, I, gq, uq, act))


def test_ffn_lora_distinguishes_misplaced_deltas():
    """Mistakes a kernel could make give different results: the gate delta
    after the activation, or the down delta taken over x instead of h."""
    x, (gq, uq, dq), lora = _ffn_case(H=48, I=48)
    I = H = 48
    out, h = oracle.ffn_lora(x, I, gq, uq, dq, oracle.ACT_SILU, lora)
    wrong_over_x = oracle.lora_apply(x, *lora["down"], oracle.gemv(h, *dq, H))
    assert not np.array_equal(out, wrong_over_x)
    no_gate = dict(lora, gate=None)
    h_plain = oracle.ffn_lora(x, I, gq, uq, dq, oracle.ACT_SILU, no_gate)[1]
    assert not np.array_equal(h, h_plain)


def test_ffn_lora_with_zero_b_is_the_plain_ffn():
    x, (gq, uq, dq), lora = _ffn_case()
    I = gq[0].shape[0]
    zero = {k: (v[0], np.zeros_like(v[1])) for k, v in lora.items() if k != "rank"}
    zero["rank"] = lora["rank"]
    out, h = oracle.ffn_lora(x, I, gq, uq, dq, oracle.ACT_GELU_TANH, zero)
    assert np.array_equal(out, oracle.ffn(x, I, gq, uq, dq, oracle.ACT_GELU_TANH))
    assert np.array_equal(h, oracle.ffn_hidden(x, I, gq, uq, oracle.ACT_GELU_TANH))
    out2, _ = oracle.ffn_lora(x, I, gq, uq, dq, oracle.ACT_GELU_TANH, None)
    assert np.array_equal(out2, out)
