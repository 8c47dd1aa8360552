"""Pins of the CPU oracle against facts fixed outside it (CPU only).

Each test checks the oracle against a published table, an independent
implementation (torch's own fp8/bf16 converters), a closed form, an invariant
of the mathematics, or an exact hand-expanded sum on tiny shapes.  A dropped
term, a swapped nibble, a transposed operand or a wrong sign in the oracle
breaks at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()
            rows.append((a, b))
    return rows


# ---------------------------------------------------------------- codecs

def test_e2m1_table_matches_published_values():
    rows = _read_pairs("e2m1_table.txt")
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s, 16), float(val_s)
        got = oracle.e2m1_decode(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_e2m1_rounding_table():
    for q_s, code_s in _read_pairs("e2m1_rounding.txt"):
        q = float(np.float32(float(q_s)))
        assert oracle.e2m1_encode(q) == int(code_s, 16), q_s


def test_e2m1_encode_decode_roundtrip_and_nearest():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_decode(c)) == c
    grid = sorted({abs(oracle.e2m1_decode(c)) for c in range(8)})
    rng = np.random.default_rng(1)
    for q in rng.uniform(-7.0, 7.0, 4000).astype(np.float32):
        code = oracle.e2m1_encode(float(q))
        v = oracle.e2m1_decode(code)
        best = min(abs(abs(float(q)) - g) for g in grid)
        if abs(q) <= 6:
            assert abs(abs(v) - abs(float(q))) == best
        else:
            assert abs(v) == 6.0
        assert (code >> 3) == (1 if np.signbit(q) else 0)


def test_e4m3_golden_values():
    for b_s, v_s in _read_pairs("e4m3_values.txt"):
        b = int(b_s, 16)
        got = oracle.e4m3_decode(b)
        if v_s == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v_s) and math.copysign(1, got) == math.copysign(1, float(v_s))


def test_e4m3_decode_matches_torch_for_all_bytes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double()
    for b in range(256):
        got = oracle.e4m3_decode(b)
        r = ref[b].item()
        if math.isnan(r):
            assert math.isnan(got), b
        else:
            assert got == r, b


def test_e4m3_encode_rne_matches_torch_in_range():
    # Every finite non-negative e4m3 value, every midpoint between neighbours,
    # points just either side of each midpoint, and random values below 448.
    vals = sorted({oracle.e4m3_decode(b) for b in range(0x7F)})
    pts = list(vals)
    for a, b in zip(vals[:-1], vals[1:]):
        m = (a + b) / 2
        pts += [m, float(np.nextafter(np.float32(m), np.float32(0))),
                float(np.nextafter(np.float32(m), np.float32(1e9)))]
    rng = np.random.default_rng(2)
    pts += list(rng.uniform(0, 448, 3000)) + list(rng.uniform(0, 0.02, 1000))
    q = np.array(pts, np.float32)
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(q, ref):
        assert oracle.e4m3_encode(float(v)) == int(r), float(v)


def test_e4m3_roundtrip_and_saturation():
    for b in range(256):
        if (b & 0x7F) == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(b)) == b
    for v in (448.0, 449.0, 464.0, 479.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E


def test_bf16_rounding_matches_torch_on_floats():
    rng = np.random.default_rng(3)
    f = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1e-40, -3e-39, 3.3e38, 3.4e38]]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for v, r in zip(f, ref):
        assert oracle.bf16_from_double(float(v)) == int(r), float(v)


def test_bf16_rounding_is_single_rounding_from_double():
    # 1 + 2^-8 + 2^-30 lies above the bf16 midpoint 1 + 2^-8; a detour through
    # fp32 would land on the midpoint first and then tie to 1.0.
    assert oracle.bf16_from_double(1 + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.bf16_from_double(1 + 2 ** -8) == 0x3F80           # tie -> even
    assert oracle.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82       # tie -> even (up)
    assert oracle.bf16_from_double(-(1 + 2 ** -8 + 2 ** -30)) == 0xBF81
    for b in (0x0001, 0x3F80, 0x7F7F, 0x8001, 0xC2F7):
        assert oracle.bf16_from_double(oracle.bf16_decode(b)) == b


# ---------------------------------------------------------- representable tensors

E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def representable_weight(N, K, j, rng, force_six=True):
    """W whose NVFP4 encoding is known in advance: scale2 = 2^j, per-block
    scales s (exact e4m3), each block holding a +-6 element so its amax is
    6*s*2^j, and block 0 using s = 448 so the tensor amax is 2688*2^j.
    Returns (W fp32, codes, scales) with codes packed element 2j -> low nibble."""
    scales = rng.integers(1, 0x7F, size=(N, K // 16)).astype(np.uint8)
    scales[0, 0] = 0x7E
    codes_el = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    if force_six:
        pos = rng.integers(0, 16, size=(N, K // 16))
        for n in range(N):
            for b in range(K // 16):
                codes_el[n, b * 16 + pos[n, b]] = 7 | (codes_el[n, b * 16 + pos[n, b]] & 8)
    W = np.zeros((N, K), np.float32)
    s_val = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).float().numpy()
    for n in range(N):
        for k in range(K):
            c = codes_el[n, k]
            mag = E2M1_MAGS[c & 7]
            v = mag * float(s_val[n, k // 16]) * 2.0 ** j
            W[n, k] = -v if (c & 8) else v
    packed = (codes_el[:, 0::2] | (codes_el[:, 1::2] << 4)).astype(np.uint8)
    return W, packed, scales


@pytest.mark.parametrize("j", [-9, -3, 0, 2])
def test_quantize_exact_on_representable_tensor(j):
    rng = np.random.default_rng(10 + j)
    N, K = 8, 64
    W, codes, scales = representable_weight(N, K, j, rng)
    c2, s2, scale2 = oracle.quantize(W)
    assert scale2 == 2.0 ** j
    np.testing.assert_array_equal(s2, scales)
    np.testing.assert_array_equal(c2, codes)
    D = oracle.dequantize(c2, s2, scale2, N, K)
    np.testing.assert_array_equal(D, W.astype(np.float64))


def test_quantize_ties_inside_a_block():
    # scale2 = 1 (amax 2688), block scale 448 -> q = w / 448 exactly.
    s = 448.0
    row = [6 * s, 0.25 * s, 0.75 * s, 1.25 * s, 1.75 * s, 2.5 * s, 3.5 * s, 5 * s,
           -0.25 * s, -0.75 * s, -2.5 * s, -5 * s, 0.0, -0.0, 7 * s / 7, -6 * s]
    W = np.array([row], np.float32)
    codes, scales, scale2 = oracle.quantize(W)
    assert scale2 == 1.0 and scales[0, 0] == 0x7E
    el = np.empty(16, np.uint8)
    el[0::2] = codes[0] & 15
    el[1::2] = codes[0] >> 4
    expect = [0x7, 0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x8, 0xA, 0xC, 0xE, 0x0, 0x8, 0x2, 0xF]
    assert list(el) == expect


def test_quantize_equal_magnitude_block_gives_six():
    rng = np.random.default_rng(5)
    W = np.zeros((4, 64), np.float32)
    W[0, :] = 3.0                      # sets the tensor amax
    for b in range(4):
        a = np.float32(rng.uniform(0.01, 3.0))
        sg = rng.choice([-1.0, 1.0], 16).astype(np.float32)
        W[1 + b % 3, b * 16:(b + 1) * 16] = sg * a
    codes, scales, _ = oracle.quantize(W)
    for n in range(4):
        for b in range(4):
            blk = W[n, b * 16:(b + 1) * 16]
            if not np.all(np.abs(blk) == np.abs(blk[0])) or blk[0] == 0:
                continue
            el = np.empty(16, np.uint8)
            el[0::2] = codes[n, b * 8:(b + 1) * 8] & 15
            el[1::2] = codes[n, b * 8:(b + 1) * 8] >> 4
            assert np.all((el & 7) == 7), (n, b)


def test_quantize_zero_tensor():
    W = np.zeros((3, 32), np.float32)
    W[1, 5] = -0.0
    codes, scales, scale2 = oracle.quantize(W)
    assert scale2 == 1.0
    assert np.all(scales == 0)
    assert codes[1, 2] == 0x80 and np.count_nonzero(codes) == 1


def test_quantize_bf16_source_equals_widened_fp32():
    rng = np.random.default_rng(6)
    w = torch.from_numpy(rng.standard_normal((16, 128)).astype(np.float32) * 0.02).bfloat16()
    bits = w.view(torch.int16).numpy().view(np.uint16)
    a = oracle.quantize_bf16(bits)
    b = oracle.quantize(w.float().numpy())
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert a[2] == b[2]


def test_quantize_error_bound_on_gaussian():
    # Each element lands on the nearest point of its block's grid
    # {0,.5,1,1.5,2,3,4,6} * s * scale2: the error is at most half the local
    # gap (0.25 below 2, 0.5 up to 4, 1 up to 6, in units of s*scale2), and
    # s*scale2 is bamax/6 to within the e4m3 rounding (at most 1/16).
    rng = np.random.default_rng(7)
    W = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    codes, scales, scale2 = oracle.quantize(W)
    D = oracle.dequantize(codes, scales, scale2, 64, 256)
    s = oracle.dequantize(np.full_like(codes, 0x22), scales, scale2, 64, 256)  # e2m1 1.0 * s * scale2
    unit = np.abs(s)
    q = np.abs(W) / np.where(unit > 0, unit, 1)
    half_gap = np.where(q <= 2, 0.25, np.where(q <= 4, 0.5, 1.0))
    assert np.all(np.abs(W - D) <= half_gap * unit * (1 + 1e-6) + 1e-12)
    bamax = np.abs(W.reshape(64, 16, 16)).max(axis=2).repeat(16, axis=1)
    assert np.all(unit <= bamax / 6 * (1 + 1 / 16) * (1 + 1e-6))
    assert np.all(unit >= bamax / 6 * (1 - 1 / 16) * (1 - 1e-6))


# ---------------------------------------------------------------- activations

@pytest.mark.parametrize("t", [-30.0, -4.0, -1.0, -1e-3, 0.5, 1.0, 3.0, 17.0])
def test_activation_identities(t):
    # SiLU(t) = t*sigmoid(t) = t/2 * (1 + tanh(t/2)); act(t) - act(-t) = t for
    # both SiLU and the tanh GeLU; GeLU-tanh stays within 1e-3 of erf GeLU.
    s = oracle.silu(t)
    e = math.exp(t)
    assert s == pytest.approx(t * e / (1.0 + e), rel=1e-13, abs=1e-300)
    if abs(t) <= 8:
        assert s == pytest.approx(0.5 * t * (1.0 + math.tanh(t / 2.0)), rel=1e-13)
    assert s - oracle.silu(-t) == pytest.approx(t, rel=1e-13, abs=1e-15)
    g = oracle.gelu_tanh(t)
    assert g - oracle.gelu_tanh(-t) == pytest.approx(t, rel=1e-13, abs=1e-15)
    assert abs(g - 0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0)))) < 1e-3


def test_activations_vanish_at_zero():
    assert oracle.silu(0.0) == 0.0
    assert oracle.gelu_tanh(0.0) == 0.0


# ---------------------------------------------------------------- GEMV / FFN

def _exact_gemv(xi, W_exact, scale2):
    """Hand-expanded sum with exact rationals: y[m][n] = sum_k x*w."""
    M, K = len(xi), len(xi[0])
    N = len(W_exact)
    return [[sum(Fraction(int(xi[m][k])) * W_exact[n][k] for k in range(K)) for n in range(N)]
            for m in range(M)]


def _bf16_bits_of(values):
    t = torch.tensor(values, dtype=torch.float64).float().bfloat16()
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (2, 48, 32), (3, 16, 32), (3, 48, 16)])
def test_gemv_brute_force_tiny(M, N, K):
    rng = np.random.default_rng(100 + M * N + K)
    j = -4
    W, codes, scales = representable_weight(N, K, j, rng)
    W_exact = [[Fraction(float(v)) for v in row] for row in W]
    xi = rng.integers(-8, 9, size=(M, K))
    x_bits = _bf16_bits_of(xi.astype(np.float64))
    c2, s2, scale2 = oracle.quantize(W)
    y = oracle.gemv_f64(x_bits, c2, s2, scale2, N)
    exact = _exact_gemv(xi, W_exact, scale2)
    for m in range(M):
        for n in range(N):
            assert Fraction(float(y[m, n])) == exact[m][n], (m, n)
    yb = oracle.gemv(x_bits, c2, s2, scale2, N)
    want = _bf16_bits_of([[float(exact[m][n]) for n in range(N)] for m in range(M)])
    np.testing.assert_array_equal(yb, want)


def test_gemv_scale2_power_of_two_scales_exactly():
    rng = np.random.default_rng(11)
    W = (rng.standard_normal((32, 64)) * 0.02).astype(np.float32)
    codes, scales, s2 = oracle.quantize(W)
    x = _bf16_bits_of(rng.standard_normal((2, 64)))
    a = oracle.gemv_f64(x, codes, scales, s2, 32)
    for k in (-3, 5):
        b = oracle.gemv_f64(x, codes, scales, np.float32(s2 * 2.0 ** k), 32)
        np.testing.assert_array_equal(b, a * 2.0 ** k)


def test_gemv_row_permutation_and_zero_inputs():
    rng = np.random.default_rng(12)
    W = (rng.standard_normal((48, 64)) * 0.02).astype(np.float32)
    codes, scales, s2 = oracle.quantize(W)
    x = _bf16_bits_of(rng.standard_normal((5, 64)))
    y = oracle.gemv(x, codes, scales, s2, 48)
    perm = [3, 0, 4, 1, 2]
    np.testing.assert_array_equal(oracle.gemv(x[perm], codes, scales, s2, 48), y[perm])
    z = oracle.gemv(np.zeros_like(x), codes, scales, s2, 48)
    assert np.all((z & 0x7FFF) == 0)
    zc, zs, z2 = oracle.quantize(np.zeros((48, 64), np.float32))
    assert np.all((oracle.gemv(x, zc, zs, z2, 48) & 0x7FFF) == 0)


@pytest.mark.parametrize("act", [oracle.ACT_SILU, oracle.ACT_GELU_TANH])
def test_ffn_zero_gate_gives_zero(act):
    rng = np.random.default_rng(13)
    H, I = 32, 48
    x = _bf16_bits_of(rng.standard_normal((2, H)))
    gate = oracle.quantize(np.zeros((I, H), np.float32))
    up = oracle.quantize((rng.standard_normal((I, H)) * 0.02).astype(np.float32))
    down = oracle.quantize((rng.standard_normal((H, I)) * 0.02).astype(np.float32))
    h = oracle.ffn_hidden(x, I, gate, up, act)
    assert np.all((h & 0x7FFF) == 0)
    out = oracle.ffn(x, I, gate, up, down, act)
    assert np.all((out & 0x7FFF) == 0)


@pytest.mark.parametrize("act", [oracle.ACT_SILU, oracle.ACT_GELU_TANH])
def test_ffn_brute_force_tiny(act):
    # gate/up/down exactly representable, x small integers: g and u are exact
    # rationals rounded once to bf16; h is checked against an independent
    # statement of the activation (SiLU through tanh, GeLU from its definition
    # with Python's math) to one bf16 step; out = bf16 of the exact down sum
    # over the oracle's own h.
    rng = np.random.default_rng(14 + act)
    M, H, I = 2, 32, 48
    Wg, _, _ = representable_weight(I, H, -13, rng)   # keeps g, u of order one
    Wu, _, _ = representable_weight(I, H, -12, rng)
    Wd, _, _ = representable_weight(H, I, -6, rng)
    xi = rng.integers(-4, 5, size=(M, H))
    x = _bf16_bits_of(xi.astype(np.float64))
    gq, uq, dq = oracle.quantize(Wg), oracle.quantize(Wu), oracle.quantize(Wd)
    h = oracle.ffn_hidden(x, I, gq, uq, act)
    g_ex = _exact_gemv(xi, [[Fraction(float(v)) for v in r] for r in Wg], 1)
    u_ex = _exact_gemv(xi, [[Fraction(float(v)) for v in r] for r in Wu], 1)
    hv = oracle.bf16_bits_to_f64(h)
    for m in range(M):
        for i in range(I):
            g = float(oracle.bf16_bits_to_f64(_bf16_bits_of([float(g_ex[m][i])]))[0])
            u = float(oracle.bf16_bits_to_f64(_bf16_bits_of([float(u_ex[m][i])]))[0])
            if act == oracle.ACT_SILU:
                # two cancellation-free forms of t*sigmoid(t), one per sign
                a = 0.5 * g * (1.0 + math.tanh(0.5 * g)) if g >= 0 else \
                    g * math.exp(g) / (1.0 + math.exp(g))
            else:
                a = 0.5 * g * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))
            want = a * u
            assert abs(hv[m, i] - want) <= abs(want) * 2 ** -8 + 1e-30, (m, i)
    out = oracle.ffn(x, I, gq, uq, dq, act)
    d_ex = [[sum(Fraction(float(hv[m, i])) * Fraction(float(Wd[n, i])) for i in range(I))
             for n in range(H)] for m in range(M)]
    want = _bf16_bits_of([[float(d_ex[m][n]) for n in range(H)] for m in range(M)])
    np.testing.assert_array_equal(out, want)


def test_nibble_order_low_nibble_is_even_element():
    # One nonzero element at an odd position must come out of the odd slot.
    W = np.zeros((1, 16), np.float32)
    W[0, 3] = 2688.0
    codes, scales, s2 = oracle.quantize(W)
    assert codes[0, 1] == 0x70 and codes[0, 0] == 0 and scales[0, 0] == 0x7E
    x = np.zeros((1, 16), np.uint16)
    x[0, 3] = 0x3F80  # 1.0
    assert oracle.gemv_f64(x, codes, scales, s2, 1)[0, 0] == 2688.0
    x[0, 3] = 0
    x[0, 2] = 0x3F80
    assert oracle.gemv_f64(x, codes, scales, s2, 1)[0, 0] == 0.0


def test_array_forms_agree_with_scalar_functions():
    rng = np.random.default_rng(21)
    v = np.concatenate([rng.standard_normal(500) * 10.0 ** rng.integers(-5, 5, 500),
                        [0.0, -0.0, 1 + 2 ** -8 + 2 ** -30]])
    b = oracle.bf16_from_double_array(v)
    assert [oracle.bf16_from_double(float(t)) for t in v] == list(b)
    for act, fn in ((oracle.ACT_SILU, oracle.silu), (oracle.ACT_GELU_TANH, oracle.gelu_tanh)):
        np.testing.assert_array_equal(oracle.act_array(v, act), [fn(float(t)) for t in v])


@pytest.mark.parametrize("t", [-12.0, -9.5, -7.0, -5.0, -3.0, -1.0, -0.01, 0.3, 2.0, 6.0, 11.0])
def test_activations_match_high_precision_evaluation(t):
    # Both activations in 150-digit decimal arithmetic straight from their
    # definitions (tanh through exp); the oracle must agree to ~1e-14
    # relative everywhere, including the far negative tails where a literal
    # 1 + tanh(z) in double precision cancels.
    from decimal import Decimal, getcontext
    getcontext().prec = 150
    T = Decimal(t)
    pi = Decimal("3.14159265358979323846264338327950288419716939937510")
    z = (Decimal(2) / pi).sqrt() * (T + Decimal("0.044715") * T ** 3)
    tanh = ((2 * z).exp() - 1) / ((2 * z).exp() + 1)
    gelu = Decimal("0.5") * T * (1 + tanh)
    silu = T / (1 + (-T).exp())
    assert oracle.gelu_tanh(t) == pytest.approx(float(gelu), rel=1e-14, abs=1e-300)
    assert oracle.silu(t) == pytest.approx(float(silu), rel=1e-14, abs=1e-300)
