"""Pins of the oracle's block-scaled FP8 path (the dense-FFN page's native FP8
arm: E4M3 bytes [N, K] and an FP32 grid [ceil(N/128), ceil(K/128)], weight =
e4m3(q[n][k]) * grid[n/128][k/128]).

Every expected value here comes from something other than the oracle: torch's
float8_e4m3fn converter for the byte values, exact rational sums (Fraction),
an independent bf16 rounding of rationals, and the NVFP4 oracle on weights
that both formats represent exactly.  Mistakes a plausible implementation
could make -- a transposed grid index, a 64- instead of 128-wide block, a
dropped scale, the down projection over x -- change the results these pins
compare."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

from test_lora_oracle_pins import bf16_rne, bits_to_fr


def e4m3_fr(b):
    """Exact value of an E4M3 byte through torch's converter."""
    t = torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    return Fraction(float(t.item()))


E4M3_TABLE = [e4m3_fr(b) if b not in (0x7F, 0xFF) else None for b in range(256)]


def finite_codes(rng, shape, lo=0, hi=256):
    """Random E4M3 bytes without the two NaN encodings."""
    q = rng.integers(lo, hi, size=shape).astype(np.uint8)
    q[(q == 0x7F) | (q == 0xFF)] = 0x7E
    return q


def small_x(rng, shape, lo=-4, hi=4):
    """bf16-exact small integers (as bit patterns)."""
    v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_gemv(x_bits, q, bs):
    M, K = x_bits.shape
    N = q.shape[0]
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        xs = [bits_to_fr(x_bits[m, k]) for k in range(K)]
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                if xs[k]:
                    s += xs[k] * E4M3_TABLE[q[n, k]] * Fraction(float(bs[n // 128, k // 128]))
            out[m][n] = s
    return out


def pow2_grid(rng, shape, lo=-6, hi=3):
    return (2.0 ** rng.integers(lo, hi + 1, size=shape)).astype(np.float32)


def test_e4m3_table_is_torchs():
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        assert Fraction(oracle.e4m3_decode(b)) == E4M3_TABLE[b], hex(b)


def test_grid_shape_rounds_up():
    assert oracle.fp8_grid_shape(128, 128) == (1, 1)
    assert oracle.fp8_grid_shape(129, 257) == (2, 3)
    assert oracle.fp8_grid_shape(5120, 17408) == (40, 136)


def test_dequantize_block_index():
    """Every cell of a 3 x 3 grid holds a distinct power of two, so a
    transposed index, a 64-wide block or an off-by-one boundary moves some
    weight to another cell's scale."""
    rng = np.random.default_rng(0)
    N, K = 300, 290
    q = finite_codes(rng, (N, K))
    bs = np.array([[2.0 ** (3 * i + j - 4) for j in range(3)] for i in range(3)], np.float32)
    w = oracle.fp8_dequantize(q, bs)
    for n in (0, 127, 128, 255, 256, 299):
        for k in (0, 63, 64, 127, 128, 200, 256, 289):
            assert Fraction(w[n, k]) == E4M3_TABLE[q[n, k]] * Fraction(float(bs[n // 128, k // 128]))


@pytest.mark.parametrize("N,K,M", [(130, 200, 2), (7, 384, 1), (256, 136, 3)])
def test_gemv_exact_sums(N, K, M):
    """Dyadic inputs (small-integer x, E4M3 bytes, power-of-two scales) make
    the double sum exact: f64 output == the rational sum, bf16 output == its
    independent round-to-nearest-even."""
    rng = np.random.default_rng(N + K + M)
    x = small_x(rng, (M, K))
    q = finite_codes(rng, (N, K), 0, 0x60)  # magnitudes up to 2^4 keep sums well inside 2^53
    q |= (rng.integers(0, 2, size=(N, K)) * 0x80).astype(np.uint8)
    bs = pow2_grid(rng, oracle.fp8_grid_shape(N, K))
    ref = exact_gemv(x, q, bs)
    got64 = oracle.gemv_fp8_f64(x, q, bs)
    got = oracle.gemv_fp8(x, q, bs)
    for m in range(M):
        for n in range(N):
            assert Fraction(got64[m, n]) == ref[m][n], (m, n)
            assert bits_to_fr(got[m, n]) == bf16_rne(ref[m][n]), (m, n)


def test_gemv_rounds_once_from_the_exact_sum():
    """A sum that lies exactly halfway between two bf16 values rounds to the
    even one (257 -> 256, 259 -> 260): one rounding, from the exact value."""
    x = small_x(np.random.default_rng(0), (1, 2), 1, 1)  # x = [1, 1]
    q = np.array([[0x78, 0x38], [0x78, 0x48]], np.uint8)  # 256 + 1, 256 + 4 (e4m3)
    bs = np.ones((1, 1), np.float32)
    assert [E4M3_TABLE[b] for b in (0x78, 0x38, 0x48)] == [256, 1, 4]
    y = oracle.gemv_fp8(x, q, bs)
    assert bits_to_fr(y[0, 0]) == 256 and bits_to_fr(y[0, 1]) == 260


def test_uniform_grid_is_a_per_tensor_scale():
    """A per-tensor scalar broadcast to the whole grid scales every output by
    exactly that scalar (a power of two here, so the bf16 results move by the
    same power of two)."""
    rng = np.random.default_rng(3)
    N, K, M = 200, 300, 2
    x = small_x(rng, (M, K))
    q = finite_codes(rng, (N, K))
    ones = np.ones(oracle.fp8_grid_shape(N, K), np.float32)
    y1 = oracle.gemv_fp8_f64(x, q, ones)
    y8 = oracle.gemv_fp8_f64(x, q, ones * np.float32(0.125))
    assert np.array_equal(y8, y1 * 0.125)


def test_fp8_agrees_with_nvfp4_on_shared_weights():
    """An NVFP4 weight with unit block scales and scale2 = 2^-3 equals an FP8
    weight with the same E2M1 magnitudes as E4M3 bytes and a uniform 2^-3 grid
    (every E2M1 value is an E4M3 value): the two oracle paths agree bit for
    bit, through different code."""
    rng = np.random.default_rng(4)
    N, K, M = 160, 256, 3
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)  # e4m3 1.0
    e2m1 = {0: 0x00, 1: 0x30, 2: 0x38, 3: 0x3C, 4: 0x40, 5: 0x44, 6: 0x48, 7: 0x4C}
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(N, K)
    q = np.array([[e2m1[int(c) & 7] | (0x80 if c & 8 else 0) for c in row] for row in nib],
                 np.uint8)
    for c, b in e2m1.items():
        assert Fraction(oracle.e2m1_decode(c)) == E4M3_TABLE[b]
    x = small_x(rng, (M, K))
    bs = np.full(oracle.fp8_grid_shape(N, K), 0.125, np.float32)
    assert np.array_equal(oracle.gemv_fp8(x, q, bs), oracle.gemv(x, codes, scales, 0.125, N))


def _fp8_ffn_case(H=40, I=136, M=2, seed=5):
    rng = np.random.default_rng(seed)
    proj = []
    for n, k in ((I, H), (I, H), (H, I)):
        q = finite_codes(rng, (n, k), 0, 0x58)
        q |= (rng.integers(0, 2, size=(n, k)) * 0x80).astype(np.uint8)
        proj.append((q, pow2_grid(rng, oracle.fp8_grid_shape(n, k), -7, -3)))
    x = small_x(rng, (M, H), -3, 3)
    return x, proj


@pytest.mark.parametrize("act", [oracle.ACT_SILU, oracle.ACT_GELU_TANH])
def test_ffn_fp8_brute_force(act):
    """g, u from exact sums with the independent bf16 rounding; h from the
    oracle's pinned activation; out from the exact down sum over that h."""
    x, (g, u, d) = _fp8_ffn_case()
    gx, ux = exact_gemv(x, *g), exact_gemv(x, *u)
    M, I = len(gx), len(gx[0])
    h_ref = np.zeros((M, I), np.uint16)
    for m in range(M):
        for i in range(I):
            gv = float(bf16_rne(gx[m][i]))
            uv = float(bf16_rne(ux[m][i]))
            h_ref[m, i] = oracle.bf16_from_double(oracle.act(gv, act) * uv)
    h = oracle.ffn_fp8_hidden(x, g, u, act)
    assert np.array_equal(h, h_ref)
    od = exact_gemv(h_ref, *d)
    out = oracle.ffn_fp8(x, g, u, d, act)
    for m in range(M):
        for n in range(len(od[0])):
            assert bits_to_fr(out[m, n]) == bf16_rne(od[m][n]), (m, n)


def test_ffn_fp8_distinguishes_misplaced_steps():
    """A transposed down grid or the down projection taken over x (H == I
    here) gives a different output."""
    x, (g, u, d) = _fp8_ffn_case(H=256, I=256, M=1, seed=9)
    d = (d[0], np.array([[1.0, 0.25], [0.5, 2.0]], np.float32))
    out = oracle.ffn_fp8(x, g, u, d)
    h = oracle.ffn_fp8_hidden(x, g, u)
    assert np.array_equal(out, oracle.gemv_fp8(h, *d))
    assert not np.array_equal(out, oracle.gemv_fp8(h, d[0], d[1].T.copy()))
    assert not np.array_equal(out, oracle.gemv_fp8(x, *d))
