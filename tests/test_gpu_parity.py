"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: quantise (codes, scales, scale2) and the repack/unpack round trip.
Floating point: every bf16 output within |gpu - oracle| <= 1e-2 * max(1, |oracle|),
and, tighter, inside its valid rounding interval (parity_checks): bit-exact
wherever the specified bf16 rounding is determined by the exact value and the
accumulation error bound.  The oracle always quantises the weights itself; the
GPU path uses its own quantiser, so a parity pass covers quantise -> repack ->
kernels end to end.
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_gb300 import ffi, synth

import parity_checks as pc
from test_oracle_pins import representable_weight

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ffi.load(build_if_missing=True)
    return torch.device("cuda:0")


def assert_close(got, ref_bits, what=""):
    g = got.float().cpu().double().numpy()
    r = oracle.bf16_bits_to_f64(ref_bits)
    assert g.shape == r.shape
    err = np.abs(g - r)
    bound = TOL * np.maximum(1.0, np.abs(r))
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of tolerance, first {bad[:5].tolist()}, "
                           f"max err {err.max():.3e}")
    return float(err.max())


def gpu_quant(w, dev):
    return ffi.nvfp4_quantize(w.to(dev))


def check_quant(w, dev):
    c, s, s2 = gpu_quant(w, dev)
    if w.dtype == torch.bfloat16:
        rc, rs, rs2 = oracle.quantize_bf16(synth.bf16_bits(w))
    else:
        rc, rs, rs2 = oracle.quantize(w.numpy())
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert np.float32(s2) == np.float32(rs2)
    return (c, s, s2), (rc, rs, rs2)


# ------------------------------------------------------------------ quantise

@pytest.mark.parametrize("N,K", [(256, 512), (200, 272), (17, 48), (1, 16), (1024, 4096)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_bit_exact(dev, N, K, dtype):
    w = synth.weights_f32(N, K, seed=N * 7 + K).to(dtype)
    check_quant(w, dev)


@pytest.mark.parametrize("j", [-9, 0, 3])
def test_quantize_representable_round_trip(dev, j):
    rng = np.random.default_rng(40 + j)
    W, codes, scales = representable_weight(32, 128, j, rng)
    (c, s, s2), _ = check_quant(torch.from_numpy(W), dev)
    np.testing.assert_array_equal(c.cpu().numpy(), codes)
    np.testing.assert_array_equal(s.cpu().numpy(), scales)
    assert s2 == 2.0 ** j


def test_quantize_special_values(dev):
    s = 448.0
    row = [6 * s, 0.25 * s, 0.75 * s, 1.25 * s, 1.75 * s, 2.5 * s, 3.5 * s, 5 * s,
           -0.25 * s, -0.75 * s, -2.5 * s, -5 * s, 0.0, -0.0, -0.1 * s, -6 * s]
    W = np.zeros((4, 64), np.float32)
    W[0, :16] = row
    W[1, 16:32] = -0.0                    # a zero block with negative zeros
    W[2, 32:48] = 1e-3                    # equal magnitudes
    W[3, 48:64] = np.linspace(-1e-6, 1e-6, 16)  # tiny next to a large amax
    check_quant(torch.from_numpy(W), dev)
    check_quant(torch.zeros(8, 32), dev)
    big = (synth.weights_f32(16, 64, seed=3) * 1e30)
    check_quant(big, dev)
    small = (synth.weights_f32(16, 64, seed=4) * 1e-30)
    check_quant(small, dev)


# ------------------------------------------------------------------ repack

@pytest.mark.parametrize("N,K", [(256, 512), (200, 272), (130, 80), (5120, 1024)])
def test_repack_unpack_round_trip(dev, N, K):
    g = torch.Generator().manual_seed(N + K)
    codes = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.uint8)
    scales = torch.randint(0, 127, (N, K // 16), generator=g, dtype=torch.uint8)
    p = ffi.nvfp4_repack(codes.to(dev), scales.to(dev), N, K)
    c2, s2 = ffi.nvfp4_unpack(p, N, K)
    assert torch.equal(c2.cpu(), codes) and torch.equal(s2.cpu(), scales)
    if N % 256 == 0 and K % 256 == 0:
        # a pure permutation: same multiset of bytes
        a = torch.bincount(torch.cat([codes.flatten(), scales.flatten()]).long(), minlength=256)
        b = torch.bincount(p.cpu().long(), minlength=256)
        assert torch.equal(a, b)


# ------------------------------------------------------------------ GEMV

def run_gemv_case(dev, N, K, M, seed=0, outliers=0.0, x_scale=1.0):
    w = synth.weights_f32(N, K, seed=1000 + seed)
    x = synth.activations_bf16(M, K, seed=seed, outlier_frac=outliers)
    if x_scale != 1.0:
        x = (x.float() * x_scale).to(torch.bfloat16)
    (c, s, s2), (rc, rs, rs2) = check_quant(w, dev)
    p = ffi.nvfp4_repack(c, s, N, K)
    y = ffi.nvfp4_gemv(x.to(dev), p, s2, N)
    ref = oracle.gemv(synth.bf16_bits(x), rc, rs, rs2, N)
    err = assert_close(y, ref, f"gemv N={N} K={K} M={M}")
    pc.check_gemv(synth.bf16_bits(y), synth.bf16_bits(x), (rc, rs, rs2), N, f"gemv N={N} K={K} M={M}")
    return err, y, p, x, s2


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_gemv_all_m(dev, M):
    run_gemv_case(dev, 384, 1024, M, seed=M)


@pytest.mark.parametrize("N,K,M", [(200, 272, 3), (130, 80, 1), (16, 16, 2), (1, 2048, 9),
                                   (4096, 4096, 1), (1000, 2000, 16), (2048, 6144, 8),
                                   (300, 21504, 4)])
def test_gemv_shapes(dev, N, K, M):
    run_gemv_case(dev, N, K, M, seed=N + K + M)


def test_gemv_extreme_activation_scales(dev):
    run_gemv_case(dev, 256, 512, 2, seed=5, x_scale=2.0 ** 60)
    run_gemv_case(dev, 256, 512, 2, seed=6, x_scale=2.0 ** -60)
    run_gemv_case(dev, 256, 512, 10, seed=7, outliers=0.01)


def test_gemv_deterministic_and_reusable_workspace(dev):
    N, K, M = 2048, 4096, 5
    _, y, p, x, s2 = run_gemv_case(dev, N, K, M, seed=9)
    ws = ffi.workspace(ffi.nvfp4_gemv_workspace_bytes(M, N, K), dev)
    a = ffi.nvfp4_gemv(x.to(dev), p, s2, N, ws=ws)
    b = ffi.nvfp4_gemv(x.to(dev), p, s2, N, ws=ws)
    assert torch.equal(a, b) and torch.equal(a, y)
    assert ffi.nvfp4_workspace_status(ws) == 0


@pytest.mark.parametrize("M", [2, 5, 12])
def test_gemv_token_rows_are_independent(dev, M):
    """Permuting the token rows permutes the outputs bit for bit (each row is
    scaled and accumulated on its own), and the FFN on a permutation of x is
    the same permutation of its output."""
    N, K = 1024, 2048
    w = synth.weights_f32(N, K, seed=31)
    c, s, s2 = gpu_quant(w, dev)
    p = ffi.nvfp4_repack(c, s, N, K)
    x = synth.activations_bf16(M, K, seed=32, outlier_frac=0.05).to(dev)
    perm = torch.from_numpy(np.random.default_rng(M).permutation(M)).to(dev)
    y = ffi.nvfp4_gemv(x, p, s2, N)
    yp = ffi.nvfp4_gemv(x[perm].contiguous(), p, s2, N)
    assert torch.equal(yp, y[perm])
    H, I = 256, 512
    gu, dn, q, _ = build_ffn(dev, H, I)
    xf = synth.activations_bf16(M, H, seed=33, outlier_frac=0.05).to(dev)
    o = ffi.ffn_swiglu_nvfp4(xf, gu, q[0][2], q[1][2], dn, q[2][2], I)
    op = ffi.ffn_swiglu_nvfp4(xf[perm].contiguous(), gu, q[0][2], q[1][2], dn, q[2][2], I)
    assert torch.equal(op, o[perm])


@pytest.mark.slow
@pytest.mark.parametrize("N,K,M", [(5120, 17408, 1), (5120, 17408, 8), (17408, 5120, 16),
                                   (4096, 21504, 1), (65536, 4096, 16), (21504, 5376, 3)])
def test_gemv_full_size(dev, N, K, M):
    run_gemv_case(dev, N, K, M, seed=11, outliers=0.01 if M > 1 else 0.0)


@pytest.mark.slow
def test_gemv_largest_sweep_shape_sampled_rows(dev):
    """N=65536, K=21504 (the top of the standalone GEMV sweep), M=2: the oracle
    quantises the whole weight, the GPU runs the GEMV on those codes, and 640
    rows (both ends and a seeded sample) are checked against the oracle's GEMV
    of just those rows."""
    N, K, M = 65536, 21504, 2
    w = synth.weights_f32(N, K, seed=77)
    rc, rs, rs2 = oracle.quantize(w.numpy())
    del w
    p = ffi.nvfp4_repack(torch.from_numpy(rc).to(dev), torch.from_numpy(rs).to(dev), N, K)
    x = synth.activations_bf16(M, K, seed=5, outlier_frac=0.01)
    y = ffi.nvfp4_gemv(x.to(dev), p, float(rs2), N)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N),
                                     rng.choice(N, 512, replace=False)]))
    ref = oracle.gemv(synth.bf16_bits(x), rc[rows], rs[rows], rs2, len(rows))
    ys = y[:, torch.from_numpy(rows).to(dev)]
    assert_close(ys, ref, "gemv 65536x21504 sampled rows")
    pc.check_gemv(synth.bf16_bits(ys), synth.bf16_bits(x), (rc[rows], rs[rows], rs2), len(rows),
                  "gemv 65536x21504 sampled rows")


def test_gemv_many_ranges_per_cta_sampled_rows(dev):
    """N=65536, K=10240, M=16: with two token groups the staged token rows
    limit a range to 11 steps, so each CTA walks about seven ranges and up to
    nine partial segments.  Some CTAs therefore pass the publisher warp's
    eight events and count the rest in-warp, and resolve pending tiles early.
    The oracle quantises the whole weight; 640 rows are checked against its
    GEMV of just those rows."""
    N, K, M = 65536, 10240, 16
    w = synth.weights_f32(N, K, seed=78)
    rc, rs, rs2 = oracle.quantize(w.numpy())
    del w
    p = ffi.nvfp4_repack(torch.from_numpy(rc).to(dev), torch.from_numpy(rs).to(dev), N, K)
    x = synth.activations_bf16(M, K, seed=6, outlier_frac=0.01)
    y = ffi.nvfp4_gemv(x.to(dev), p, float(rs2), N)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N),
                                     rng.choice(N, 512, replace=False)]))
    ref = oracle.gemv(synth.bf16_bits(x), rc[rows], rs[rows], rs2, len(rows))
    ys = y[:, torch.from_numpy(rows).to(dev)]
    assert_close(ys, ref, "gemv 65536x10240 M=16 sampled rows")
    pc.check_gemv(synth.bf16_bits(ys), synth.bf16_bits(x), (rc[rows], rs[rows], rs2), len(rows),
                  "gemv 65536x10240 M=16 sampled rows")


# ------------------------------------------------------------------ FFN

def build_ffn(dev, H, I, layer=0):
    w = [synth.weights_f32(I, H, seed=synth.layer_seed(layer, synth.GATE)),
         synth.weights_f32(I, H, seed=synth.layer_seed(layer, synth.UP)),
         synth.weights_f32(H, I, seed=synth.layer_seed(layer, synth.DOWN))]
    q, rq = zip(*[check_quant(t, dev) for t in w])
    gu = ffi.nvfp4_repack_gate_up(q[0][0], q[0][1], q[1][0], q[1][1], I, H)
    dn = ffi.nvfp4_repack(q[2][0], q[2][1], H, I)
    return gu, dn, q, rq


def run_ffn_case(dev, H, I, M, act, outliers=0.0, seed=0):
    """FFN parity.  h must lie in its valid rounding interval and match the
    oracle bit for bit wherever the rounding is determined (parity_checks);
    out likewise against the oracle's down projection of the GPU's own h; and
    end to end against the oracle's FFN, where elements may leave the
    tolerance only through the legitimately different h (at most 0.5%, a
    backstop: the count is printed)."""
    gu, dn, q, rq = build_ffn(dev, H, I)
    x = synth.activations_bf16(M, H, seed=seed, outlier_frac=outliers)
    xb = synth.bf16_bits(x)
    ws = ffi.workspace(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), dev)
    out = ffi.ffn_swiglu_nvfp4(x.to(dev), gu, q[0][2], q[1][2], dn, q[2][2], I, act, ws=ws)
    torch.cuda.synchronize()
    h_bits = synth.bf16_bits(ffi.ffn_hidden_view(ws, M, I))
    sh = pc.check_hidden(h_bits, xb, rq[0], rq[1], act, f"h H={H} I={I} M={M} act={act}")
    out_bits = synth.bf16_bits(out)
    so = pc.check_gemv(out_bits, h_bits, rq[2], H, f"out H={H} I={I} M={M} act={act}")
    err = assert_close(out, oracle.gemv(h_bits, rq[2][0], rq[2][1], rq[2][2], H),
                       f"ffn down(h_gpu) H={H} I={I} M={M} act={act}")
    ref = oracle.ffn(xb, I, rq[0], rq[1], rq[2], act)
    n_out = pc.count_beyond_tolerance(out_bits, ref)
    print(f"PARITY ffn H={H} I={I} M={M} act={act} outliers={outliers}: "
          f"h {sh['n']} elements, {sh['determined']} determined, {sh['differs']} differ from "
          f"the oracle; out {so['n']}, {so['determined']} determined, {so['differs']} differ "
          f"from down(h_gpu); end to end {n_out} beyond 1e-2")
    assert n_out <= 0.005 * ref.size, f"ffn end to end: {n_out} of {ref.size} out of tolerance"
    assert ffi.nvfp4_workspace_status(ws) == 0
    return err, n_out


def _small_scale_weight(N, K, j, rng):
    """Canonical NVFP4 codes/scales whose every dot product with small-integer
    activations is exact in fp32: E4M3 scales from {0.5, 1, 1.5, 2}, any
    E2M1 code, scale2 = 2^j (products are multiples of 2^(j-2), sums far
    below 2^24 of them)."""
    scales = rng.choice(np.array([0x30, 0x38, 0x3C, 0x40], np.uint8), size=(N, K // 16))
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    return codes, scales, 2.0 ** j


@pytest.mark.parametrize("M", [1, 3, 12])
def test_ffn_exact_intermediates_canary(dev, M):
    """x holds small integers and the gate/up weights small scales, so g and u
    are exact on both sides (every partial sum is representable in fp32) and
    their bf16 roundings must agree bit for bit; h must then match the oracle
    everywhere except within the kernel's fp32 activation error of a bf16 tie.
    A truncating or round-toward-zero bf16 conversion anywhere fails this."""
    H, I = 1024, 2048
    rng = np.random.default_rng(100 + M)
    gate = _small_scale_weight(I, H, -6, rng)
    up = _small_scale_weight(I, H, -6, rng)
    down = _small_scale_weight(H, I, -8, rng)
    xt = torch.from_numpy(rng.integers(-3, 4, size=(M, H)).astype(np.float32)).to(torch.bfloat16)
    xb = synth.bf16_bits(xt)
    gu = ffi.nvfp4_repack_gate_up(*(torch.from_numpy(t).to(dev) for t in
                                    (gate[0], gate[1], up[0], up[1])), I, H)
    dn = ffi.nvfp4_repack(torch.from_numpy(down[0]).to(dev), torch.from_numpy(down[1]).to(dev),
                          H, I)
    ws = ffi.workspace(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), dev)
    for act in (ffi.NVFP4_ACT_SILU, ffi.NVFP4_ACT_GELU_TANH):
        out = ffi.ffn_swiglu_nvfp4(xt.to(dev), gu, gate[2], up[2], dn, down[2], I, act, ws=ws)
        torch.cuda.synchronize()
        h_bits = synth.bf16_bits(ffi.ffn_hidden_view(ws, M, I))
        sh = pc.check_hidden(h_bits, xb, gate, up, act, f"canary h M={M} act={act}", acc_eps=0.0)
        assert sh["determined"] >= 0.99 * sh["n"], sh
        so = pc.check_gemv(synth.bf16_bits(out), h_bits, down, H, f"canary out M={M} act={act}")
        print(f"PARITY canary M={M} act={act}: h {sh}, out {so}")
    assert ffi.nvfp4_workspace_status(ws) == 0


def test_ffn_tiny_config(dev):
    run_ffn_case(dev, 256, 512, 1, ffi.NVFP4_ACT_SILU)


@pytest.mark.parametrize("M,act", [(1, ffi.NVFP4_ACT_SILU), (5, ffi.NVFP4_ACT_GELU_TANH),
                                   (12, ffi.NVFP4_ACT_SILU)])
def test_gate_up_entry_point(dev, M, act):
    H, I = 1024, 2816
    gu, dn, q, rq = build_ffn(dev, H, I)
    x = synth.activations_bf16(M, H, seed=M, outlier_frac=0.01)
    h = ffi.ffn_gate_up_nvfp4(x.to(dev), gu, q[0][2], q[1][2], I, act)
    h_ref = oracle.ffn_hidden(synth.bf16_bits(x), I, rq[0], rq[1], act)
    assert_close(h, h_ref, "gate/up h")
    # the same kernel inside the full FFN leaves the identical h in its workspace
    ws = ffi.workspace(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), dev)
    ffi.ffn_swiglu_nvfp4(x.to(dev), gu, q[0][2], q[1][2], dn, q[2][2], I, act, ws=ws)
    assert torch.equal(ffi.ffn_hidden_view(ws, M, I), h)
    # and finishing with the standalone GEMV reproduces the full FFN bit for bit
    out = ffi.nvfp4_gemv(h, dn, q[2][2], H)
    full = ffi.ffn_swiglu_nvfp4(x.to(dev), gu, q[0][2], q[1][2], dn, q[2][2], I, act)
    assert torch.equal(out, full)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 9, 16])
@pytest.mark.parametrize("act", [ffi.NVFP4_ACT_SILU, ffi.NVFP4_ACT_GELU_TANH])
def test_ffn_batch_m(dev, M, act):
    run_ffn_case(dev, 512, 1536, M, act, outliers=0.01 if M >= 4 else 0.0, seed=M)


@pytest.mark.parametrize("H,I,M", [(192, 400, 3), (320, 272, 1), (4096, 12288, 2),
                                   (4096, 12288, 3)])
def test_ffn_shapes(dev, H, I, M):
    run_ffn_case(dev, H, I, M, ffi.NVFP4_ACT_SILU, seed=H + I)


def test_ffn_zero_gate_and_zero_input(dev):
    H, I, M = 256, 512, 2
    zero = ffi.nvfp4_quantize(torch.zeros(I, H, device=dev))
    up = ffi.nvfp4_quantize(synth.weights_f32(I, H, seed=1).to(dev))
    dn = ffi.nvfp4_quantize(synth.weights_f32(H, I, seed=2).to(dev))
    gu = ffi.nvfp4_repack_gate_up(zero[0], zero[1], up[0], up[1], I, H)
    d = ffi.nvfp4_repack(dn[0], dn[1], H, I)
    x = synth.activations_bf16(M, H, seed=3).to(dev)
    for act in (ffi.NVFP4_ACT_SILU, ffi.NVFP4_ACT_GELU_TANH):
        out = ffi.ffn_swiglu_nvfp4(x, gu, zero[2], up[2], d, dn[2], I, act)
        assert torch.count_nonzero(out.float()) == 0
    gu2 = ffi.nvfp4_repack_gate_up(up[0], up[1], up[0], up[1], I, H)
    out = ffi.ffn_swiglu_nvfp4(torch.zeros_like(x), gu2, up[2], up[2], d, dn[2], I)
    assert torch.count_nonzero(out.float()) == 0


@pytest.mark.slow
@pytest.mark.parametrize("M,act,outliers", [(1, ffi.NVFP4_ACT_SILU, 0.0),
                                            (8, ffi.NVFP4_ACT_GELU_TANH, 0.01),
                                            (16, ffi.NVFP4_ACT_SILU, 0.01)])
def test_ffn_full_size(dev, M, act, outliers):
    run_ffn_case(dev, 5120, 17408, M, act, outliers=outliers, seed=M)


@pytest.mark.slow
@pytest.mark.parametrize("M,act", [(1, ffi.NVFP4_ACT_SILU), (5, ffi.NVFP4_ACT_GELU_TANH),
                                   (12, ffi.NVFP4_ACT_SILU), (16, ffi.NVFP4_ACT_GELU_TANH)])
def test_ffn_large_dense_shape(dev, M, act):
    """The large dense FFN sweep's layer shape, H=5376, I=21504.  At M=16 the
    down kernel's token rows take ring space (three stages) so that each CTA
    keeps one range."""
    run_ffn_case(dev, 5376, 21504, M, act, outliers=0.0, seed=100 + M)


def test_error_codes_raise(dev):
    x = torch.zeros(65, 64, dtype=torch.bfloat16, device=dev)
    p = torch.zeros(4096, dtype=torch.uint8, device=dev)
    with pytest.raises(ffi.Nvfp4Error) as e:
        ffi.nvfp4_gemv(x, p, 1.0, 64)
    assert e.value.code == 4
    with pytest.raises(ffi.Nvfp4Error) as e:
        ffi.nvfp4_gemv(x[:2], p, 1.0, 64, ws=torch.zeros(16, dtype=torch.uint8, device=dev))
    assert e.value.code == 5


def test_one_workspace_serves_any_sequence_of_shapes(dev):
    """A workspace zero-filled once serves every later call, whatever its entry
    point and shape: each result equals the same call on a fresh workspace."""
    shapes = [(1, 2048, 6144), (8, 1024, 2816), (16, 512, 1536), (3, 4096, 1024), (1, 1024, 2816)]
    nbytes = max(max(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I),
                     ffi.nvfp4_gemv_workspace_bytes(M, H, I)) for M, H, I in shapes)
    shared = ffi.workspace(nbytes, dev)
    built = {}
    for rep in range(2):
        for M, H, I in shapes:
            if (H, I) not in built:
                built[(H, I)] = build_ffn(dev, H, I, layer=H % 7)
            gu, dn, q, _ = built[(H, I)]
            x = synth.activations_bf16(M, H, seed=M + rep, outlier_frac=0.01).to(dev)
            ref = ffi.ffn_swiglu_nvfp4(x, gu, q[0][2], q[1][2], dn, q[2][2], I)
            got = ffi.ffn_swiglu_nvfp4(x, gu, q[0][2], q[1][2], dn, q[2][2], I, ws=shared)
            assert torch.equal(got, ref), (M, H, I, rep)
            h = synth.activations_bf16(M, I, seed=M + 5, outlier_frac=0.01).to(dev)
            ref_y = ffi.nvfp4_gemv(h, dn, q[2][2], H)
            assert torch.equal(ffi.nvfp4_gemv(h, dn, q[2][2], H, ws=shared), ref_y), (M, H, I)
    assert ffi.nvfp4_workspace_status(shared) == 0



# ------------------------------------------------------------------ M = 17..64

@pytest.mark.parametrize("N,K,M", [(384, 1024, 17), (1000, 2000, 33), (256, 4096, 64),
                                   (4096, 5120, 24)])
def test_gemv_large_batches(dev, N, K, M):
    """M > 16 (verify batches, small prefill): groups of 16 rows and a rest."""
    run_gemv_case(dev, N, K, M, seed=M + N, outliers=0.01)


@pytest.mark.parametrize("M,act", [(17, ffi.NVFP4_ACT_SILU), (40, ffi.NVFP4_ACT_GELU_TANH),
                                   (64, ffi.NVFP4_ACT_SILU)])
def test_ffn_large_batches(dev, M, act):
    run_ffn_case(dev, 512, 1536, M, act, outliers=0.01, seed=M)


@pytest.mark.slow
def test_ffn_large_batch_full_size(dev):
    run_ffn_case(dev, 5120, 17408, 17, ffi.NVFP4_ACT_SILU, seed=17)


def test_large_batch_equals_its_groups_bit_for_bit(dev):
    """A 37-row call is the 16 + 16 + 5 row calls of its groups."""
    H, I, M = 512, 1536, 37
    gu, dn, q, _ = build_ffn(dev, H, I)
    x = synth.activations_bf16(M, H, seed=4, outlier_frac=0.01).to(dev)
    full = ffi.ffn_swiglu_nvfp4(x, gu, q[0][2], q[1][2], dn, q[2][2], I)
    parts = [ffi.ffn_swiglu_nvfp4(x[a:b].contiguous(), gu, q[0][2], q[1][2], dn, q[2][2], I)
             for a, b in ((0, 16), (16, 32), (32, 37))]
    assert torch.equal(full, torch.cat(parts))
    h = ffi.ffn_gate_up_nvfp4(x, gu, q[0][2], q[1][2], I)
    y = ffi.nvfp4_gemv(h, dn, q[2][2], H)
    assert torch.equal(y, full)
