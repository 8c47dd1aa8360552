"""Parity of the block-scaled FP8 (w8a16) path with the oracle, through the C ABI.

Bit-exact: the repack/unpack round trip of codes and grid.  Floating point:
every bf16 output inside its valid rounding interval (parity_checks: bit-exact
wherever the rounding is determined) and within 1e-2 * max(1, |oracle|).  The
weights are seeded stand-ins for an FP8 checkpoint (synth.fp8_weights); the
GPU and the oracle read the same bytes.
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_gb300 import ffi, synth

import parity_checks as pc

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ffi.load(build_if_missing=True)
    return torch.device("cuda:0")


def np_proj(codes, grid):
    return codes.cpu().numpy(), grid.cpu().numpy()


def count_beyond(got_bits, ref_bits):
    return pc.count_beyond_tolerance(got_bits, ref_bits, TOL)


@pytest.mark.parametrize("N,K", [(256, 512), (300, 272), (130, 80), (5120, 1024), (17, 4096)])
def test_repack_unpack_round_trip(dev, N, K):
    codes, grid = synth.fp8_weights(N, K, seed=N + K)
    p = ffi.w8a16_repack(codes.to(dev), grid.to(dev))
    assert p.numel() == ffi.load().w8a16_repacked_bytes(N, K)
    c2, g2 = ffi.w8a16_unpack(p, N, K)
    assert torch.equal(c2.cpu(), codes)
    assert torch.equal(g2.cpu(), grid)


def test_repack_is_a_permutation_plus_one_scale_per_tile_and_chunk(dev):
    N, K = 512, 1024
    codes, grid = synth.fp8_weights(N, K, seed=3)
    p = ffi.w8a16_repack(codes.to(dev), grid.to(dev)).cpu()
    group = 16 * 1024 + 16 * 4
    groups = p.view(-1, group)
    code_bytes = groups[:, :16 * 1024].reshape(-1)
    a = torch.bincount(codes.flatten().long(), minlength=256)
    b = torch.bincount(code_bytes.long(), minlength=256)
    assert torch.equal(a, b)
    scales = groups[:, 16 * 1024:].contiguous().view(torch.float32)  # [RB*C, 16 tiles]
    C = K // 64
    for rb in range(N // 256):
        for c in range(C):
            for t in range(16):
                assert scales[rb * C + c, t] == grid[(rb * 256 + 16 * t) // 128, (64 * c) // 128]


def run_gemv_case(dev, N, K, M, seed=0, outliers=0.0):
    codes, grid = synth.fp8_weights(N, K, seed=2000 + seed)
    x = synth.activations_bf16(M, K, seed=seed, outlier_frac=outliers)
    p = ffi.w8a16_repack(codes.to(dev), grid.to(dev))
    y = ffi.w8a16_gemv(x.to(dev), p, N)
    q = np_proj(codes, grid)
    xb, yb = synth.bf16_bits(x), synth.bf16_bits(y)
    ref = oracle.gemv_fp8(xb, *q)
    st = pc.check_gemv_fp8(yb, xb, q, f"w8a16 gemv N={N} K={K} M={M}")
    assert count_beyond(yb, ref) == 0
    return st, y, p, x


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_gemv_all_m(dev, M):
    run_gemv_case(dev, 384, 1024, M, seed=M, outliers=0.01 if M > 4 else 0.0)


@pytest.mark.parametrize("N,K,M", [(300, 272, 3), (130, 80, 1), (16, 16, 2), (1, 2048, 9),
                                   (1000, 4096, 16), (4096, 1024, 5)])
def test_gemv_shapes(dev, N, K, M):
    run_gemv_case(dev, N, K, M, seed=N % 97)


@pytest.mark.parametrize("N,K,M", [(384, 1024, 17), (1000, 2000, 40), (256, 4096, 64)])
def test_gemv_large_batches(dev, N, K, M):
    run_gemv_case(dev, N, K, M, seed=M, outliers=0.01)


def test_gemv_deterministic_and_reusable_workspace(dev):
    N, K, M = 2048, 4096, 4
    codes, grid = synth.fp8_weights(N, K, seed=11)
    p = ffi.w8a16_repack(codes.to(dev), grid.to(dev))
    x = synth.activations_bf16(M, K, seed=5).to(dev)
    ws = ffi.workspace(ffi.load().w8a16_gemv_workspace_bytes(M, N, K), dev)
    y0 = ffi.w8a16_gemv(x, p, N, ws=ws)
    for _ in range(3):
        assert torch.equal(ffi.w8a16_gemv(x, p, N, ws=ws), y0)
    assert ffi.nvfp4_workspace_status(ws) == 0


@pytest.mark.slow
@pytest.mark.parametrize("N,K,M", [(17408, 5120, 1), (5120, 17408, 8), (17408, 5120, 16)])
def test_gemv_full_size(dev, N, K, M):
    st, *_ = run_gemv_case(dev, N, K, M, seed=7)
    print(f"PARITY w8a16 gemv N={N} K={K} M={M}: {st}")


def build_ffn(dev, H, I, layer=0):
    proj = [synth.fp8_weights(I, H, seed=synth.layer_seed(layer, synth.GATE) + 77),
            synth.fp8_weights(I, H, seed=synth.layer_seed(layer, synth.UP) + 77),
            synth.fp8_weights(H, I, seed=synth.layer_seed(layer, synth.DOWN) + 77)]
    gu = ffi.w8a16_repack_gate_up(proj[0][0].to(dev), proj[0][1].to(dev),
                                  proj[1][0].to(dev), proj[1][1].to(dev))
    dn = ffi.w8a16_repack(proj[2][0].to(dev), proj[2][1].to(dev))
    return gu, dn, [np_proj(*t) for t in proj]


def run_ffn_case(dev, H, I, M, act, outliers=0.0, seed=0):
    """h inside its interval (bit-exact where determined), out likewise against
    the oracle's down projection of the GPU's own h, and end to end against the
    oracle's FFN (misses only through a legitimately different h; printed)."""
    gu, dn, q = build_ffn(dev, H, I)
    x = synth.activations_bf16(M, H, seed=seed, outlier_frac=outliers)
    xb = synth.bf16_bits(x)
    ws = ffi.workspace(ffi.load().ffn_swiglu_w8a16_workspace_bytes(M, H, I), dev)
    out = ffi.ffn_swiglu_w8a16(x.to(dev), gu, dn, I, act, ws=ws)
    torch.cuda.synchronize()
    h_bits = synth.bf16_bits(ffi.ffn_hidden_view(ws, M, I))
    sh = pc.check_hidden_fp8(h_bits, xb, q[0], q[1], act, f"w8a16 h H={H} I={I} M={M} act={act}")
    ob = synth.bf16_bits(out)
    so = pc.check_gemv_fp8(ob, h_bits, q[2], f"w8a16 out H={H} I={I} M={M} act={act}")
    ref = oracle.ffn_fp8(xb, q[0], q[1], q[2], act)
    n_out = count_beyond(ob, ref)
    print(f"PARITY w8a16 ffn H={H} I={I} M={M} act={act} outliers={outliers}: h {sh}, out {so}, "
          f"end to end {n_out} beyond 1e-2")
    assert n_out <= 0.005 * ref.size
    assert ffi.nvfp4_workspace_status(ws) == 0
    return out


@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16])
@pytest.mark.parametrize("act", [ffi.NVFP4_ACT_SILU, ffi.NVFP4_ACT_GELU_TANH])
def test_ffn_batch_m(dev, M, act):
    run_ffn_case(dev, 512, 1536, M, act, outliers=0.01 if M >= 8 else 0.0, seed=M)


@pytest.mark.parametrize("H,I,M", [(192, 400, 3), (320, 272, 1), (4096, 12288, 2), (512, 1536, 33)])
def test_ffn_shapes(dev, H, I, M):
    run_ffn_case(dev, H, I, M, ffi.NVFP4_ACT_SILU, seed=H % 13)


@pytest.mark.slow
@pytest.mark.parametrize("M,act,outliers", [(1, ffi.NVFP4_ACT_SILU, 0.0),
                                            (8, ffi.NVFP4_ACT_GELU_TANH, 0.01)])
def test_ffn_full_size(dev, M, act, outliers):
    run_ffn_case(dev, 5120, 17408, M, act, outliers, seed=M)


def test_ffn_matches_its_two_gemvs_bit_for_bit(dev):
    """The FFN's down step is the standalone GEMV on the FFN's own h."""
    H, I, M = 512, 1536, 5
    gu, dn, q = build_ffn(dev, H, I, layer=3)
    x = synth.activations_bf16(M, H, seed=21).to(dev)
    ws = ffi.workspace(ffi.load().ffn_swiglu_w8a16_workspace_bytes(M, H, I), dev)
    out = ffi.ffn_swiglu_w8a16(x, gu, dn, I, ws=ws)
    h = ffi.ffn_hidden_view(ws, M, I).clone()
    assert torch.equal(ffi.w8a16_gemv(h, dn, H), out)


def test_error_codes(dev):
    L = ffi.load()
    x = torch.zeros(65, 64, dtype=torch.bfloat16, device=dev)
    p = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    with pytest.raises(ffi.Nvfp4Error) as e:
        ffi.w8a16_gemv(x, p, 64)
    assert e.value.code == 4
    with pytest.raises(ffi.Nvfp4Error) as e:
        ffi.w8a16_gemv(x[:2], p, 64, ws=torch.zeros(16, dtype=torch.uint8, device=dev))
    assert e.value.code == 5
    with pytest.raises(ValueError):
        ffi.w8a16_repack(torch.zeros(300, 256, dtype=torch.uint8, device=dev),
                         torch.zeros(2, 2, dtype=torch.float32, device=dev))
    assert L.w8a16_repacked_bytes(0, 256) == 0
