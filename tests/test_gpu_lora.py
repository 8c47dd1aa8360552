"""GPU parity of the LoRA overlay (the dense-FFN page's apply_lora_gate_up /
apply_lora_down) through the C ABI: ffn_swiglu_nvfp4_lora and
nvfp4_lora_apply against the oracle.  Every rounded quantity (xa, the delta,
g and u after their deltas, h, out) must lie in its valid rounding interval,
bit-exact wherever the interval is a single value."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_gb300 import ffi, synth

import parity_checks as pc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ffi.load(build_if_missing=True)
    return torch.device("cuda:0")


def _bf16(shape, seed, std):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _pairs(H, I, r, seed, which=("gate", "up", "down")):
    shapes = {"gate": ((r, H), (I, r)), "up": ((r, H), (I, r)), "down": ((r, I), (H, r))}
    return {k: (_bf16(shapes[k][0], seed + 10 * i, 0.05), _bf16(shapes[k][1], seed + 10 * i + 1,
                                                                  0.05))
            if k in which else None for i, k in enumerate(("gate", "up", "down"))}


def _build(dev, H, I):
    w = [synth.weights_f32(I, H, seed=synth.layer_seed(3, synth.GATE)),
         synth.weights_f32(I, H, seed=synth.layer_seed(3, synth.UP)),
         synth.weights_f32(H, I, seed=synth.layer_seed(3, synth.DOWN))]
    q = [ffi.nvfp4_quantize(t.to(dev)) for t in w]
    rq = [oracle.quantize(t.numpy()) for t in w]
    for a, b in zip(q, rq):
        assert np.array_equal(a[0].cpu().numpy(), b[0]) and np.array_equal(a[1].cpu().numpy(), b[1])
    gu = ffi.nvfp4_repack_gate_up(q[0][0], q[0][1], q[1][0], q[1][1], I, H)
    dn = ffi.nvfp4_repack(q[2][0], q[2][1], H, I)
    return gu, dn, q, rq


def _check_lora_ffn(dev, H, I, M, r, act, which, outliers=0.0):
    gu, dn, q, rq = _build(dev, H, I)
    pairs = _pairs(H, I, r, seed=M * 100 + r, which=which)
    x = synth.activations_bf16(M, H, seed=M + r, outlier_frac=outliers)
    xb = synth.bf16_bits(x)
    ws = ffi.workspace(ffi.load().ffn_swiglu_nvfp4_lora_workspace_bytes(M, H, I, r), dev)
    dpairs = {k: (v[0].to(dev), v[1].to(dev)) if v is not None else None for k, v in pairs.items()}
    out = ffi.ffn_swiglu_nvfp4_lora(x.to(dev), gu, q[0][2], q[1][2], dn, q[2][2], I, act,
                                    ws=ws, **dpairs)
    torch.cuda.synchronize()
    h_bits = synth.bf16_bits(ffi.ffn_hidden_view(ws, M, I))
    obits = {k: (synth.bf16_bits(v[0]), synth.bf16_bits(v[1])) if v is not None else None
             for k, v in pairs.items()}
    ref_out, ref_h = oracle.ffn_lora(xb, I, rq[0], rq[1], rq[2], act,
                                     dict(rank=r, **obits))
    xf = pc.bf16_f64(xb)

    def with_delta(lo, hi, name, v_lo, v_hi):
        if obits[name] is None:
            return lo, hi
        d_lo, d_hi = pc.lora_delta_interval(v_lo, v_hi, *obits[name])
        return pc.bf16_round(lo + d_lo), pc.bf16_round(hi + d_hi)

    g_lo, g_hi = with_delta(*pc.gemv_interval(xb, rq[0], I), "gate", xf, xf)
    u_lo, u_hi = with_delta(*pc.gemv_interval(xb, rq[1], I), "up", xf, xf)
    h_lo, h_hi = pc.hidden_interval_from(g_lo, g_hi, u_lo, u_hi, act)
    sh = pc.check_interval(h_bits, h_lo, h_hi, ref_h, f"lora h M={M} r={r}")
    # out against the oracle's down projection (and down delta) of the GPU's h
    hf = pc.bf16_f64(h_bits)
    o_lo, o_hi = with_delta(*pc.gemv_interval(h_bits, rq[2], H), "down", hf, hf)
    ref_o = oracle.lora_apply(h_bits, *obits["down"], oracle.gemv(h_bits, *rq[2], H)) \
        if obits["down"] is not None else oracle.gemv(h_bits, *rq[2], H)
    so = pc.check_interval(synth.bf16_bits(out), o_lo, o_hi, ref_o, f"lora out M={M} r={r}")
    n_out = pc.count_beyond_tolerance(synth.bf16_bits(out), ref_out)
    print(f"PARITY lora H={H} I={I} M={M} r={r} act={act} pairs={which}: h {sh}, out {so}, "
          f"end to end {n_out} beyond 1e-2")
    assert n_out <= 0.005 * ref_out.size
    assert ffi.nvfp4_workspace_status(ws) == 0
    return out, x, gu, dn, q, pairs, ws


@pytest.mark.parametrize("M,r,act", [(1, 8, 0), (3, 16, 1), (16, 64, 0), (8, 1, 1)])
def test_lora_ffn_all_pairs(dev, M, r, act):
    _check_lora_ffn(dev, 512, 1536, M, r, act, ("gate", "up", "down"), outliers=0.01)


@pytest.mark.parametrize("which", [("gate",), ("up",), ("down",), ("gate", "down")])
def test_lora_ffn_single_pairs(dev, which):
    _check_lora_ffn(dev, 256, 768, 2, 16, 0, which)


def test_lora_ffn_full_size(dev):
    _check_lora_ffn(dev, 5120, 17408, 1, 16, 0, ("gate", "up", "down"))


def test_lora_zero_b_is_the_plain_ffn_bit_for_bit(dev):
    H, I, M, r = 512, 1536, 4, 16
    gu, dn, q, _ = _build(dev, H, I)
    x = synth.activations_bf16(M, H, seed=9).to(dev)
    z = lambda n, k: torch.zeros((n, k), dtype=torch.bfloat16, device=dev)  # noqa: E731
    a = _bf16((r, H), 1, 0.05).to(dev)
    out = ffi.ffn_swiglu_nvfp4_lora(x, gu, q[0][2], q[1][2], dn, q[2][2], I,
                                    gate=(a, z(I, r)), up=(a, z(I, r)),
                                    down=(_bf16((r, I), 2, 0.05).to(dev), z(H, r)))
    plain = ffi.ffn_swiglu_nvfp4(x, gu, q[0][2], q[1][2], dn, q[2][2], I)
    assert torch.equal(out, plain)
    again = ffi.ffn_swiglu_nvfp4_lora(x, gu, q[0][2], q[1][2], dn, q[2][2], I)  # no pairs
    assert torch.equal(again, plain)


@pytest.mark.parametrize("M,K,N,r", [(1, 5120, 17408, 16), (5, 4096, 300, 64), (16, 512, 64, 3),
                                     (2, 1030, 100, 8),      # K % 8 != 0: 4-byte vectors
                                     (3, 70000, 64, 24)])    # more K slices than the cap
def test_lora_apply_standalone(dev, M, K, N, r):
    v = _bf16((M, K), 3, 1.0)
    a = _bf16((r, K), 4, 0.05)
    b = _bf16((N, r), 5, 0.05)
    base = _bf16((M, N), 6, 1.0)
    got = ffi.nvfp4_lora_apply(v.to(dev), a.to(dev), b.to(dev), base.to(dev).clone())
    vb, ab, bb, baseb = (synth.bf16_bits(t) for t in (v, a, b, base))
    ref = oracle.lora_apply(vb, ab, bb, baseb)
    vf = pc.bf16_f64(vb)
    d_lo, d_hi = pc.lora_delta_interval(vf, vf, ab, bb)
    bf = pc.bf16_f64(baseb)
    st = pc.check_interval(synth.bf16_bits(got), pc.bf16_round(bf + d_lo),
                           pc.bf16_round(bf + d_hi), ref, f"lora_apply M={M} K={K} N={N} r={r}")
    print(f"PARITY lora_apply M={M} K={K} N={N} r={r}: {st}")


def test_lora_rejects_half_pairs_and_bad_rank(dev):
    H, I, M = 256, 512, 1
    gu, dn, q, _ = _build(dev, H, I)
    x = synth.activations_bf16(M, H, seed=1).to(dev)
    a = _bf16((4, H), 1, 0.05).to(dev)
    with pytest.raises(ffi.Nvfp4Error) as e:
        ffi.ffn_swiglu_nvfp4_lora(x, gu, q[0][2], q[1][2], dn, q[2][2], I,
                                  gate=(a, torch.empty(0, dtype=torch.bfloat16, device=dev)))
    assert e.value.code in (1, 2, 5)
    big = _bf16((65, H), 1, 0.05).to(dev)
    with pytest.raises(ffi.Nvfp4Error) as e:
        ffi.ffn_swiglu_nvfp4_lora(x, gu, q[0][2], q[1][2], dn, q[2][2], I,
                                  gate=(big, _bf16((I, 65), 2, 0.05).to(dev)))
    assert e.value.code == 4
