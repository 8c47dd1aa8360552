"""The kernels' bounded waits, driven to run out on purpose.

The testing switch nvfp4_testing_inject_stall makes every launch's producer
issue no weight copies, so the consumers' first wait on a stage can never
complete; with a short limit each kernel gives up after it, sets the device
status word and returns, with every wait ended and no copy in flight.  The
status word must then read NVFP4_ERR_TIMEOUT, and once the switch is off and
the workspace zero-filled again the very next call must be correct."""
import pytest
import torch

import oracle
from nvfp4_weight_only_gb300 import ffi, synth

import parity_checks as pc

pytestmark = pytest.mark.gpu

TIMEOUT = 7
WAIT_NS = 2_000_000  # 2 ms


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ffi.load(build_if_missing=True)
    return torch.device("cuda:0")


def _quant(w, dev):
    c, s, s2 = ffi.nvfp4_quantize(w.to(dev))
    return (c, s, s2), oracle.quantize(w.numpy())


@pytest.mark.parametrize("M", [1, 5, 12])
def test_abandoned_wait_reports_timeout_then_next_call_is_correct(dev, M):
    H, I = 512, 1536
    w = [synth.weights_f32(I, H, seed=synth.layer_seed(7, synth.GATE)),
         synth.weights_f32(I, H, seed=synth.layer_seed(7, synth.UP)),
         synth.weights_f32(H, I, seed=synth.layer_seed(7, synth.DOWN))]
    q, rq = zip(*[_quant(t, dev) for t in w])
    gu = ffi.nvfp4_repack_gate_up(q[0][0], q[0][1], q[1][0], q[1][1], I, H)
    dn = ffi.nvfp4_repack(q[2][0], q[2][1], H, I)
    x = synth.activations_bf16(M, H, seed=M, outlier_frac=0.01)
    xd = x.to(dev)
    ws = ffi.workspace(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), dev)
    ws_g = ffi.workspace(ffi.nvfp4_gemv_workspace_bytes(M, H, I), dev)
    h = torch.zeros((M, I), dtype=torch.bfloat16, device=dev)
    L = ffi.load()
    assert L.nvfp4_testing_inject_stall(1, WAIT_NS) == 0
    try:
        ffi.ffn_swiglu_nvfp4(xd, gu, q[0][2], q[1][2], dn, q[2][2], I, ws=ws)
        assert ffi.nvfp4_workspace_status(ws) == TIMEOUT
        ffi.nvfp4_gemv(h, dn, q[2][2], H, ws=ws_g)
        assert ffi.nvfp4_workspace_status(ws_g) == TIMEOUT
    finally:
        assert L.nvfp4_testing_inject_stall(0, 0) == 0
    assert ffi.nvfp4_workspace_status(ws) == 0  # read-and-clear: clear now
    # the counters of a call that gave up may be off zero: zero-fill, then reuse
    ffi.nvfp4_workspace_init(ws)
    ffi.nvfp4_workspace_init(ws_g)
    out = ffi.ffn_swiglu_nvfp4(xd, gu, q[0][2], q[1][2], dn, q[2][2], I, ws=ws)
    torch.cuda.synchronize()
    assert ffi.nvfp4_workspace_status(ws) == 0
    xb = synth.bf16_bits(x)
    h_bits = synth.bf16_bits(ffi.ffn_hidden_view(ws, M, I))
    pc.check_hidden(h_bits, xb, rq[0], rq[1], oracle.ACT_SILU, f"h after timeout M={M}")
    pc.check_gemv(synth.bf16_bits(out), h_bits, rq[2], H, f"out after timeout M={M}")
    y = ffi.nvfp4_gemv(ffi.ffn_hidden_view(ws, M, I).contiguous(), dn, q[2][2], H, ws=ws_g)
    assert torch.equal(y, out)
    assert ffi.nvfp4_workspace_status(ws_g) == 0


@pytest.mark.parametrize("M", [1, 8, 12])
def test_fp8_abandoned_wait_reports_timeout_then_next_call_is_correct(dev, M):
    """The block-scaled FP8 kernels share the bounded waits: the same switch
    makes their first wait run out, the status reports it, and after a
    zero-fill the next call on the workspace is correct."""
    H, I = 512, 1536
    proj = [synth.fp8_weights(I, H, seed=71), synth.fp8_weights(I, H, seed=72),
            synth.fp8_weights(H, I, seed=73)]
    gu = ffi.w8a16_repack_gate_up(*(t.to(dev) for t in (*proj[0], *proj[1])))
    dn = ffi.w8a16_repack(proj[2][0].to(dev), proj[2][1].to(dev))
    q = [(c.numpy(), g.numpy()) for c, g in proj]
    x = synth.activations_bf16(M, H, seed=M, outlier_frac=0.01)
    xd = x.to(dev)
    L = ffi.load()
    ws = ffi.workspace(L.ffn_swiglu_w8a16_workspace_bytes(M, H, I), dev)
    assert L.nvfp4_testing_inject_stall(1, WAIT_NS) == 0
    try:
        ffi.ffn_swiglu_w8a16(xd, gu, dn, I, ws=ws)
        assert ffi.nvfp4_workspace_status(ws) == TIMEOUT
    finally:
        assert L.nvfp4_testing_inject_stall(0, 0) == 0
    assert ffi.nvfp4_workspace_status(ws) == 0  # read-and-clear
    ffi.nvfp4_workspace_init(ws)
    out = ffi.ffn_swiglu_w8a16(xd, gu, dn, I, ws=ws)
    torch.cuda.synchronize()
    assert ffi.nvfp4_workspace_status(ws) == 0
    xb = synth.bf16_bits(x)
    h_bits = synth.bf16_bits(ffi.ffn_hidden_view(ws, M, I))
    pc.check_hidden_fp8(h_bits, xb, q[0], q[1], oracle.ACT_SILU, f"fp8 h after timeout M={M}")
    pc.check_gemv_fp8(synth.bf16_bits(out), h_bits, q[2], f"fp8 out after timeout M={M}")
