"""ffn_swiglu_nvfp4_noalloc: the FFN for callers that cannot allocate a device
workspace (a process whose device memory is all reserved up front, or code
that must avoid an allocation's implicit synchronisation).  It runs on the
library's fixed device array and the same two kernels as ffn_swiglu_nvfp4, so
its results must equal those of ffn_swiglu_nvfp4 on a caller workspace bit
for bit.  This file is collected last on purpose: if it fails, a run that
stops at the first failure has already run every other test."""
import ctypes

import pytest
import torch

from nvfp4_weight_only_gb300 import ffi, synth

pytestmark = pytest.mark.gpu

OK, RANGE, ALIGN, WORKSPACE, TIMEOUT = 0, 4, 3, 5, 7


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ffi.load(build_if_missing=True)
    return torch.device("cuda:0")


def _weights(dev, H, I, layer):
    q = [ffi.nvfp4_quantize(synth.weights_f32(n, k, seed=synth.layer_seed(layer, p), device=dev))
         for p, (n, k) in ((synth.GATE, (I, H)), (synth.UP, (I, H)), (synth.DOWN, (H, I)))]
    gu = ffi.nvfp4_repack_gate_up(q[0][0], q[0][1], q[1][0], q[1][1], I, H)
    dn = ffi.nvfp4_repack(q[2][0], q[2][1], H, I)
    return gu, q[0][2], q[1][2], dn, q[2][2]


def _call(L, dev, x, M, H, I, w, act, out):
    """The entry point through the C ABI, on torch's current stream."""
    gu, g2, u2, dn, d2 = w
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    return L.ffn_swiglu_nvfp4_noalloc(ctypes.c_void_p(x.data_ptr()), M, H, I,
                                      ctypes.c_void_p(gu.data_ptr()), g2, u2,
                                      ctypes.c_void_p(dn.data_ptr()), d2, act,
                                      ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("M,H,I,act", [(1, 5120, 17408, 0), (8, 1024, 2816, 1), (16, 512, 1536, 0)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(dev, M, H, I, act):
    w = _weights(dev, H, I, layer=M)
    L = ffi.load()
    for call in range(2):
        x = synth.activations_bf16(M, H, seed=100 * M + call, outlier_frac=0.01, device=dev)
        ref = ffi.ffn_swiglu_nvfp4(x, w[0], w[1], w[2], w[3], w[4], I, act)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        rc = _call(L, dev, x, M, H, I, w, act, out)
        assert rc == OK, ffi.STATUS_NAMES.get(rc, rc)
        assert L.nvfp4_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)) == OK
        assert torch.equal(out, ref)


def test_noalloc_rejected_calls_change_nothing_and_nothing_is_allocated(dev):
    M, H, I = 4, 1024, 2816
    w = _weights(dev, H, I, layer=3)
    L = ffi.load()
    x = synth.activations_bf16(M, H, seed=7, device=dev)
    ref = ffi.ffn_swiglu_nvfp4(x, w[0], w[1], w[2], w[3], w[4], I, 0)
    outs = [torch.empty((M, H), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    assert _call(L, dev, x, M, H, I, w, 0, outs[0]) == OK  # first call: set-up done
    bad = outs[0].view(-1)[1:].view(torch.uint8)  # 2 bytes past a 16-byte boundary
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(dev)[0]
    for out in outs[1:]:
        # rejected calls (an unknown activation, a misaligned output) first
        assert _call(L, dev, x, M, H, I, w, 7, out) == RANGE
        assert L.ffn_swiglu_nvfp4_noalloc(ctypes.c_void_p(x.data_ptr()), M, H, I,
                                          ctypes.c_void_p(w[0].data_ptr()), w[1], w[2],
                                          ctypes.c_void_p(w[3].data_ptr()), w[4], 0,
                                          ctypes.c_void_p(bad.data_ptr()), stream) == ALIGN
        assert _call(L, dev, x, M, H, I, w, 0, out) == OK
        torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info(dev)[0]
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    for out in outs:
        assert torch.equal(out, ref)
    assert L.nvfp4_noalloc_status(stream) == OK


def test_noalloc_timeout_is_reported_and_repaired(dev):
    M, H, I = 2, 512, 1536
    w = _weights(dev, H, I, layer=5)
    L = ffi.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    x = synth.activations_bf16(M, H, seed=9, device=dev)
    ref = ffi.ffn_swiglu_nvfp4(x, w[0], w[1], w[2], w[3], w[4], I, 0)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    assert L.nvfp4_testing_inject_stall(1, 2_000_000) == OK
    try:
        assert _call(L, dev, x, M, H, I, w, 0, out) == OK  # launched; gives up on the GPU
        assert L.nvfp4_noalloc_status(stream) == TIMEOUT
    finally:
        assert L.nvfp4_testing_inject_stall(0, 0) == OK
    assert L.nvfp4_noalloc_status(stream) == OK
    for _ in range(2):
        assert _call(L, dev, x, M, H, I, w, 0, out) == OK
        assert L.nvfp4_noalloc_status(stream) == OK
        assert torch.equal(out, ref)


def test_noalloc_rejects_shapes_beyond_its_workspace(dev):
    L = ffi.load()
    assert L.ffn_swiglu_nvfp4_workspace_bytes(16, 8192, 32768) > (24 << 20)
    A = [ctypes.c_void_p(0x10000000 * i) for i in range(1, 5)]
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.ffn_swiglu_nvfp4_noalloc(A[0], 16, 8192, 32768, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3],
                                    stream)
    assert rc == WORKSPACE
