"""ffn_swiglu_nvfp4_noalloc: the FFN for callers that cannot allocate a device
workspace (a process whose device memory is all reserved up front, or code
that must avoid an allocation's implicit synchronisation).  It runs on the
library's fixed device array; its results must match ffn_swiglu_nvfp4 on a
caller workspace.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_weight_only_gb300 import ffi, synth

pytestmark = pytest.mark.gpu

TOL = 1e-2


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


def _close(a, b):
    a = a.float().cpu().double().numpy()
    b = b.float().cpu().double().numpy()
    assert np.all(np.abs(a - b) <= TOL * np.maximum(1.0, np.abs(b)))


@pytest.mark.parametrize("M,H,I,act", [(1, 5120, 17408, 0), (8, 1024, 2816, 1), (16, 512, 1536, 0)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(dev, M, H, I, act):
    gu, g2, u2, dn, d2 = _weights(dev, H, I, layer=M)
    L = ffi.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for call in range(2):
        x = synth.activations_bf16(M, H, seed=100 * M + call, outlier_frac=0.01, device=dev)
        ref = ffi.ffn_swiglu_nvfp4(x, gu, g2, u2, dn, d2, I, act)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        rc = L.ffn_swiglu_nvfp4_noalloc(ctypes.c_void_p(x.data_ptr()), M, H, I,
                                        ctypes.c_void_p(gu.data_ptr()), g2, u2,
                                        ctypes.c_void_p(dn.data_ptr()), d2, act,
                                        ctypes.c_void_p(out.data_ptr()), stream)
        assert rc == 0, ffi.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        _close(out, ref)


def test_noalloc_rejects_shapes_beyond_its_workspace(dev):
    L = ffi.load()
    assert L.ffn_swiglu_nvfp4_workspace_bytes(16, 8192, 32768) > (24 << 20)
    A = [ctypes.c_void_p(0x10000 * i) for i in range(1, 5)]
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.ffn_swiglu_nvfp4_noalloc(A[0], 16, 8192, 32768, A[1], 1.0, 1.0, A[2], 1.0, 0, A[3],
                                    stream)
    assert rc == 5  # NVFP4_ERR_WORKSPACE
