"""Thin ctypes binding over libnvfp4ffn.so (argument marshalling only).

Every function here takes torch tensors, checks dtypes/devices, allocates the
outputs with torch, and forwards raw pointers, sizes and the current CUDA
stream to the C entry point of the same name.  All arithmetic runs in the
library's kernels; there is no CPU or PyTorch fallback, and a missing library
raises.
"""
import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4ffn.so")

NVFP4_ACT_SILU = 0
NVFP4_ACT_GELU_TANH = 1
NVFP4_SRC_F32 = 0
NVFP4_SRC_BF16 = 1

STATUS_NAMES = {0: "NVFP4_OK", 1: "NVFP4_ERR_NULL", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
                4: "NVFP4_ERR_RANGE", 5: "NVFP4_ERR_WORKSPACE", 6: "NVFP4_ERR_CUDA",
                7: "NVFP4_ERR_TIMEOUT", 8: "NVFP4_ERR_ALIAS"}

# Every symbol declared in include/nvfp4ffn.h.
EXPORTS = [
    "nvfp4_quantize_scratch_bytes", "nvfp4_quantize", "nvfp4_repacked_bytes", "nvfp4_repack",
    "nvfp4_repacked_gate_up_bytes", "nvfp4_repack_gate_up", "nvfp4_unpack",
    "nvfp4_gemv_workspace_bytes", "nvfp4_gemv", "ffn_swiglu_nvfp4_workspace_bytes",
    "ffn_swiglu_nvfp4_hidden_offset",
    "ffn_swiglu_nvfp4", "ffn_gate_up_nvfp4_workspace_bytes", "ffn_gate_up_nvfp4",
    "ffn_swiglu_nvfp4_noalloc", "nvfp4_noalloc_status",
    "ffn_swiglu_nvfp4_lora_workspace_bytes", "ffn_swiglu_nvfp4_lora",
    "nvfp4_lora_apply_scratch_bytes", "nvfp4_lora_apply",
    "w8a16_repacked_bytes", "w8a16_repacked_gate_up_bytes", "w8a16_repack",
    "w8a16_repack_gate_up", "w8a16_unpack", "w8a16_gemv_workspace_bytes", "w8a16_gemv",
    "ffn_swiglu_w8a16_workspace_bytes", "ffn_swiglu_w8a16",
    "nvfp4_workspace_init", "nvfp4_workspace_status", "nvfp4_status_string",
]
# Every symbol declared in include/nvfp4ffn_testing.h (test hooks).
TESTING_EXPORTS = ["nvfp4_testing_inject_stall", "nvfp4_testing_plan_aligned",
                   "nvfp4_testing_plan_aligned_w8a16"]


class Nvfp4Error(RuntimeError):
    def __init__(self, fn, code, lib):
        name = STATUS_NAMES.get(code, str(code))
        msg = lib.nvfp4_status_string(code).decode()
        super().__init__(f"{fn} failed: {name} ({msg})")
        self.code = code


_lib = None


def load(build_if_missing: bool = False):
    """Load the library (optionally building it first).  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run nvfp4_weight_only_gb300.build.build() "
                           "(or __graft_entry__.build()) first")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    sig = {
        "nvfp4_quantize_scratch_bytes": (sz, [i32, i32]),
        "nvfp4_quantize": (i32, [vp, i32, i32, i32, vp, vp, ctypes.POINTER(f32), vp, sz, vp]),
        "nvfp4_repacked_bytes": (sz, [i32, i32]),
        "nvfp4_repack": (i32, [vp, vp, i32, i32, vp, vp]),
        "nvfp4_repacked_gate_up_bytes": (sz, [i32, i32]),
        "nvfp4_repack_gate_up": (i32, [vp, vp, vp, vp, i32, i32, vp, vp]),
        "nvfp4_unpack": (i32, [vp, i32, i32, vp, vp, vp]),
        "nvfp4_gemv_workspace_bytes": (sz, [i32, i32, i32]),
        "nvfp4_gemv": (i32, [vp, i32, i32, vp, f32, i32, vp, vp, sz, vp]),
        "ffn_swiglu_nvfp4_workspace_bytes": (sz, [i32, i32, i32]),
        "ffn_swiglu_nvfp4_hidden_offset": (sz, []),
        "ffn_swiglu_nvfp4": (i32, [vp, i32, i32, i32, vp, f32, f32, vp, f32, i32, vp, vp, sz, vp]),
        "ffn_gate_up_nvfp4_workspace_bytes": (sz, [i32, i32, i32]),
        "ffn_gate_up_nvfp4": (i32, [vp, i32, i32, i32, vp, f32, f32, i32, vp, vp, sz, vp]),
        "ffn_swiglu_nvfp4_noalloc": (i32, [vp, i32, i32, i32, vp, f32, f32, vp, f32, i32, vp, vp]),
        "nvfp4_noalloc_status": (i32, [vp]),
        "ffn_swiglu_nvfp4_lora_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "ffn_swiglu_nvfp4_lora": (i32, [vp, i32, i32, i32, vp, f32, f32, vp, f32, i32, i32,
                                        vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "nvfp4_lora_apply_scratch_bytes": (sz, [i32, i32]),
        "nvfp4_lora_apply": (i32, [vp, i32, i32, vp, vp, i32, i32, vp, vp, sz, vp]),
        "nvfp4_testing_inject_stall": (i32, [i32, ctypes.c_ulonglong]),
        "nvfp4_testing_plan_aligned": (i32, [i32, i32, i32, i32, i32]),
        "nvfp4_testing_plan_aligned_w8a16": (i32, [i32, i32, i32, i32, i32]),
        "w8a16_repacked_bytes": (sz, [i32, i32]),
        "w8a16_repacked_gate_up_bytes": (sz, [i32, i32]),
        "w8a16_repack": (i32, [vp, vp, i32, i32, vp, vp]),
        "w8a16_repack_gate_up": (i32, [vp, vp, vp, vp, i32, i32, vp, vp]),
        "w8a16_unpack": (i32, [vp, i32, i32, vp, vp, vp]),
        "w8a16_gemv_workspace_bytes": (sz, [i32, i32, i32]),
        "w8a16_gemv": (i32, [vp, i32, i32, vp, i32, vp, vp, sz, vp]),
        "ffn_swiglu_w8a16_workspace_bytes": (sz, [i32, i32, i32]),
        "ffn_swiglu_w8a16": (i32, [vp, i32, i32, i32, vp, vp, i32, vp, vp, sz, vp]),
        "nvfp4_workspace_init": (i32, [vp, sz, vp]),
        "nvfp4_workspace_status": (i32, [vp, vp]),
        "nvfp4_status_string": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(fn, code):
    if code != 0:
        raise Nvfp4Error(fn, code, load())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ quantise / repack

def nvfp4_quantize(w: torch.Tensor):
    """W fp32/bf16 [N, K] (CUDA) -> (codes u8 [N, K/2], scales u8 [N, K/16], scale2 float)."""
    _cuda(w, "w")
    if w.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("w must be float32 or bfloat16")
    N, K = w.shape
    L = load()
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    nscr = L.nvfp4_quantize_scratch_bytes(N, K)
    scratch = torch.empty(nscr, dtype=torch.uint8, device=w.device)
    s2 = ctypes.c_float(0.0)
    dt = NVFP4_SRC_BF16 if w.dtype == torch.bfloat16 else NVFP4_SRC_F32
    _check("nvfp4_quantize", L.nvfp4_quantize(_ptr(w), dt, N, K, _ptr(codes), _ptr(scales),
                                              ctypes.byref(s2), _ptr(scratch), nscr,
                                              _stream(w.device)))
    return codes, scales, s2.value


def nvfp4_repack(codes: torch.Tensor, scales: torch.Tensor, N: int, K: int) -> torch.Tensor:
    _cuda(codes, "codes", torch.uint8)
    _cuda(scales, "scales", torch.uint8)
    L = load()
    out = torch.empty(L.nvfp4_repacked_bytes(N, K), dtype=torch.uint8, device=codes.device)
    _check("nvfp4_repack", L.nvfp4_repack(_ptr(codes), _ptr(scales), N, K, _ptr(out),
                                          _stream(codes.device)))
    return out


def nvfp4_repack_gate_up(gate_codes, gate_scales, up_codes, up_scales, I: int, H: int):
    for n, t in (("gate_codes", gate_codes), ("gate_scales", gate_scales),
                 ("up_codes", up_codes), ("up_scales", up_scales)):
        _cuda(t, n, torch.uint8)
    L = load()
    out = torch.empty(L.nvfp4_repacked_gate_up_bytes(I, H), dtype=torch.uint8,
                      device=gate_codes.device)
    _check("nvfp4_repack_gate_up",
           L.nvfp4_repack_gate_up(_ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes),
                                  _ptr(up_scales), I, H, _ptr(out), _stream(gate_codes.device)))
    return out


def nvfp4_unpack(packed: torch.Tensor, N: int, K: int):
    _cuda(packed, "packed", torch.uint8)
    L = load()
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=packed.device)
    scales = torch.empty((N, K // 16), dtype=torch.uint8, device=packed.device)
    _check("nvfp4_unpack", L.nvfp4_unpack(_ptr(packed), N, K, _ptr(codes), _ptr(scales),
                                          _stream(packed.device)))
    return codes, scales


# ------------------------------------------------------------------ GEMV / FFN

def nvfp4_gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    return load().nvfp4_gemv_workspace_bytes(M, N, K)


def ffn_swiglu_nvfp4_workspace_bytes(M: int, H: int, I: int) -> int:
    return load().ffn_swiglu_nvfp4_workspace_bytes(M, H, I)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled workspace buffer of at least `nbytes` (torch allocation)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def nvfp4_gemv(x: torch.Tensor, packed_w: torch.Tensor, scale2: float, N: int,
               ws: torch.Tensor = None, out: torch.Tensor = None) -> torch.Tensor:
    """y bf16 [M, N] = one NVFP4 projection of x bf16 [M, K]."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(packed_w, "packed_w", torch.uint8)
    M, K = x.shape
    L = load()
    if ws is None:
        ws = workspace(L.nvfp4_gemv_workspace_bytes(M, N, K), x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _check("nvfp4_gemv", L.nvfp4_gemv(_ptr(x), M, K, _ptr(packed_w), float(scale2), N, _ptr(out),
                                      _ptr(ws), ws.numel(), _stream(x.device)))
    return out


def ffn_swiglu_nvfp4(x: torch.Tensor, gate_up_packed: torch.Tensor, gate_scale2: float,
                     up_scale2: float, down_packed: torch.Tensor, down_scale2: float, I: int,
                     act: int = NVFP4_ACT_SILU, ws: torch.Tensor = None,
                     out: torch.Tensor = None) -> torch.Tensor:
    """out bf16 [M, H] = down(act(gate(x)) * up(x)) for x bf16 [M, H]."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(gate_up_packed, "gate_up_packed", torch.uint8)
    _cuda(down_packed, "down_packed", torch.uint8)
    M, H = x.shape
    L = load()
    if ws is None:
        ws = workspace(L.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), x.device)
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _check("ffn_swiglu_nvfp4",
           L.ffn_swiglu_nvfp4(_ptr(x), M, H, I, _ptr(gate_up_packed), float(gate_scale2),
                              float(up_scale2), _ptr(down_packed), float(down_scale2), int(act),
                              _ptr(out), _ptr(ws), ws.numel(), _stream(x.device)))
    return out


def ffn_swiglu_nvfp4_noalloc(x: torch.Tensor, gate_up_packed: torch.Tensor, gate_scale2: float,
                             up_scale2: float, down_packed: torch.Tensor, down_scale2: float,
                             I: int, act: int = NVFP4_ACT_SILU,
                             out: torch.Tensor = None) -> torch.Tensor:
    """ffn_swiglu_nvfp4 on the library's fixed device workspace (for callers that
    cannot allocate one); only the output is allocated here, and only when `out`
    is not given."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(gate_up_packed, "gate_up_packed", torch.uint8)
    _cuda(down_packed, "down_packed", torch.uint8)
    M, H = x.shape
    L = load()
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _check("ffn_swiglu_nvfp4_noalloc",
           L.ffn_swiglu_nvfp4_noalloc(_ptr(x), M, H, I, _ptr(gate_up_packed), float(gate_scale2),
                                      float(up_scale2), _ptr(down_packed), float(down_scale2),
                                      int(act), _ptr(out), _stream(x.device)))
    return out


def ffn_swiglu_nvfp4_lora(x: torch.Tensor, gate_up_packed: torch.Tensor, gate_scale2: float,
                          up_scale2: float, down_packed: torch.Tensor, down_scale2: float, I: int,
                          act: int = NVFP4_ACT_SILU, gate=None, up=None, down=None,
                          ws: torch.Tensor = None, out: torch.Tensor = None) -> torch.Tensor:
    """The FFN with the LoRA overlay; gate/up/down = (A, B) bf16 pairs or None."""
    _cuda(x, "x", torch.bfloat16)
    M, H = x.shape
    pairs = [gate, up, down]
    rank = next((p[0].shape[0] for p in pairs if p is not None), 1)
    for p in pairs:
        if p is not None:
            _cuda(p[0], "lora A", torch.bfloat16)
            _cuda(p[1], "lora B", torch.bfloat16)
    L = load()
    if ws is None:
        ws = workspace(L.ffn_swiglu_nvfp4_lora_workspace_bytes(M, H, I, rank), x.device)
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    ptrs = []
    for p in pairs:
        ptrs += [_ptr(p[0]), _ptr(p[1])] if p is not None else [_ptr(None), _ptr(None)]
    _check("ffn_swiglu_nvfp4_lora",
           L.ffn_swiglu_nvfp4_lora(_ptr(x), M, H, I, _ptr(gate_up_packed), float(gate_scale2),
                                   float(up_scale2), _ptr(down_packed), float(down_scale2),
                                   int(act), rank, *ptrs, _ptr(out), _ptr(ws), ws.numel(),
                                   _stream(x.device)))
    return out


def nvfp4_lora_apply(v: torch.Tensor, a: torch.Tensor, b: torch.Tensor,
                     base: torch.Tensor) -> torch.Tensor:
    """base [M, N] = bf16(base + bf16(b bf16(a v))) in place (returns base)."""
    for n, t in (("v", v), ("a", a), ("b", b), ("base", base)):
        _cuda(t, n, torch.bfloat16)
    M, K = v.shape
    rank = a.shape[0]
    N = b.shape[0]
    L = load()
    scratch = workspace(L.nvfp4_lora_apply_scratch_bytes(M, rank), v.device)
    _check("nvfp4_lora_apply",
           L.nvfp4_lora_apply(_ptr(v), M, K, _ptr(a), _ptr(b), rank, N, _ptr(base),
                              _ptr(scratch), scratch.numel(), _stream(v.device)))
    return base


def ffn_gate_up_nvfp4_workspace_bytes(M: int, H: int, I: int) -> int:
    return load().ffn_gate_up_nvfp4_workspace_bytes(M, H, I)


def ffn_gate_up_nvfp4(x: torch.Tensor, gate_up_packed: torch.Tensor, gate_scale2: float,
                      up_scale2: float, I: int, act: int = NVFP4_ACT_SILU,
                      ws: torch.Tensor = None, h: torch.Tensor = None) -> torch.Tensor:
    """h bf16 [M, I] = act(gate(x)) * up(x) for x bf16 [M, H]."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(gate_up_packed, "gate_up_packed", torch.uint8)
    M, H = x.shape
    L = load()
    if ws is None:
        ws = workspace(L.ffn_gate_up_nvfp4_workspace_bytes(M, H, I), x.device)
    if h is None:
        h = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
    _cuda(h, "h", torch.bfloat16)
    _check("ffn_gate_up_nvfp4",
           L.ffn_gate_up_nvfp4(_ptr(x), M, H, I, _ptr(gate_up_packed), float(gate_scale2),
                               float(up_scale2), int(act), _ptr(h), _ptr(ws), ws.numel(),
                               _stream(x.device)))
    return h


def ffn_hidden_view(ws: torch.Tensor, M: int, I: int) -> torch.Tensor:
    """The bf16 activation h [M, I] that ffn_swiglu_nvfp4 leaves in its workspace."""
    off = load().ffn_swiglu_nvfp4_hidden_offset()
    return ws[off:off + M * I * 2].view(torch.bfloat16).view(M, I)


def nvfp4_workspace_init(ws: torch.Tensor) -> None:
    _check("nvfp4_workspace_init",
           load().nvfp4_workspace_init(_ptr(ws), ws.numel(), _stream(ws.device)))


def nvfp4_workspace_status(ws: torch.Tensor) -> int:
    """Synchronise, read and clear the device status word (0 = OK, 7 = timeout)."""
    return load().nvfp4_workspace_status(_ptr(ws), _stream(ws.device))


def nvfp4_noalloc_status(device=None) -> int:
    """Status of the fixed-workspace FFN calls (0 = OK, 7 = timeout, after which
    the library has zero-filled its array again)."""
    return load().nvfp4_noalloc_status(_stream(device))


# ------------------------------------------------------------------ block-scaled FP8 (w8a16)

def _fp8_projection(codes, grid, name):
    _cuda(codes, f"{name} codes", torch.uint8)
    _cuda(grid, f"{name} grid", torch.float32)
    N, K = codes.shape
    if tuple(grid.shape) != ((N + 127) // 128, (K + 127) // 128):
        raise ValueError(f"{name} grid must be [ceil(N/128), ceil(K/128)], got {tuple(grid.shape)}")
    return N, K


def w8a16_repack(codes: torch.Tensor, grid: torch.Tensor) -> torch.Tensor:
    """E4M3 bytes [N, K] + fp32 block grid -> the kernel layout (uint8 blob)."""
    N, K = _fp8_projection(codes, grid, "w8a16_repack")
    L = load()
    out = torch.empty(L.w8a16_repacked_bytes(N, K), dtype=torch.uint8, device=codes.device)
    _check("w8a16_repack", L.w8a16_repack(_ptr(codes), _ptr(grid), N, K, _ptr(out),
                                          _stream(codes.device)))
    return out


def w8a16_repack_gate_up(gate_codes, gate_grid, up_codes, up_grid) -> torch.Tensor:
    I, H = _fp8_projection(gate_codes, gate_grid, "gate")
    if _fp8_projection(up_codes, up_grid, "up") != (I, H):
        raise ValueError("gate and up must have the same shape")
    L = load()
    out = torch.empty(L.w8a16_repacked_gate_up_bytes(I, H), dtype=torch.uint8,
                      device=gate_codes.device)
    _check("w8a16_repack_gate_up",
           L.w8a16_repack_gate_up(_ptr(gate_codes), _ptr(gate_grid), _ptr(up_codes),
                                  _ptr(up_grid), I, H, _ptr(out), _stream(gate_codes.device)))
    return out


def w8a16_unpack(packed: torch.Tensor, N: int, K: int):
    _cuda(packed, "packed", torch.uint8)
    L = load()
    codes = torch.empty((N, K), dtype=torch.uint8, device=packed.device)
    grid = torch.empty(((N + 127) // 128, (K + 127) // 128), dtype=torch.float32,
                       device=packed.device)
    _check("w8a16_unpack", L.w8a16_unpack(_ptr(packed), N, K, _ptr(codes), _ptr(grid),
                                          _stream(packed.device)))
    return codes, grid


def w8a16_gemv(x: torch.Tensor, packed_w: torch.Tensor, N: int, ws: torch.Tensor = None,
               out: torch.Tensor = None) -> torch.Tensor:
    """y bf16 [M, N] = one block-scaled FP8 projection of x bf16 [M, K]."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(packed_w, "packed_w", torch.uint8)
    M, K = x.shape
    L = load()
    if ws is None:
        ws = workspace(L.w8a16_gemv_workspace_bytes(M, N, K), x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _check("w8a16_gemv", L.w8a16_gemv(_ptr(x), M, K, _ptr(packed_w), N, _ptr(out), _ptr(ws),
                                      ws.numel(), _stream(x.device)))
    return out


def ffn_swiglu_w8a16(x: torch.Tensor, gate_up_packed: torch.Tensor, down_packed: torch.Tensor,
                     I: int, act: int = NVFP4_ACT_SILU, ws: torch.Tensor = None,
                     out: torch.Tensor = None) -> torch.Tensor:
    """out bf16 [M, H] = down(act(gate(x)) * up(x)) on block-scaled FP8 weights."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(gate_up_packed, "gate_up_packed", torch.uint8)
    _cuda(down_packed, "down_packed", torch.uint8)
    M, H = x.shape
    L = load()
    if ws is None:
        ws = workspace(L.ffn_swiglu_w8a16_workspace_bytes(M, H, I), x.device)
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _check("ffn_swiglu_w8a16",
           L.ffn_swiglu_w8a16(_ptr(x), M, H, I, _ptr(gate_up_packed), _ptr(down_packed), int(act),
                              _ptr(out), _ptr(ws), ws.numel(), _stream(x.device)))
    return out
