"""CPU oracle for the NVFP4 weight-only SwiGLU FFN decode -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  It wraps nvfp4_oracle.c (plain C, fp64 accumulation) through
ctypes and converts numpy arrays in and out; all arithmetic lives in the C
file.  bf16 tensors cross this boundary as uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        i64 = ctypes.c_int64
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_bf16_decode.argtypes = [ctypes.c_uint16]
        L.orc_bf16_decode.restype = ctypes.c_double
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_quantize_f32.argtypes = [f32p, i64, i64, u8p, u8p, ctypes.POINTER(ctypes.c_float)]
        L.orc_quantize_f32.restype = ctypes.c_int
        L.orc_quantize_bf16.argtypes = [u16p, i64, i64, u8p, u8p, ctypes.POINTER(ctypes.c_float)]
        L.orc_quantize_bf16.restype = ctypes.c_int
        L.orc_dequantize.argtypes = [u8p, u8p, ctypes.c_float, i64, i64, f64p]
        L.orc_dequantize.restype = None
        L.orc_gemv_f64.argtypes = [u16p, i64, i64, u8p, u8p, ctypes.c_float, i64, f64p]
        L.orc_gemv_f64.restype = None
        L.orc_gemv.argtypes = [u16p, i64, i64, u8p, u8p, ctypes.c_float, i64, u16p]
        L.orc_gemv.restype = None
        L.orc_silu.argtypes = [ctypes.c_double]
        L.orc_silu.restype = ctypes.c_double
        L.orc_gelu_tanh.argtypes = [ctypes.c_double]
        L.orc_gelu_tanh.restype = ctypes.c_double
        L.orc_ffn_hidden.argtypes = [u16p, i64, i64, i64, u8p, u8p, ctypes.c_float,
                                     u8p, u8p, ctypes.c_float, ctypes.c_int, u16p]
        L.orc_ffn_hidden.restype = None
        L.orc_ffn.argtypes = [u16p, i64, i64, i64, u8p, u8p, ctypes.c_float,
                              u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float,
                              ctypes.c_int, u16p]
        L.orc_ffn.restype = None
        L.orc_bf16_from_double_array.argtypes = [f64p, i64, u16p]
        L.orc_bf16_from_double_array.restype = None
        L.orc_act_array.argtypes = [f64p, i64, ctypes.c_int, f64p]
        L.orc_act_array.restype = None
        L.orc_lora_xa.argtypes = [u16p, i64, i64, u16p, i64, u16p]
        L.orc_lora_xa.restype = None
        L.orc_lora_delta.argtypes = [u16p, i64, i64, u16p, i64, u16p]
        L.orc_lora_delta.restype = None
        L.orc_lora_add.argtypes = [u16p, u16p, i64]
        L.orc_lora_add.restype = None
        L.orc_lora_apply.argtypes = [u16p, i64, i64, u16p, u16p, i64, i64, u16p]
        L.orc_lora_apply.restype = None
        vp = ctypes.c_void_p
        L.orc_ffn_lora.argtypes = [u16p, i64, i64, i64, u8p, u8p, ctypes.c_float,
                                   u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float,
                                   ctypes.c_int, i64, vp, vp, vp, vp, vp, vp, u16p, u16p]
        L.orc_ffn_lora.restype = None
        L.orc_fp8_dequantize.argtypes = [u8p, f32p, i64, i64, f64p]
        L.orc_fp8_dequantize.restype = None
        L.orc_gemv_fp8_f64.argtypes = [u16p, i64, i64, u8p, f32p, i64, f64p]
        L.orc_gemv_fp8_f64.restype = None
        L.orc_gemv_fp8.argtypes = [u16p, i64, i64, u8p, f32p, i64, u16p]
        L.orc_gemv_fp8.restype = None
        L.orc_ffn_fp8_hidden.argtypes = [u16p, i64, i64, i64, u8p, f32p, u8p, f32p, ctypes.c_int,
                                         u16p]
        L.orc_ffn_fp8_hidden.restype = None
        L.orc_ffn_fp8.argtypes = [u16p, i64, i64, i64, u8p, f32p, u8p, f32p, u8p, f32p,
                                  ctypes.c_int, u16p]
        L.orc_ffn_fp8.restype = None
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_set_threads.restype = ctypes.c_int
        _lib = L
    return _lib


ACT_SILU = 0
ACT_GELU_TANH = 1


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (0 keeps it); returns the count in use."""
    return lib().orc_set_threads(int(n))


def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(code)


def e4m3_decode(b: int) -> float:
    return lib().orc_e4m3_decode(b)


def e2m1_encode(q: float) -> int:
    return lib().orc_e2m1_encode(q)


def e4m3_encode(q: float) -> int:
    return lib().orc_e4m3_encode(q)


def bf16_decode(b: int) -> float:
    return lib().orc_bf16_decode(b)


def bf16_from_double(v: float) -> int:
    return lib().orc_bf16_from_double(v)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def quantize(w):
    """fp32 [N, K] -> (codes u8 [N, K/2], scales u8 [N, K/16], scale2 float)."""
    w = _c(w, np.float32)
    N, K = w.shape
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    s2 = ctypes.c_float(0.0)
    rc = lib().orc_quantize_f32(w, N, K, codes, scales, ctypes.byref(s2))
    if rc != 0:
        raise ValueError(f"oracle quantize rejected shape {w.shape}")
    return codes, scales, s2.value


def quantize_bf16(w_bits):
    """bf16 bit patterns (uint16) [N, K] -> (codes, scales, scale2)."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    s2 = ctypes.c_float(0.0)
    rc = lib().orc_quantize_bf16(w, N, K, codes, scales, ctypes.byref(s2))
    if rc != 0:
        raise ValueError(f"oracle quantize rejected shape {w.shape}")
    return codes, scales, s2.value


def dequantize(codes, scales, scale2, N, K):
    out = np.zeros((N, K), np.float64)
    lib().orc_dequantize(_c(codes, np.uint8), _c(scales, np.uint8), scale2, N, K, out)
    return out


def gemv_f64(x_bits, codes, scales, scale2, N):
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    y = np.zeros((M, N), np.float64)
    lib().orc_gemv_f64(x, M, K, _c(codes, np.uint8), _c(scales, np.uint8), scale2, N, y)
    return y


def gemv(x_bits, codes, scales, scale2, N):
    """bf16 bits [M, K] -> bf16 bits [M, N]."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    y = np.zeros((M, N), np.uint16)
    lib().orc_gemv(x, M, K, _c(codes, np.uint8), _c(scales, np.uint8), scale2, N, y)
    return y


def silu(t: float) -> float:
    return lib().orc_silu(t)


def gelu_tanh(t: float) -> float:
    return lib().orc_gelu_tanh(t)


def act(t: float, which: int = 0) -> float:
    """SiLU (which=0) or GeLU-tanh (which=1) of one value."""
    return silu(t) if which == ACT_SILU else gelu_tanh(t)


def ffn_hidden(x_bits, I, gate, up, act=ACT_SILU):
    """gate/up = (codes, scales, scale2).  Returns h bf16 bits [M, I]."""
    x = _c(x_bits, np.uint16)
    M, H = x.shape
    h = np.zeros((M, I), np.uint16)
    lib().orc_ffn_hidden(x, M, H, I, _c(gate[0], np.uint8), _c(gate[1], np.uint8), gate[2],
                         _c(up[0], np.uint8), _c(up[1], np.uint8), up[2], int(act), h)
    return h


def ffn(x_bits, I, gate, up, down, act=ACT_SILU):
    """Full FFN; returns out bf16 bits [M, H]."""
    x = _c(x_bits, np.uint16)
    M, H = x.shape
    out = np.zeros((M, H), np.uint16)
    lib().orc_ffn(x, M, H, I, _c(gate[0], np.uint8), _c(gate[1], np.uint8), gate[2],
                  _c(up[0], np.uint8), _c(up[1], np.uint8), up[2],
                  _c(down[0], np.uint8), _c(down[1], np.uint8), down[2], int(act), out)
    return out


def bf16_from_double_array(v):
    """Elementwise bf16_from_double over a float64 array (same shape, uint16)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.zeros(v.shape, np.uint16)
    lib().orc_bf16_from_double_array(v.reshape(-1), v.size, out.reshape(-1))
    return out


def act_array(v, act=ACT_SILU):
    """Elementwise SiLU (act=0) or GeLU-tanh (act=1) over a float64 array."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.zeros(v.shape, np.float64)
    lib().orc_act_array(v.reshape(-1), v.size, int(act), out.reshape(-1))
    return out


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns to float64 (numpy bit shift)."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- LoRA overlay

def lora_xa(v_bits, A_bits):
    """xa bf16 bits [M, r] = bf16(A v) for v bf16 [M, K], A bf16 [r, K]."""
    v = _c(v_bits, np.uint16)
    A = _c(A_bits, np.uint16)
    M, K = v.shape
    r = A.shape[0]
    xa = np.zeros((M, r), np.uint16)
    lib().orc_lora_xa(v, M, K, A, r, xa)
    return xa


def lora_delta(xa_bits, B_bits):
    """delta bf16 bits [M, N] = bf16(B xa) for xa [M, r], B bf16 [N, r]."""
    xa = _c(xa_bits, np.uint16)
    B = _c(B_bits, np.uint16)
    M, r = xa.shape
    N = B.shape[0]
    d = np.zeros((M, N), np.uint16)
    lib().orc_lora_delta(xa, M, r, B, N, d)
    return d


def lora_add(base_bits, delta_bits):
    """bf16(base + delta), elementwise (returns a new array)."""
    out = np.array(base_bits, np.uint16, copy=True, order="C")
    lib().orc_lora_add(out.reshape(-1), _c(delta_bits, np.uint16).reshape(-1), out.size)
    return out


def lora_apply(v_bits, A_bits, B_bits, base_bits):
    """base + dW v with dW = B A (returns a new array)."""
    v = _c(v_bits, np.uint16)
    M, K = v.shape
    A = _c(A_bits, np.uint16)
    B = _c(B_bits, np.uint16)
    out = np.array(base_bits, np.uint16, copy=True, order="C")
    lib().orc_lora_apply(v, M, K, A, B, A.shape[0], B.shape[0], out)
    return out


def ffn_lora(x_bits, I, gate, up, down, act=ACT_SILU, lora=None):
    """FFN with the LoRA overlay.  lora = dict(rank=r, gate=(A, B) or None,
    up=..., down=...) with bf16-bit arrays.  Returns (out [M, H], h [M, I])."""
    x = _c(x_bits, np.uint16)
    M, H = x.shape
    lora = lora or {}
    r = int(lora.get("rank", 1))
    keep = []

    def ptr(pair, i):
        if not pair:
            return None
        a = _c(pair[i], np.uint16)
        keep.append(a)
        return a.ctypes.data

    out = np.zeros((M, H), np.uint16)
    h = np.zeros((M, I), np.uint16)
    lib().orc_ffn_lora(x, M, H, I, _c(gate[0], np.uint8), _c(gate[1], np.uint8), gate[2],
                       _c(up[0], np.uint8), _c(up[1], np.uint8), up[2],
                       _c(down[0], np.uint8), _c(down[1], np.uint8), down[2], int(act), r,
                       ptr(lora.get("gate"), 0), ptr(lora.get("gate"), 1),
                       ptr(lora.get("up"), 0), ptr(lora.get("up"), 1),
                       ptr(lora.get("down"), 0), ptr(lora.get("down"), 1), out, h)
    return out, h


# ---------------------------------------------------------------- block-scaled FP8

def fp8_grid_shape(N, K):
    """Shape of the FP32 block-scale grid of an FP8 projection [N, K]."""
    return (N + 127) // 128, (K + 127) // 128


def fp8_dequantize(q, bs):
    """E4M3 bytes [N, K] and FP32 grid -> weights [N, K] (float64)."""
    q = _c(q, np.uint8)
    N, K = q.shape
    assert tuple(np.shape(bs)) == fp8_grid_shape(N, K)
    w = np.zeros((N, K), np.float64)
    lib().orc_fp8_dequantize(q, _c(bs, np.float32), N, K, w)
    return w


def gemv_fp8_f64(x_bits, q, bs):
    x = _c(x_bits, np.uint16)
    q = _c(q, np.uint8)
    M, K = x.shape
    N = q.shape[0]
    assert q.shape[1] == K and tuple(np.shape(bs)) == fp8_grid_shape(N, K)
    y = np.zeros((M, N), np.float64)
    lib().orc_gemv_fp8_f64(x, M, K, q, _c(bs, np.float32), N, y)
    return y


def gemv_fp8(x_bits, q, bs):
    """bf16 bits [M, K] x FP8 projection (q [N, K], grid) -> bf16 bits [M, N]."""
    x = _c(x_bits, np.uint16)
    q = _c(q, np.uint8)
    M, K = x.shape
    N = q.shape[0]
    assert q.shape[1] == K and tuple(np.shape(bs)) == fp8_grid_shape(N, K)
    y = np.zeros((M, N), np.uint16)
    lib().orc_gemv_fp8(x, M, K, q, _c(bs, np.float32), N, y)
    return y


def ffn_fp8_hidden(x_bits, gate, up, act=ACT_SILU):
    """gate/up = (q [I, H], grid).  Returns h bf16 bits [M, I]."""
    x = _c(x_bits, np.uint16)
    M, H = x.shape
    I = gate[0].shape[0]
    h = np.zeros((M, I), np.uint16)
    lib().orc_ffn_fp8_hidden(x, M, H, I, _c(gate[0], np.uint8), _c(gate[1], np.float32),
                             _c(up[0], np.uint8), _c(up[1], np.float32), int(act), h)
    return h


def ffn_fp8(x_bits, gate, up, down, act=ACT_SILU):
    """Full FP8 FFN; returns out bf16 bits [M, H]."""
    x = _c(x_bits, np.uint16)
    M, H = x.shape
    I = gate[0].shape[0]
    out = np.zeros((M, H), np.uint16)
    lib().orc_ffn_fp8(x, M, H, I, _c(gate[0], np.uint8), _c(gate[1], np.float32),
                      _c(up[0], np.uint8), _c(up[1], np.float32),
                      _c(down[0], np.uint8), _c(down[1], np.float32), int(act), out)
    return out
