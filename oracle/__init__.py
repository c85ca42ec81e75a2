"""CPU oracle for the FP8 block-scaled linear path (act_quant, weight_dequant, fp8_gemm).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package. It wraps ``oracle.c`` (plain single-threaded C,
binary64 arithmetic) through ctypes and shares no code with the CUDA library.

Sources: "DeepSeek-V3 Administrator & Developer Guide" §8.5.1-§8.5.3 (the three kernels) and
§6.3 (scale shapes); "DeepSeek-V3 User Guide", FAQ "What is scale_fmt: ue8m0?".

Arrays are numpy, row-major and contiguous: bf16 values travel as their uint16 bit patterns,
e4m3fn values as uint8 codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

SCALE_FP32 = 0
SCALE_UE8M0 = 1
BLOCK = 128

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u8p = ctypes.POINTER(ctypes.c_uint8)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_float.restype = ctypes.c_float
            lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_f32_div.argtypes = [ctypes.c_float, ctypes.c_float]
            lib.oracle_f32_div.restype = ctypes.c_float
            lib.oracle_act_quant.argtypes = [u16p, u8p, f32p, i64, i64, ctypes.c_int]
            lib.oracle_act_quant.restype = None
            lib.oracle_weight_dequant.argtypes = [u8p, f32p, u16p, i64, i64]
            lib.oracle_weight_dequant.restype = None
            lib.oracle_gemm.argtypes = [u8p, f32p, u8p, f32p, f64p, i64, i64, i64]
            lib.oracle_gemm.restype = None
            lib.oracle_gemm_at.argtypes = [u8p, f32p, u8p, f32p, i64p, i64p, i64, f64p,
                                           i64, i64, i64]
            lib.oracle_gemm_at.restype = None
            _lib = lib
    return _lib


def _ptr(arr: np.ndarray, ctype):
    assert arr.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return arr.ctypes.data_as(ctypes.POINTER(ctype))


def _as(arr, dtype) -> np.ndarray:
    a = np.ascontiguousarray(arr)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


# ------------------------------------------------------------------------ scalar codecs

def e4m3_decode(code: int) -> float:
    """Value of one e4m3fn code (NaN for 0x7F and 0xFF)."""
    return _load().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    """RNE, saturating binary32 -> e4m3fn code (the argument is first rounded to binary32)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(v))))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(v, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_e4m3_encode(float(x)) for x in flat), dtype=np.uint8,
                       count=flat.size).reshape(np.shape(v))


def bf16_rne(f: float) -> int:
    """bf16 bit pattern nearest the binary32 value f (ties to even)."""
    return int(_load().oracle_bf16_rne(float(np.float32(f))))


def bf16_to_float(h: int) -> float:
    return float(_load().oracle_bf16_to_float(int(h) & 0xFFFF))


def f32_div(a: float, b: float) -> float:
    return float(_load().oracle_f32_div(float(np.float32(a)), float(np.float32(b))))


# ------------------------------------------------------------------------ the path

def act_quant(x_bf16_bits: np.ndarray, scale_fmt: int = SCALE_FP32):
    """x: uint16 [M,K] (bf16 bit patterns), K % 128 == 0 -> (y uint8 [M,K], s float32 [M,K/128])."""
    x = _as(x_bf16_bits, np.uint16)
    if x.ndim != 2:
        raise ValueError("act_quant takes a 2-D input")
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 128")
    y = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, K // BLOCK), dtype=np.float32)
    _load().oracle_act_quant(_ptr(x, ctypes.c_uint16), _ptr(y, ctypes.c_uint8),
                             _ptr(s, ctypes.c_float), M, K, int(scale_fmt))
    return y, s


def weight_dequant(w: np.ndarray, s: np.ndarray) -> np.ndarray:
    """w: uint8 [N,K] e4m3 codes, s: float32 [ceil(N/128), ceil(K/128)] -> uint16 [N,K] bf16 bits."""
    w = _as(w, np.uint8)
    s = _as(s, np.float32)
    N, K = w.shape
    if s.shape != (-(-N // BLOCK), -(-K // BLOCK)):
        raise ValueError(f"scale shape {s.shape} does not match weight {w.shape}")
    y = np.empty((N, K), dtype=np.uint16)
    _load().oracle_weight_dequant(_ptr(w, ctypes.c_uint8), _ptr(s, ctypes.c_float),
                                  _ptr(y, ctypes.c_uint16), N, K)
    return y


def _gemm_args(a, a_s, b, b_s):
    a = _as(a, np.uint8)
    b = _as(b, np.uint8)
    a_s = _as(a_s, np.float32)
    b_s = _as(b_s, np.float32)
    M, K = a.shape
    N, Kb = b.shape
    if Kb != K or K % BLOCK:
        raise ValueError("A and B must share K, a multiple of 128")
    if a_s.shape != (M, K // BLOCK) or b_s.shape != (-(-N // BLOCK), K // BLOCK):
        raise ValueError("scale shapes do not match A/B")
    return a, a_s, b, b_s, M, N, K


def gemm(a, a_s, b, b_s) -> np.ndarray:
    """Block-scaled C = A B^T in binary64: float64 [M,N]."""
    a, a_s, b, b_s, M, N, K = _gemm_args(a, a_s, b, b_s)
    c = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm(_ptr(a, ctypes.c_uint8), _ptr(a_s, ctypes.c_float),
                        _ptr(b, ctypes.c_uint8), _ptr(b_s, ctypes.c_float),
                        _ptr(c, ctypes.c_double), M, N, K)
    return c


def gemm_at(a, a_s, b, b_s, mi, ni) -> np.ndarray:
    """The same sum at the chosen output positions (mi[i], ni[i]): float64 [count]."""
    a, a_s, b, b_s, M, N, K = _gemm_args(a, a_s, b, b_s)
    mi = _as(np.asarray(mi, dtype=np.int64), np.int64)
    ni = _as(np.asarray(ni, dtype=np.int64), np.int64)
    if mi.shape != ni.shape or mi.ndim != 1:
        raise ValueError("mi and ni must be 1-D and of equal length")
    if mi.size and (mi.min() < 0 or mi.max() >= M or ni.min() < 0 or ni.max() >= N):
        raise IndexError("sample position out of range")
    out = np.empty(mi.shape, dtype=np.float64)
    _load().oracle_gemm_at(_ptr(a, ctypes.c_uint8), _ptr(a_s, ctypes.c_float),
                           _ptr(b, ctypes.c_uint8), _ptr(b_s, ctypes.c_float),
                           _ptr(mi, ctypes.c_int64), _ptr(ni, ctypes.c_int64), mi.size,
                           _ptr(out, ctypes.c_double), M, N, K)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> their values as float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def linear_bf16(x: np.ndarray, w: np.ndarray, w_s: np.ndarray) -> np.ndarray:
    """The bf16 path of linear() ("DeepSeek-V3 Administrator & Developer Guide", §6.3,
    gemm_impl = "bf16"): the weight dequantised to bf16 as weight_dequant does (§8.5.2), then
    x . W'^T. x: uint16 [M,K] bf16 bits, w: uint8 [N,K] codes, w_s: float32 scales ->
    float64 [M,N], the exact product (binary64 matmul of bf16 values: every product is exact
    and K <= 2^16 sums of them stay within binary64's 53 bits to well below the tolerance)."""
    wd = bf16_bits_to_f64(weight_dequant(w, w_s))
    xd = bf16_bits_to_f64(x)
    return xd @ wd.T
