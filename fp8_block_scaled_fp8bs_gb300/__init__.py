"""FP8 block-scaled linear-layer path for NVIDIA GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/fp8bs.h`` (``libfp8bs.so``, built in place
by ``fp8_block_scaled_fp8bs_gb300.build``). Every step of the path runs in the library's CUDA
kernels; this module only marshals arguments. There is no CPU fallback: if the library is
missing or cannot be loaded, importing the binding's functions raises.

Raw entry points (same names and arguments as the C functions; pointers are ints):
    fp8bs_act_quant(x, y, s, M, K, scale_fmt, stream)
    fp8bs_weight_dequant(w, s, y, N, K, stream)
    fp8bs_gemm(a, a_s, b, b_s, c, M, N, K, scale_fmt, stream)
    fp8bs_gemm_ex(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags, stream)
    fp8bs_gemm_plan(M, N, K, scale_fmt, with_workspace) -> dict
    fp8bs_gemm_config(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags, kernel, tile, ksplit,
                      workspace, workspace_bytes, stream)
    fp8bs_gemm_grouped(a, a_s, b, b_s, c, row_offsets, groups, N, K, scale_fmt, stream)
    fp8bs_device_error(clear=True, stream=0) -> int
    fp8bs_probe_wait_timeout(timeout_ns, stream)
Tensor conveniences (PyTorch CUDA tensors; outputs allocated with torch):
    act_quant(x, scale_fmt="fp32") -> (y, s)      ("DeepSeek-V3 Administrator & Developer
    weight_dequant(w, s) -> y                        Guide", §8.5.1, §8.5.2, §8.5.3)
    fp8_gemm(a, a_s, b, b_s, scale_fmt="fp32") -> c
    fp8_gemm_grouped(a, a_s, b, b_s, row_offsets, scale_fmt="fp32") -> c
"""
from __future__ import annotations

import ctypes
import os
import threading

BLOCK = 128
SCALE_FP32 = 0
SCALE_UE8M0 = 1
STATUS = {0: "ok", 1: "invalid argument", 2: "pointer not aligned",
          3: "unsupported device (needs sm_103)", 4: "CUDA error"}
DEVERR_SCALE_NOT_POW2 = 0x10
DEVERR_PROBE = 0x100

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8bs.so")
GEMM_WEIGHTS_CONSTANT = 0x1
GEMM_QUANT_IN_KERNEL = 0x2
KERNEL_SWAPPED, KERNEL_PROMOTED, KERNEL_BLOCK_SCALED, KERNEL_BLOCK_SCALED_PAIR = 0, 1, 2, 3
EXPORTS = ("fp8bs_act_quant", "fp8bs_weight_dequant", "fp8bs_gemm", "fp8bs_gemm_ex",
           "fp8bs_gemm_ws", "fp8bs_gemm_workspace_size", "fp8bs_gemm_plan", "fp8bs_gemm_config",
           "fp8bs_gemm_noalloc",
           "fp8bs_act_quant_gemm", "fp8bs_linear_bf16",
           "fp8bs_gemm_grouped",
           "fp8bs_status_string", "fp8bs_device_error", "fp8bs_probe_wait_timeout",
           "fp8bs_probe_occupy")

_lock = threading.Lock()
_lib = None


class Fp8bsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} (status {status})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libfp8bs.so (building it first if it is missing and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            from . import build as _build
            _build.build()
        lib = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.fp8bs_act_quant.argtypes = [vp, vp, vp, i64, i64, i32, vp]
        lib.fp8bs_weight_dequant.argtypes = [vp, vp, vp, i64, i64, vp]
        lib.fp8bs_gemm.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]
        lib.fp8bs_gemm_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, ctypes.c_uint, vp]
        lib.fp8bs_gemm_ws.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, ctypes.c_uint, vp,
                                      ctypes.c_size_t, vp]
        lib.fp8bs_gemm_workspace_size.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
        ip = ctypes.POINTER(ctypes.c_int)
        lib.fp8bs_gemm_plan.argtypes = [i64, i64, i64, i32, i32, ip, ip, ip, ip]
        lib.fp8bs_gemm_config.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, ctypes.c_uint,
                                          i32, i32, i32, vp, ctypes.c_size_t, vp]
        lib.fp8bs_linear_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, ctypes.c_uint, vp]
        lib.fp8bs_act_quant_gemm.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                             ctypes.c_uint, vp, ctypes.c_size_t, vp]
        lib.fp8bs_gemm_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, ctypes.c_uint,
                                           vp]
        lib.fp8bs_gemm_grouped.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_int64),
                                           i64, i64, i64, i32, vp]
        lib.fp8bs_status_string.argtypes = [i32]
        lib.fp8bs_status_string.restype = ctypes.c_char_p
        lib.fp8bs_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), i32, vp]
        lib.fp8bs_probe_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.fp8bs_probe_occupy.argtypes = [i32, ctypes.c_uint64, vp]
        for name in EXPORTS:
            getattr(lib, name).restype = getattr(lib, name).restype or i32
        lib.fp8bs_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise Fp8bsError(fn, status)


# ----------------------------------------------------------------------- raw entry points

def fp8bs_act_quant(x, y, s, M, K, scale_fmt=SCALE_FP32, stream=0) -> None:
    _check("fp8bs_act_quant", load().fp8bs_act_quant(x, y, s, M, K, scale_fmt, stream))


def fp8bs_weight_dequant(w, s, y, N, K, stream=0) -> None:
    _check("fp8bs_weight_dequant", load().fp8bs_weight_dequant(w, s, y, N, K, stream))


def fp8bs_gemm(a, a_s, b, b_s, c, M, N, K, scale_fmt=SCALE_FP32, stream=0) -> None:
    _check("fp8bs_gemm", load().fp8bs_gemm(a, a_s, b, b_s, c, M, N, K, scale_fmt, stream))


def fp8bs_gemm_ex(a, a_s, b, b_s, c, M, N, K, scale_fmt=SCALE_FP32, flags=0, stream=0) -> None:
    _check("fp8bs_gemm_ex", load().fp8bs_gemm_ex(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags,
                                                 stream))


def fp8bs_gemm_ws(a, a_s, b, b_s, c, M, N, K, scale_fmt=SCALE_FP32, flags=0, workspace=0,
                  workspace_bytes=0, stream=0) -> None:
    _check("fp8bs_gemm_ws", load().fp8bs_gemm_ws(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags,
                                                 workspace, workspace_bytes, stream))


def fp8bs_gemm_noalloc(a, a_s, b, b_s, c, M, N, K, scale_fmt=SCALE_FP32, flags=0,
                       stream=0) -> None:
    _check("fp8bs_gemm_noalloc", load().fp8bs_gemm_noalloc(a, a_s, b, b_s, c, M, N, K,
                                                           scale_fmt, flags, stream))


def fp8bs_act_quant_gemm(x, y, s, b, b_s, c, M, N, K, scale_fmt=SCALE_FP32, flags=0,
                         workspace=0, workspace_bytes=0, stream=0) -> None:
    _check("fp8bs_act_quant_gemm", load().fp8bs_act_quant_gemm(
        x, y, s, b, b_s, c, M, N, K, scale_fmt, flags, workspace, workspace_bytes, stream))


def fp8bs_linear_bf16(x, w, w_s, y, M, N, K, flags=0, stream=0) -> None:
    _check("fp8bs_linear_bf16", load().fp8bs_linear_bf16(x, w, w_s, y, M, N, K, flags, stream))


def fp8bs_gemm_workspace_size() -> int:
    out = ctypes.c_size_t(0)
    _check("fp8bs_gemm_workspace_size", load().fp8bs_gemm_workspace_size(ctypes.byref(out)))
    return out.value


def fp8bs_gemm_plan(M, N, K, scale_fmt=SCALE_FP32, with_workspace=True) -> dict:
    """The kernel, tile, K split and stream-K choice fp8bs_gemm_ws (with_workspace) or
    fp8bs_gemm_ex would make for this shape on the current device."""
    out = [ctypes.c_int(0) for _ in range(4)]
    _check("fp8bs_gemm_plan", load().fp8bs_gemm_plan(M, N, K, scale_fmt, int(with_workspace),
                                                     *[ctypes.byref(o) for o in out]))
    return {"kernel": out[0].value, "tile": out[1].value, "ksplit": out[2].value,
            "stream_k": bool(out[3].value)}


def fp8bs_gemm_config(a, a_s, b, b_s, c, M, N, K, scale_fmt=SCALE_FP32, flags=0,
                      kernel=KERNEL_PROMOTED, tile=128, ksplit=1, workspace=0, workspace_bytes=0,
                      stream=0) -> None:
    _check("fp8bs_gemm_config", load().fp8bs_gemm_config(
        a, a_s, b, b_s, c, M, N, K, scale_fmt, flags, kernel, tile, ksplit, workspace,
        workspace_bytes, stream))


def fp8bs_gemm_grouped(a, a_s, b, b_s, c, row_offsets, groups, N, K, scale_fmt=SCALE_FP32,
                       stream=0) -> None:
    """row_offsets: a sequence of groups+1 ints (host memory)."""
    offs = (ctypes.c_int64 * (int(groups) + 1))(*[int(x) for x in row_offsets])
    _check("fp8bs_gemm_grouped", load().fp8bs_gemm_grouped(a, a_s, b, b_s, c, offs, groups, N, K,
                                                           scale_fmt, stream))


def fp8bs_device_error(clear: bool = True, stream=0) -> int:
    out = ctypes.c_uint(0)
    _check("fp8bs_device_error", load().fp8bs_device_error(ctypes.byref(out), int(clear), stream))
    return out.value


def fp8bs_probe_wait_timeout(timeout_ns: int, stream=0) -> None:
    _check("fp8bs_probe_wait_timeout", load().fp8bs_probe_wait_timeout(timeout_ns, stream))


def fp8bs_probe_occupy(ctas: int, duration_ns: int, stream=0) -> None:
    _check("fp8bs_probe_occupy", load().fp8bs_probe_occupy(ctas, duration_ns, stream))


# ----------------------------------------------------------------------- tensor helpers

def _fmt(scale_fmt) -> int:
    if scale_fmt in (SCALE_FP32, "fp32", None):
        return SCALE_FP32
    if scale_fmt in (SCALE_UE8M0, "ue8m0"):
        return SCALE_UE8M0
    raise ValueError(f"unknown scale_fmt {scale_fmt!r}")


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _require(t, dtype, ndim, name, host_ok=False):
    """t must be a contiguous CUDA tensor of dtype and rank ndim; with host_ok, a pinned host
    tensor is accepted too (the kernels that read x or write C reach pinned host memory in
    place)."""
    import torch
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (host_ok and t.is_pinned())):
        raise TypeError(f"{name} must be a CUDA tensor" + (" or a pinned host tensor" if host_ok
                                                          else ""))
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def _output(out, shape, device):
    """The bf16 output: a new CUDA tensor, or the caller's `out` (CUDA or pinned host), checked
    to be a contiguous bf16 tensor of exactly `shape` so that no kernel writes past its end."""
    import torch
    if out is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=device)
    _require(out, torch.bfloat16, len(shape), "out", host_ok=True)
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out must have shape {tuple(shape)}, got {tuple(out.shape)}")
    return out


def _workspace_args(workspace):
    """(pointer, bytes) of a stream-K workspace: None, or a contiguous uint8 CUDA tensor (its
    size is checked by the library against fp8bs_gemm_workspace_size)."""
    import torch
    if workspace is None:
        return 0, 0
    _require(workspace, torch.uint8, workspace.dim() if isinstance(workspace, torch.Tensor) else 1,
             "workspace")
    return workspace.data_ptr(), workspace.numel()


def _cuda_device(*tensors):
    import torch
    for t in tensors:
        if t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def act_quant(x, scale_fmt="fp32"):
    """x: bf16 [M,K] (K % 128 == 0) -> (y float8_e4m3fn [M,K], s float32 [M,K/128])."""
    import torch
    _require(x, torch.bfloat16, 2, "x", host_ok=True)
    M, K = x.shape
    dev = _cuda_device(x)
    y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    s = torch.empty((M, K // BLOCK), dtype=torch.float32, device=dev)
    fp8bs_act_quant(x.data_ptr(), y.data_ptr(), s.data_ptr(), M, K, _fmt(scale_fmt), _stream())
    return y, s


def weight_dequant(w, s):
    """w: float8_e4m3fn [N,K], s: float32 [ceil(N/128), ceil(K/128)] -> bf16 [N,K]."""
    import torch
    _require(w, torch.float8_e4m3fn, 2, "w")
    _require(s, torch.float32, 2, "s")
    N, K = w.shape
    if tuple(s.shape) != (-(-N // BLOCK), -(-K // BLOCK)):
        raise ValueError(f"scale shape {tuple(s.shape)} does not match weight {tuple(w.shape)}")
    y = torch.empty((N, K), dtype=torch.bfloat16, device=w.device)
    fp8bs_weight_dequant(w.data_ptr(), s.data_ptr(), y.data_ptr(), N, K, _stream())
    return y


_workspaces = {}


def gemm_workspace(device=None, stream=None):
    """The zero-filled workspace fp8_gemm uses on `device` for calls on `stream` (one per
    device and stream, so that calls that may overlap never share one), allocated on first use."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = (dev.index, stream if stream is not None else _stream())
    ws = _workspaces.get(key)
    if ws is None:
        with torch.cuda.device(dev):
            ws = torch.zeros(fp8bs_gemm_workspace_size(), dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def fp8_gemm(a, a_s, b, b_s, scale_fmt="fp32", out=None, weights_constant=False,
             workspace="auto"):
    """C[M,N] bf16 = A[M,K] . B[N,K]^T with per-128-K-block scales a_s [M,K/128] and
    b_s [ceil(N/128), K/128]. workspace: "auto" (a cached one per device and stream), None (no
    split K loops) or a zero-filled uint8 CUDA tensor of fp8bs_gemm_workspace_size() bytes."""
    import torch
    _require(a, torch.float8_e4m3fn, 2, "a")
    _require(b, torch.float8_e4m3fn, 2, "b")
    _require(a_s, torch.float32, 2, "a_s")
    _require(b_s, torch.float32, 2, "b_s")
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K or tuple(a_s.shape) != (M, K // BLOCK) or \
            tuple(b_s.shape) != (-(-N // BLOCK), K // BLOCK):
        raise ValueError("operand or scale shapes do not match")
    c = _output(out, (M, N), a.device)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = gemm_workspace(a.device)
    ws_ptr, ws_bytes = _workspace_args(workspace)
    fp8bs_gemm_ws(a.data_ptr(), a_s.data_ptr(), b.data_ptr(), b_s.data_ptr(), c.data_ptr(),
                  M, N, K, _fmt(scale_fmt), GEMM_WEIGHTS_CONSTANT if weights_constant else 0,
                  ws_ptr, ws_bytes, _stream())
    return c


def act_quant_gemm(x, b, b_s, scale_fmt="fp32", weights_constant=False, workspace="auto",
                   quant_in_kernel=False, out=None):
    """linear() on the FP8 path: x bf16 [M,K] -> (c bf16 [M,N], y e4m3 [M,K], s fp32
    [M,K/128]): act_quant then the GEMM (quant_in_kernel: one kernel, M <= 16); see fp8_gemm
    for `workspace`. x and `out` (c) may be pinned host tensors."""
    import torch
    _require(x, torch.bfloat16, 2, "x", host_ok=True)
    _require(b, torch.float8_e4m3fn, 2, "b")
    _require(b_s, torch.float32, 2, "b_s")
    M, K = x.shape
    N = b.shape[0]
    if b.shape[1] != K or tuple(b_s.shape) != (-(-N // BLOCK), K // BLOCK):
        raise ValueError("operand or scale shapes do not match")
    y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=b.device)
    s = torch.empty((M, K // BLOCK), dtype=torch.float32, device=b.device)
    c = _output(out, (M, N), b.device)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = gemm_workspace(b.device)
    ws_ptr, ws_bytes = _workspace_args(workspace)
    flags = (GEMM_WEIGHTS_CONSTANT if weights_constant else 0) | \
        (GEMM_QUANT_IN_KERNEL if quant_in_kernel else 0)
    fp8bs_act_quant_gemm(x.data_ptr(), y.data_ptr(), s.data_ptr(), b.data_ptr(), b_s.data_ptr(),
                         c.data_ptr(), M, N, K, _fmt(scale_fmt), flags, ws_ptr, ws_bytes,
                         _stream())
    return c, y, s


def linear_bf16(x, w, w_s, weights_constant=False, out=None):
    """bf16 path of linear(): x bf16 [M,K] . bf16(dequant(w, w_s))^T -> y bf16 [M,N]."""
    import torch
    _require(x, torch.bfloat16, 2, "x")
    _require(w, torch.float8_e4m3fn, 2, "w")
    _require(w_s, torch.float32, 2, "w_s")
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or tuple(w_s.shape) != (-(-N // BLOCK), -(-K // BLOCK)):
        raise ValueError("operand or scale shapes do not match")
    y = _output(out, (M, N), x.device)
    fp8bs_linear_bf16(x.data_ptr(), w.data_ptr(), w_s.data_ptr(), y.data_ptr(), M, N, K,
                      GEMM_WEIGHTS_CONSTANT if weights_constant else 0, _stream())
    return y


def fp8_gemm_grouped(a, a_s, b, b_s, row_offsets, scale_fmt="fp32", out=None):
    """Per-group block-scaled GEMMs: a [T,K] e4m3 with rows grouped by row_offsets (groups+1
    host ints), b [G,N,K] e4m3, b_s [G, ceil(N/128), K/128] -> c [T,N] bf16."""
    import torch
    _require(a, torch.float8_e4m3fn, 2, "a")
    _require(b, torch.float8_e4m3fn, 3, "b")
    _require(a_s, torch.float32, 2, "a_s")
    _require(b_s, torch.float32, 3, "b_s")
    T, K = a.shape
    G, N = b.shape[0], b.shape[1]
    offs = [int(x) for x in row_offsets]
    if len(offs) != G + 1 or offs[0] != 0 or offs[-1] != T or b.shape[2] != K or \
            tuple(a_s.shape) != (T, K // BLOCK) or tuple(b_s.shape) != (G, -(-N // BLOCK), K // BLOCK):
        raise ValueError("operand, scale or offset shapes do not match")
    c = _output(out, (T, N), a.device)
    fp8bs_gemm_grouped(a.data_ptr(), a_s.data_ptr(), b.data_ptr(), b_s.data_ptr(), c.data_ptr(),
                       offs, G, N, K, _fmt(scale_fmt), _stream())
    return c
