"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, exports every
function that include/*.h declares, and rejects bad arguments before touching the device."""
import ctypes
import glob
import os
import re

import pytest

import fp8_block_scaled_fp8bs_gb300 as fp8bs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, MISALIGNED, UNSUPPORTED, CUDA = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    return fp8bs.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"FP8BS_API\s+[\w\s\*]+?\b(fp8bs_\w+)\s*\(", text)
    return sorted(set(names))


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"fp8bs_act_quant", "fp8bs_weight_dequant", "fp8bs_gemm"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code, text in fp8bs.STATUS.items():
        assert lib.fp8bs_status_string(code).decode() == text
    assert lib.fp8bs_status_string(99) == b"unknown status"


A16, B16, C16 = 0x10000, 0x20000, 0x30000  # fake, 16-byte aligned; never dereferenced


@pytest.mark.parametrize("args,expect", [
    ((A16, B16, C16, 4, 100, 0), INVALID),   # K % 128
    ((A16, B16, C16, -1, 128, 0), INVALID),  # negative M
    ((A16, B16, C16, 4, 128, 7), INVALID),   # bad scale format
    ((None, B16, C16, 4, 128, 0), INVALID),  # null input
    ((A16 + 2, B16, C16, 4, 128, 0), MISALIGNED),
    ((A16, B16 + 8, C16, 4, 128, 0), MISALIGNED),
    ((A16, B16, C16 + 2, 4, 128, 0), MISALIGNED),
    ((None, None, None, 0, 128, 0), OK),     # empty: no-op
    ((None, None, None, 4, 0, 0), OK),
])
def test_act_quant_argument_checks(lib, args, expect):
    assert lib.fp8bs_act_quant(*args, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, B16, C16, -1, 5), INVALID),
    ((None, B16, C16, 3, 5), INVALID),
    ((A16, B16 + 1, C16, 3, 5), MISALIGNED),
    ((A16 + 4, B16, C16, 3, 32), MISALIGNED),  # vector path needs 16-byte alignment
    ((None, None, None, 0, 5), OK),
])
def test_weight_dequant_argument_checks(lib, args, expect):
    assert lib.fp8bs_weight_dequant(*args, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, B16, C16, B16, C16, 8, 256, 200, 0), INVALID),       # K % 128
    ((A16, B16, C16, B16, C16, 8, -2, 256, 0), INVALID),
    ((A16, B16, C16, B16, C16, 8, 256, 256, 3), INVALID),
    ((A16, B16, None, B16, C16, 8, 256, 256, 0), INVALID),
    ((A16, B16, C16, B16, None, 8, 256, 256, 0), INVALID),
    ((A16 + 8, B16, C16, B16, C16, 8, 256, 256, 0), MISALIGNED),
    ((A16, B16, C16 + 4, B16, C16, 8, 256, 256, 0), MISALIGNED),
    ((A16, B16 + 2, C16, B16, C16, 8, 256, 256, 0), MISALIGNED),
    ((A16, B16, C16, B16, C16 + 8, 8, 256, 256, 0), MISALIGNED),
    ((None, None, None, None, None, 0, 256, 256, 0), OK),
    ((None, None, None, None, None, 8, 0, 256, 0), OK),
    ((A16, B16, C16, B16, C16, 1 << 32, 256, 256, 0), INVALID),  # beyond 32-bit coordinates
])
def test_gemm_argument_checks(lib, args, expect):
    assert lib.fp8bs_gemm(*args, None) == expect


def test_valid_call_without_a_gpu_reports_an_error_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.fp8bs_act_quant(A16, B16, C16, 4, 128, 0, None) in (CUDA, UNSUPPORTED)
    assert lib.fp8bs_gemm(A16, B16, C16, B16, C16, 8, 256, 256, 0, None) in (CUDA, UNSUPPORTED)


def test_python_binding_raises_on_error_status():
    with pytest.raises(fp8bs.Fp8bsError) as ei:
        fp8bs.fp8bs_gemm(A16, B16, C16, B16, C16, 8, 256, 200)
    assert ei.value.status == INVALID


def test_product_package_does_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "fp8_block_scaled_fp8bs_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if os.path.isfile(path) and path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            text = open(path).read()
            assert "import oracle" not in text and "oracle." not in text, path
            assert "liboracle" not in text, path


def _offs(*v):
    return (ctypes.c_int64 * len(v))(*v)


@pytest.mark.parametrize("offs,groups,N,K,expect", [
    ((0, 4, 9), 2, 256, 100, INVALID),            # K % 128
    ((0, 4, 9), 2, -1, 256, INVALID),
    ((0, 4, 9), 300, 256, 256, INVALID),          # more groups than supported
    ((1, 4, 9), 2, 256, 256, INVALID),            # offsets must start at 0
    ((0, 5, 3), 2, 256, 256, INVALID),            # offsets must not decrease
    ((0, 0, 0), 2, 256, 256, OK),                 # no rows: no-op
    ((0,), 0, 256, 256, OK),                      # no groups: no-op
])
def test_gemm_grouped_argument_checks(lib, offs, groups, N, K, expect):
    assert lib.fp8bs_gemm_grouped(A16, B16, C16, B16, C16, _offs(*offs), groups, N, K, 0,
                                  None) == expect


def test_gemm_grouped_rejects_misaligned_and_null(lib):
    o = _offs(0, 3, 8)
    assert lib.fp8bs_gemm_grouped(A16 + 4, B16, C16, B16, C16, o, 2, 256, 256, 0, None) == MISALIGNED
    assert lib.fp8bs_gemm_grouped(A16, B16, C16, B16, None, o, 2, 256, 256, 0, None) == INVALID
    assert lib.fp8bs_gemm_grouped(A16, B16, C16, B16, C16, None, 2, 256, 256, 0, None) == INVALID


def test_gemm_ex_rejects_unknown_flags(lib):
    assert lib.fp8bs_gemm_ex(A16, B16, C16, B16, C16, 8, 256, 256, 0, 0x2, None) == INVALID
    # FP8BS_GEMM_QUANT_IN_KERNEL (0x2) belongs to fp8bs_act_quant_gemm only
    assert lib.fp8bs_gemm_ex(None, None, None, None, None, 0, 256, 256, 0, 0x1, None) == OK


@pytest.mark.parametrize("args,expect", [
    ((A16, B16, C16, B16, C16, 8, 256, 200, 0, 0), INVALID),      # K % 128
    ((A16, B16, C16, B16, C16, 8, 256, 256, 0, 0x2), INVALID),    # unknown flag
    ((A16, B16, C16, B16, C16, -1, 256, 256, 0, 0), INVALID),
    ((A16 + 8, B16, C16, B16, C16, 8, 256, 256, 0, 0), MISALIGNED),
    ((None, None, None, None, None, 0, 256, 256, 1, 0), OK),
])
def test_gemm_ws_argument_checks(lib, args, expect):
    """fp8bs_gemm_ws checks its arguments as fp8bs_gemm_ex does, with or without a workspace."""
    for ws, nbytes in ((None, 0), (C16, 1 << 24)):
        assert lib.fp8bs_gemm_ws(*args, ws, nbytes, None) == expect


def test_gemm_workspace_size_without_a_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    out = ctypes.c_size_t(0)
    assert lib.fp8bs_gemm_workspace_size(ctypes.byref(out)) in (CUDA, UNSUPPORTED)
    assert lib.fp8bs_gemm_workspace_size(None) == INVALID


@pytest.mark.parametrize("args,expect", [
    ((A16, B16, C16, B16, C16, C16, 8, 256, 200, 0, 0), INVALID),    # K % 128
    ((A16, B16, C16, B16, C16, C16, 8, 256, 256, 2, 0), INVALID),    # bad scale_fmt
    ((A16, B16, C16, B16, C16, C16, 8, 256, 256, 0, 0x4), INVALID),  # unknown flag
    ((A16 + 8, B16, C16, B16, C16, C16, 8, 256, 256, 0, 0), MISALIGNED),
    ((A16, B16 + 4, C16, B16, C16, C16, 8, 256, 256, 0, 0), MISALIGNED),
    ((A16, None, C16, B16, C16, C16, 8, 256, 256, 0, 0), INVALID),
    ((None, None, None, None, None, None, 0, 256, 256, 0, 0), OK),
])
def test_act_quant_gemm_argument_checks(lib, args, expect):
    assert lib.fp8bs_act_quant_gemm(*args, None, 0, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, B16, C16, C16, 8, 256, 200, 0), INVALID),      # K % 128
    ((A16, B16, C16, C16, 8, 256, 256, 0x2), INVALID),    # unknown flag
    ((A16 + 2, B16, C16, C16, 8, 256, 256, 0), MISALIGNED),
    ((A16, B16, C16 + 2, C16, 8, 256, 256, 0), MISALIGNED),
    ((A16, None, C16, C16, 8, 256, 256, 0), INVALID),
    ((None, None, None, None, 0, 256, 256, 0), OK),
])
def test_linear_bf16_argument_checks(lib, args, expect):
    assert lib.fp8bs_linear_bf16(*args, None) == expect


def test_gemm_plan_argument_checks(lib):
    """fp8bs_gemm_plan checks its arguments before looking at the device."""
    out = [ctypes.c_int(0) for _ in range(4)]
    refs = [ctypes.byref(o) for o in out]
    assert lib.fp8bs_gemm_plan(8, 256, 200, 0, 1, *refs) == INVALID       # K % 128
    assert lib.fp8bs_gemm_plan(0, 256, 256, 0, 1, *refs) == INVALID       # empty shape
    assert lib.fp8bs_gemm_plan(8, 256, 256, 3, 1, *refs) == INVALID       # bad scale_fmt
    assert lib.fp8bs_gemm_plan(8, 256, 256, 0, 1, None, *refs[1:]) == INVALID
    import torch
    if not torch.cuda.is_available():
        assert lib.fp8bs_gemm_plan(8, 256, 256, 0, 1, *refs) in (CUDA, UNSUPPORTED)


@pytest.mark.parametrize("args,expect", [
    ((A16, B16, C16, B16, C16, 8, 256, 200, 0, 0, 1, 128, 1), INVALID),      # K % 128
    ((A16, B16, C16, B16, C16, 8, 256, 256, 0, 0x2, 1, 128, 1), INVALID),    # unknown flag
    ((A16 + 8, B16, C16, B16, C16, 300, 256, 256, 0, 0, 1, 128, 1), MISALIGNED),
    ((None, None, None, None, None, 0, 256, 256, 0, 0, 1, 128, 1), OK),      # empty: no-op
])
def test_gemm_config_argument_checks(lib, args, expect):
    """fp8bs_gemm_config checks the arguments it shares with fp8bs_gemm_ws first; the
    configuration itself is checked against the device's kernels (GPU tests)."""
    assert lib.fp8bs_gemm_config(*args, None, 0, None) == expect


def test_probe_occupy_argument_checks(lib):
    assert lib.fp8bs_probe_occupy(0, 1000, None) == INVALID
    assert lib.fp8bs_probe_occupy(2000, 1000, None) == INVALID


def test_tensor_helpers_check_out_and_workspace_before_any_launch():
    """The binding's tensor helpers check a caller's `out` (contiguous bf16 of exactly the
    result's shape, on the GPU or in pinned host memory) and workspace (a uint8 CUDA tensor)
    before anything reaches the library, so that no kernel can write past their ends."""
    import torch
    from fp8_block_scaled_fp8bs_gb300 import _output, _workspace_args
    with pytest.raises(TypeError):          # pageable host memory is not reachable in place
        _output(torch.empty(3, 4, dtype=torch.bfloat16), (3, 4), "cpu")
    with pytest.raises(TypeError):
        _output(torch.empty(3, 4, dtype=torch.float32), (3, 4), "cpu")
    with pytest.raises(TypeError):
        _workspace_args(torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(TypeError):
        _workspace_args(bytearray(16))
    assert _workspace_args(None) == (0, 0)
