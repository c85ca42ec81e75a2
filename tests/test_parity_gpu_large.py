"""GPU parity at the largest index spaces: outputs (and for act_quant and weight_dequant, inputs)
with more than 2^31 elements, so that every offset past the 32-bit range is exercised in each
kernel's loads and stores. The device inputs are a seeded synthetic pattern of rows (synth, or
the oracle's act_quant of synth) tiled on the device; the sampled output rows or columns --
both sides of the 2^31-byte and 2^31-element boundaries, the last row and column, and random
ones -- are compared with the oracle applied to the pattern rows they were tiled from.
Bit-exact for act_quant and weight_dequant; the GEMM tolerance for fp8_gemm and the bf16 path.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import assert_gemm_close, host_bf16_bits, host_bf16_f64, host_codes

pytestmark = pytest.mark.gpu

FMTS = {"fp32": oracle.SCALE_FP32, "ue8m0": oracle.SCALE_UE8M0}
TWO31 = 2 ** 31


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"
    torch.cuda.empty_cache()


def tiled_u8(pattern: np.ndarray, rows: int) -> torch.Tensor:
    """The pattern's rows repeated down to `rows` rows, on the device (uint8)."""
    p = torch.from_numpy(np.ascontiguousarray(pattern)).cuda()
    reps = -(-rows // pattern.shape[0])
    return p.repeat(reps, 1)[:rows].contiguous()


def tiled_bf16(bits: np.ndarray, rows: int) -> torch.Tensor:
    p = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    reps = -(-rows // bits.shape[0])
    return p.repeat(reps, 1)[:rows].contiguous().view(torch.bfloat16)


def tiled_f32(a: np.ndarray, rows: int) -> torch.Tensor:
    p = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    reps = -(-rows // a.shape[0])
    return p.repeat(reps, 1)[:rows].contiguous()


def boundary_rows(M: int, row_elems: int, elem_bytes: int, seed: int, extra: int = 12):
    """Rows on both sides of the 2^31-byte and 2^31-element offsets of a [M, row_elems] output,
    the first and last rows, and random ones."""
    picks = {0, M - 1}
    for limit in (TWO31 // elem_bytes, TWO31):
        r = limit // row_elems
        picks.update(x for x in (r - 1, r, r + 1) if 0 <= x < M)
    picks.update(np.random.default_rng(seed).integers(0, M, extra).tolist())
    return np.array(sorted(picks), dtype=np.int64)


def take_rows(t: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    return t.index_select(0, torch.from_numpy(rows).cuda())


@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
def test_act_quant_beyond_2_31_elements(fmt):
    R, K = 64, 16384
    M = TWO31 // K + 64                      # 131136 rows, 2.149e9 elements
    assert M * K > TWO31 and M % R == 0
    pat = synth.activations(R, K, seed=31, name="huge/act", outlier_frac=0.01)
    x = tiled_bf16(pat, M)
    y, s = fp8bs.act_quant(x, fmt)
    del x
    rows = boundary_rows(M, K, 2, seed=1)
    y_s = host_codes(take_rows(y, rows))
    s_s = take_rows(s, rows).cpu().numpy()
    y_ref, s_ref = oracle.act_quant(pat, FMTS[fmt])
    for i, r in enumerate(rows):
        assert np.array_equal(s_s[i].view(np.uint32), s_ref[r % R].view(np.uint32)), \
            f"row {r}: scales differ"
        assert np.array_equal(y_s[i], y_ref[r % R]), f"row {r}: codes differ"


def test_weight_dequant_beyond_2_31_elements():
    K = 16384
    N = TWO31 // K + 64                      # 131136 rows: the last 128-row block is half full
    pat = synth.weights(128, K, seed=32, name="huge/dq")[0]
    s = synth.weight_scales(N, K, seed=32, name="huge/dq")   # a distinct scale per block
    w = tiled_u8(pat, N).view(torch.float8_e4m3fn)
    y = fp8bs.weight_dequant(w, torch.from_numpy(s).cuda())
    del w
    rows = boundary_rows(N, K, 2, seed=2)
    got = host_bf16_bits(take_rows(y, rows))
    for i, r in enumerate(rows):
        ref = oracle.weight_dequant(pat[r % 128:r % 128 + 1], s[r // 128:r // 128 + 1])
        assert np.array_equal(got[i], ref[0]), f"row {r}"


@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
def test_gemm_many_rows_beyond_2_31_outputs(fmt):
    """The normal-orientation kernels (fp32-scale promotion; ue8m0 block-scaled MMA): C has
    65600 x 33000 > 2^31 elements, ragged in both M and N."""
    R, K = 64, 256
    M, N = 64 * 1025, 33000
    assert M * N > TWO31
    a_pat, as_pat = oracle.act_quant(synth.activations(R, K, seed=33, name="huge/A"), FMTS[fmt])
    b, b_s = synth.weights(N, K, seed=33, name="huge/B", pow2=fmt == "ue8m0")
    c = fp8bs.fp8_gemm(tiled_u8(a_pat, M).view(torch.float8_e4m3fn), tiled_f32(as_pat, M),
                       torch.from_numpy(b).cuda().view(torch.float8_e4m3fn),
                       torch.from_numpy(b_s).cuda(), fmt)
    rows = boundary_rows(M, N, 2, seed=3)
    got = host_bf16_f64(take_rows(c, rows))
    ref = oracle.gemm(a_pat[rows % R], as_pat[rows % R], b, b_s)
    assert_gemm_close(got, ref, f"{M}x{N}x{K} {fmt}")


def huge_n_columns(M: int, N: int, seed: int):
    """Columns of a [M, N] output on both sides of the 2^31-element offset in its last row, the
    edges of the first and last 128-row weight blocks, and random ones."""
    edge = TWO31 - (M - 1) * N
    picks = {0, 127, 128, N - 2, N - 1, edge - 1, edge}
    picks.update(np.random.default_rng(seed).integers(0, N, 48).tolist())
    return np.array(sorted(picks), dtype=np.int64)


@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
def test_gemm_decode_orientation_beyond_2_31_outputs(fmt):
    """The swapped-orientation kernel (M <= 128 rows): 128 x 16777400 outputs, N ragged."""
    M, K = 128, 256
    N = 16777400
    assert M * N > TWO31 and 0 < TWO31 - (M - 1) * N < N
    a, a_s = oracle.act_quant(synth.activations(M, K, seed=34, name="huge/x"), FMTS[fmt])
    bpat = synth.weights(128, K, seed=34, name="huge/Bp")[0]
    b_s = synth.weight_scales(N, K, seed=34, name="huge/Bp", pow2=fmt == "ue8m0")
    c = fp8bs.fp8_gemm(torch.from_numpy(a).cuda().view(torch.float8_e4m3fn),
                       torch.from_numpy(a_s).cuda(),
                       tiled_u8(bpat, N).view(torch.float8_e4m3fn), torch.from_numpy(b_s).cuda(),
                       fmt)
    cols = huge_n_columns(M, N, seed=4)
    got = host_bf16_f64(c.index_select(1, torch.from_numpy(cols).cuda()))
    ref = np.concatenate([oracle.gemm(a, a_s, bpat[n % 128:n % 128 + 1], b_s[n // 128:n // 128 + 1])
                          for n in cols], axis=1)
    assert_gemm_close(got, ref, f"{M}x{N}x{K} {fmt}")


def test_linear_bf16_beyond_2_31_outputs():
    """The bf16 path, one 128-row tile of x per CTA: 128 x 16777400 outputs."""
    M, K = 128, 256
    N = 16777400
    x = synth.activations(M, K, seed=35, name="huge/lx")
    wpat = synth.weights(128, K, seed=35, name="huge/W")[0]
    w_s = synth.weight_scales(N, K, seed=35, name="huge/W")
    y = fp8bs.linear_bf16(torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16),
                          tiled_u8(wpat, N).view(torch.float8_e4m3fn), torch.from_numpy(w_s).cuda())
    cols = huge_n_columns(M, N, seed=5)
    got = host_bf16_f64(y.index_select(1, torch.from_numpy(cols).cuda()))
    ref = np.concatenate([oracle.linear_bf16(x, wpat[n % 128:n % 128 + 1],
                                             w_s[n // 128:n // 128 + 1]) for n in cols], axis=1)
    assert_gemm_close(got, ref, f"bf16 path {M}x{N}x{K}")


def test_linear_bf16_many_rows_beyond_2_31_outputs():
    """The bf16 path, two 128-row tiles of x per CTA: 65600 x 33000 outputs."""
    R, K = 64, 256
    M, N = 64 * 1025, 33000
    xpat = synth.activations(R, K, seed=36, name="huge/lxm")
    w, w_s = synth.weights(N, K, seed=36, name="huge/Wm")
    y = fp8bs.linear_bf16(tiled_bf16(xpat, M), torch.from_numpy(w).cuda().view(torch.float8_e4m3fn),
                          torch.from_numpy(w_s).cuda())
    rows = boundary_rows(M, N, 2, seed=6)
    got = host_bf16_f64(take_rows(y, rows))
    ref = oracle.linear_bf16(xpat[rows % R], w, w_s)
    assert_gemm_close(got, ref, f"bf16 path {M}x{N}x{K}")
