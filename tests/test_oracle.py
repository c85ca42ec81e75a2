"""Pins for the CPU oracle: each check ties the oracle to something other than itself --
hand-derived worked cases (tests/golden), PyTorch's own fp8/bf16 casts and IEEE binary32
arithmetic (library routines), numpy's binary64 matmul of the dequantised operands, closed
forms, invariants, and exhaustive enumeration of the 256 e4m3fn codes.

The method: "DeepSeek-V3 Administrator & Developer Guide" §8.5.1 act_quant_kernel,
§8.5.2 weight_dequant_kernel, §8.5.3 fp8_gemm_kernel, §6.3 The FP8 path.
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32_bits(f):
    return struct.unpack("<I", struct.pack("<f", float(np.float32(f))))[0]


def torch_decode(codes: np.ndarray) -> np.ndarray:
    """e4m3fn codes -> float64 via PyTorch's float8_e4m3fn type (an independent decoder)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_e4m3(v: np.ndarray) -> np.ndarray:
    """float32 (|v| <= 448) -> e4m3fn codes via PyTorch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# ------------------------------------------------------------------ e4m3fn codec

def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = np.array([oracle.e4m3_decode(c) for c in codes])
    ref = torch_decode(codes)
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.all(np.isnan(ours[nan]))
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero of 0x80
    assert math.copysign(1.0, ours[0x80]) == -1.0
    assert oracle.e4m3_decode(0x7E) == 448.0


def test_encode_roundtrips_every_finite_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            assert oracle.e4m3_encode(float("nan")) == 0x7F
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_encode_midpoints_tie_to_even_and_neighbours_go_nearer():
    vals = sorted({oracle.e4m3_decode(c) for c in range(0x7F)})
    assert len(vals) == 127
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # midpoints are exact in binary32
        c_lo, c_hi = oracle.e4m3_encode(lo), oracle.e4m3_encode(hi)
        even = c_lo if c_lo % 2 == 0 else c_hi
        assert oracle.e4m3_encode(mid) == even
        assert oracle.e4m3_encode(-mid) == even | 0x80
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        assert oracle.e4m3_encode(below) == c_lo
        assert oracle.e4m3_encode(above) == c_hi


def test_encode_worked_values_from_golden():
    path = os.path.join(GOLDEN, "e4m3_encode_worked.txt")
    n = 0
    with open(path) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            val, code = line.split()[:2]
            assert oracle.e4m3_encode(float(val)) == int(code, 16), line
            n += 1
    assert n >= 20


def test_encode_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(1234)
    mag = np.exp2(rng.uniform(-14, np.log2(448.0), 20000)).astype(np.float32)
    v = (mag * rng.choice([-1, 1], mag.size)).astype(np.float32)
    v = np.clip(v, -448, 448)
    ours = oracle.e4m3_encode_array(v)
    assert np.array_equal(ours, torch_e4m3(v))


# ------------------------------------------------------------------ bf16 helpers

def test_bf16_rne_matches_torch_including_ties():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * np.exp2(rng.uniform(-30, 30, 20000))).astype(np.float32)
    # exact ties: a bf16 value plus half its ulp
    base = synth.to_bf16_bits(v[:2000])
    bf = synth.bf16_bits_to_f32(base)
    ulp_half = np.abs(bf) * np.float32(2.0 ** -8)
    tie = np.float32(bf + np.sign(bf) * np.exp2(np.floor(np.log2(ulp_half))))
    v = np.concatenate([v, tie.astype(np.float32)])
    ours = np.array([oracle.bf16_rne(x) for x in v], dtype=np.uint16)
    assert np.array_equal(ours, synth.to_bf16_bits(v))
    h = synth.to_bf16_bits(v[:100])
    assert all(oracle.bf16_to_float(int(x)) == float(y)
               for x, y in zip(h, synth.bf16_bits_to_f32(h)))


def test_f32_div_is_ieee_binary32():
    rng = np.random.default_rng(3)
    a = (rng.standard_normal(5000) * 100).astype(np.float32)
    b = np.exp2(rng.uniform(-20, 5, 5000)).astype(np.float32)
    ref = (torch.from_numpy(a) / torch.from_numpy(b)).numpy()
    ours = np.array([oracle.f32_div(x, y) for x, y in zip(a, b)], dtype=np.float32)
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ act_quant

def _golden_act_cases():
    path = os.path.join(GOLDEN, "act_quant_worked.txt")
    with open(path) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            name, fmt, lead, fill, s_hex, codes, fill_code = [f.strip() for f in line.split("|")]
            yield name, fmt, [float(t) for t in lead.split()], float(fill), int(s_hex, 16), \
                [int(c, 16) for c in codes.split()], int(fill_code, 16)


@pytest.mark.parametrize("case", list(_golden_act_cases()), ids=lambda c: f"{c[0]}-{c[1]}")
def test_act_quant_worked_cases(case):
    name, fmt, lead, fill, s_bits, codes, fill_code = case
    x = np.full(128, fill, dtype=np.float32)
    x[: len(lead)] = lead
    xb = synth.to_bf16_bits(x)[None, :]
    assert np.array_equal(synth.bf16_bits_to_f32(xb)[0], x), "worked inputs must be exact in bf16"
    y, s = oracle.act_quant(xb, oracle.SCALE_UE8M0 if fmt == "ue8m0" else oracle.SCALE_FP32)
    assert f32_bits(s[0, 0]) == s_bits
    assert list(y[0, : len(codes)]) == codes
    assert np.all(y[0, len(codes):] == fill_code)


def _torch_act_quant_fp32(xbits: np.ndarray):
    """The same steps with PyTorch binary32 ops and PyTorch's fp8 cast (independent code)."""
    x = torch.from_numpy(synth.bf16_bits_to_f32(xbits)).view(xbits.shape[0], -1, 128)
    amax = x.abs().amax(dim=-1, keepdim=True)
    s = torch.clamp(amax, min=1e-4) / 448.0
    y = (x / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return y.view(torch.uint8).reshape(xbits.shape).numpy(), s.squeeze(-1).numpy()


def test_act_quant_matches_torch_binary32_pipeline():
    x = synth.activations(37, 1024, seed=5, name="pin", outlier_frac=0.01)
    x[3, :128] = 0  # a zero block exercises the 1e-4 clamp
    x[4, 128:256] = synth.to_bf16_bits(np.full(128, 2.0 ** -16, np.float32))
    y, s = oracle.act_quant(x)
    yt, st = _torch_act_quant_fp32(x)
    assert np.array_equal(s.view(np.uint32), st.view(np.uint32))
    assert np.array_equal(y, yt)


@pytest.mark.parametrize("fmt", [oracle.SCALE_FP32, oracle.SCALE_UE8M0])
def test_act_quant_invariants(fmt):
    x = synth.activations(64, 2048, seed=11, name="inv", outlier_frac=0.01)
    x[0, :128] = 0
    y, s = oracle.act_quant(x, fmt)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(64, -1, 128)
    amax = np.abs(xf).max(-1)
    clamp = np.maximum(amax, np.float64(np.float32(1e-4)))
    s64 = s.astype(np.float64)
    if fmt == oracle.SCALE_UE8M0:
        mant, _ = np.frexp(s64)
        assert np.all(mant == 0.5), "ue8m0 scales are exact powers of two"
        assert np.all(s64 >= clamp / 448) and np.all(clamp / 448 > s64 / 2)
    else:
        assert np.all(np.abs(s64 - clamp / 448) <= s64 * 2.0 ** -24)
    dec = torch_decode(y).reshape(64, -1, 128)
    assert np.all(np.abs(dec) <= 448)
    q = xf / s64[..., None]
    mag = np.maximum(np.minimum(np.abs(q), np.abs(dec)), 2.0 ** -6)
    half_ulp = np.exp2(np.floor(np.log2(mag)) - 3) / 2
    bound = (half_ulp + 2.0 ** -23 * np.abs(q)) * s64[..., None]
    assert np.all(np.abs(dec * s64[..., None] - xf) <= bound)
    if fmt == oracle.SCALE_FP32:
        big = amax >= 1e-4
        idx = np.abs(xf).argmax(-1)
        codes = np.take_along_axis(y.reshape(64, -1, 128), idx[..., None], -1)[..., 0]
        assert np.all((codes[big] & 0x7F) == 0x7E)


# ------------------------------------------------------------------ weight_dequant

def test_weight_dequant_pow2_scales_are_exact():
    b, s = synth.weights(300, 260, seed=2, name="pin", pow2=True)
    y = oracle.weight_dequant(b, s)
    full = np.repeat(np.repeat(s, 128, 0)[:300], 128, 1)[:, :260].astype(np.float64)
    exact = torch_decode(b) * full
    assert np.array_equal(synth.bf16_bits_to_f32(y).astype(np.float64), exact)


def test_weight_dequant_matches_torch_binary32_then_bf16():
    b, s = synth.weights(333, 391, seed=4, name="pin")
    y = oracle.weight_dequant(b, s)
    wt = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float32)
    st = torch.from_numpy(s).repeat_interleave(128, 0)[:333].repeat_interleave(128, 1)[:, :391]
    ref = (wt * st).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, ref)


# ------------------------------------------------------------------ fp8_gemm

def _dequant64(codes, scales, rows_per_scale):
    full = np.repeat(np.repeat(scales, rows_per_scale, 0)[: codes.shape[0]], 128, 1)
    return torch_decode(codes) * full[:, : codes.shape[1]].astype(np.float64)


def test_gemm_matches_numpy_matmul_of_dequantised_operands():
    x = synth.activations(45, 640, seed=9, name="pinA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(200, 640, seed=9, name="pinB")
    c = oracle.gemm(a, a_s, b, b_s)
    ref = _dequant64(a, a_s, 1) @ _dequant64(b, b_s, 128).T
    assert np.max(np.abs(c - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gemm_matches_a_naive_triple_loop_on_a_tiny_ragged_shape():
    """The block-scaled sum of "DeepSeek-V3 Administrator & Developer Guide" §8.5.3 written out
    as plain nested Python loops over m, n, K blocks and k, in binary64, from torch's decoding of
    the codes: N = 130 spans two 128-row weight-scale blocks and K = 256 two K blocks, so a
    wrong scale index, a dropped block or a transposed operand shows."""
    x = synth.activations(3, 256, seed=12, name="loopA", outlier_frac=0.05)
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(130, 256, seed=12, name="loopB")
    av, bv = torch_decode(a), torch_decode(b)
    c = oracle.gemm(a, a_s, b, b_s)
    for m in range(3):
        for n in range(130):
            total, size = 0.0, 0.0
            for kb in range(2):
                part, part_abs = 0.0, 0.0
                for k in range(128 * kb, 128 * kb + 128):
                    p = float(av[m, k]) * float(bv[n, k])
                    part += p
                    part_abs += abs(p)
                scale = float(a_s[m, kb]) * float(b_s[n // 128, kb])
                total += scale * part
                size += scale * part_abs
            assert abs(c[m, n] - total) <= 1e-14 * size, (m, n)


def test_gemm_closed_forms():
    K = 512
    ones_a = np.full((3, K), 0x38, np.uint8)  # 1.0
    ones_b = np.full((256, K), 0x38, np.uint8)
    c = oracle.gemm(ones_a, np.ones((3, 4), np.float32), ones_b, np.ones((2, 4), np.float32))
    assert np.all(c == K)
    # per-K-block scales 2^kb on A and 2^(3*kb + nb) on B: C = 128 * sum_kb 2^(4kb + nb)
    a_s = np.exp2(np.arange(4, dtype=np.float32))[None, :].repeat(3, 0)
    b_s = np.exp2(3 * np.arange(4, dtype=np.float32)[None, :] + np.arange(2)[:, None]).astype(np.float32)
    c = oracle.gemm(ones_a, a_s, ones_b, b_s)
    for nb in range(2):
        expect = 128 * sum(2.0 ** (4 * kb + nb) for kb in range(4))
        assert np.all(c[:, nb * 128:(nb + 1) * 128] == expect)


def test_gemm_identity_selects_dequantised_rows():
    b, b_s = synth.weights(128, 128, seed=6, name="pinI")
    eye = np.where(np.eye(128, dtype=bool), np.uint8(0x38), np.uint8(0))
    c = oracle.gemm(eye, np.ones((128, 1), np.float32), b, b_s)
    assert np.array_equal(c, (torch_decode(b) * float(b_s[0, 0])).T)


def test_gemm_ragged_n_tail_block_uses_its_own_scale():
    x = synth.activations(5, 256, seed=1, name="tailA")
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(576, 256, seed=1, name="tailB")
    assert b_s.shape == (5, 2)
    c = oracle.gemm(a, a_s, b, b_s)
    ref = _dequant64(a, a_s, 1) @ _dequant64(b, b_s, 128).T
    assert np.max(np.abs(c - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gemm_at_agrees_with_full_gemm():
    x = synth.activations(20, 384, seed=8, name="atA")
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(130, 384, seed=8, name="atB")
    c = oracle.gemm(a, a_s, b, b_s)
    mi = np.array([0, 19, 7, 13], np.int64)
    ni = np.array([0, 129, 128, 64], np.int64)
    assert np.array_equal(oracle.gemm_at(a, a_s, b, b_s, mi, ni), c[mi, ni])


# ------------------------------------------------------------------------------ bf16 path

def test_linear_bf16_identity_rows_select_dequantised_weights():
    """x = rows of the identity: y[i, n] = W'[n, i], the bf16 weight_dequant output (pins the
    transposition, the scale indexing and the dequantisation in one go)."""
    K, N = 256, 300
    w, w_s = synth.weights(N, K, seed=31, name="linpin")
    eye = np.zeros((K, K), dtype=np.float32)
    np.fill_diagonal(eye, 1.0)
    x = synth.to_bf16_bits(eye)
    y = oracle.linear_bf16(x, w, w_s)
    wd = oracle.bf16_bits_to_f64(oracle.weight_dequant(w, w_s))
    assert np.array_equal(y, wd.T)


def test_linear_bf16_matches_block_scaled_gemm_when_both_are_exact():
    """With power-of-two weight scales the bf16 weight is exact (code x 2^e fits bf16), and x
    chosen on the e4m3 grid equals its own act_quant codes at scale 1: then the bf16 path and
    the block-scaled GEMM compute the same sum."""
    M, N, K = 7, 260, 384
    rng = np.random.default_rng(32)
    codes = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0
    xv = np.array([oracle.e4m3_decode(int(c)) for c in codes.ravel()]).reshape(M, K)
    x = synth.to_bf16_bits(xv.astype(np.float32))            # e4m3 values are exact in bf16
    w, w_s = synth.weights(N, K, seed=33, name="linpin", pow2=True)
    a_s = np.ones((M, K // 128), dtype=np.float32)
    np.testing.assert_allclose(oracle.linear_bf16(x, w, w_s), oracle.gemm(codes, a_s, w, w_s),
                               rtol=1e-13, atol=0)


def test_linear_bf16_single_block_closed_form():
    """All-ones x against a weight of code 0x38 (1.0) with scale 2^-3: y = K / 8 exactly."""
    M, N, K = 3, 128, 512
    x = synth.to_bf16_bits(np.ones((M, K), dtype=np.float32))
    w = np.full((N, K), 0x38, dtype=np.uint8)
    w_s = np.full((1, K // 128), 0.125, dtype=np.float32)
    assert np.all(oracle.linear_bf16(x, w, w_s) == K / 8)
