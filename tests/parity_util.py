"""Shared helpers for the GPU parity tests: moving synth/oracle arrays to and from the device
and the GEMM tolerance. The tolerance is the one the path's accuracy contract states:
    |C_gpu - C_ref| <= 2^-7 |C_ref| + 1e-3 rms(C_ref)   (elementwise)
where C_ref is the oracle's binary64 result. It covers the tensor cores' fp32 accumulation of
each 128-long block, the fp32 scale promotion and the final rounding to bf16 (2^-9 relative)."""
from __future__ import annotations

import numpy as np
import torch

REL_TOL = 2.0 ** -7
RMS_TOL = 1e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).cuda()


def dev_e4m3(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_codes(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rms_of(c) -> float:
    """Root mean square of a whole matrix (numpy array or CUDA tensor), in binary64."""
    if isinstance(c, torch.Tensor):
        c = c.double()
        return float(torch.sqrt(torch.mean(c * c)).item()) if c.numel() else 0.0
    c = np.asarray(c, dtype=np.float64)
    return float(np.sqrt(np.mean(c ** 2))) if c.size else 0.0


def gemm_violations(c_gpu: np.ndarray, c_ref: np.ndarray, rms: float | None = None,
                    c_full=None):
    """Elementwise tolerance check; returns (number of violations, worst ratio err/bound).

    The bound's rms term is rms(C_ref) over the whole matrix. When only sampled positions of
    C_ref exist, the whole GPU output `c_full` is passed as well and the smaller of rms(sampled
    C_ref) and rms(whole C_gpu) is used: the bound is then no looser than either estimate of the
    whole matrix's rms."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    c_ref = np.asarray(c_ref, dtype=np.float64)
    if rms is None:
        rms = rms_of(c_ref)
        if c_full is not None:
            rms = min(rms, rms_of(c_full))
    bound = REL_TOL * np.abs(c_ref) + RMS_TOL * rms
    err = np.abs(c_gpu - c_ref)
    bad = ~(err <= bound)  # NaN counts as a violation
    ratio = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    return int(bad.sum()), ratio


def assert_gemm_close(c_gpu, c_ref, what="", rms=None, c_full=None):
    n, worst = gemm_violations(c_gpu, c_ref, rms, c_full)
    assert n == 0, f"{what}: {n} elements outside tolerance (worst err/bound {worst:.3g})"
    return worst


def tile_samples(M: int, N: int, per_tile: int, seed: int, bm: int = 128, bn: int = 128):
    """Positions (mi, ni) with `per_tile` random samples inside every bm x bn output tile, plus
    the four corners of the matrix, so that every tile of any tiling down to bm x bn is hit."""
    rng = np.random.default_rng(seed)
    mt, nt = -(-M // bm), -(-N // bn)
    tm = np.repeat(np.arange(mt), nt * per_tile)
    tn = np.tile(np.repeat(np.arange(nt), per_tile), mt)
    mi = tm * bm + rng.integers(0, bm, tm.size)
    ni = tn * bn + rng.integers(0, bn, tn.size)
    keep = (mi < M) & (ni < N)
    mi = np.concatenate([mi[keep], [0, 0, M - 1, M - 1]]).astype(np.int64)
    ni = np.concatenate([ni[keep], [0, N - 1, 0, N - 1]]).astype(np.int64)
    return mi, ni


def lines_and_tiles(M: int, N: int, per_tile: int, seed: int, n_rows: int = 2, n_cols: int = 2):
    """tile_samples plus whole rows (the first, the last and n_rows random ones) and whole
    columns (likewise): every column of every tile a whole row crosses and every row (TMEM lane)
    of every tile a whole column crosses is compared, so that a wrong lane or column inside a
    tile cannot hide between the samples."""
    rng = np.random.default_rng(seed + 1)
    rows = np.unique(np.r_[0, M - 1, rng.integers(0, M, n_rows)])
    cols = np.unique(np.r_[0, N - 1, rng.integers(0, N, n_cols)])
    tm, tn = tile_samples(M, N, per_tile, seed)
    mi = np.concatenate([np.repeat(rows, N), np.repeat(np.arange(M), len(cols)), tm])
    ni = np.concatenate([np.tile(np.arange(N), len(rows)), np.tile(cols, M), tn])
    return mi.astype(np.int64), ni.astype(np.int64)
