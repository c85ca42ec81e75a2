"""GPU parity of every launch configuration, selected explicitly through fp8bs_gemm_config:
each GEMM kernel at each of its tile widths, whole tiles, K split inside a cluster and
stream-K over a workspace, and the block-scaled kernel on CTA pairs ("DeepSeek-V3
Administrator & Developer Guide", §8.5.3: one sum over K blocks, however the tiles and the K
loop are cut). The shapes are ragged in M and N; every element is compared with the oracle, and
two calls in a row must agree bit for bit. Configurations the kernels do not support are
rejected before anything is launched.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import assert_gemm_close, dev_e4m3, dev_f32, host_bf16_f64

pytestmark = pytest.mark.gpu

S, P, B, PAIR = (fp8bs.KERNEL_SWAPPED, fp8bs.KERNEL_PROMOTED, fp8bs.KERNEL_BLOCK_SCALED,
                 fp8bs.KERNEL_BLOCK_SCALED_PAIR)
FP32, UE8M0 = fp8bs.SCALE_FP32, fp8bs.SCALE_UE8M0


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"


def inputs(M, N, K, fmt, seed):
    x = synth.activations(M, K, seed=seed, name="cfgA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x, oracle.SCALE_UE8M0 if fmt == UE8M0 else oracle.SCALE_FP32)
    b, b_s = synth.weights(N, K, seed=seed + 1, name="cfgB", pow2=fmt == UE8M0)
    return a, a_s, b, b_s


def run_config(a, a_s, b, b_s, fmt, kernel, tile, ksplit, ws=None):
    M, K = a.shape
    N = b.shape[0]
    A, AS, Bd, BS = dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s)
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8bs_gemm_config(A.data_ptr(), AS.data_ptr(), Bd.data_ptr(), BS.data_ptr(),
                            c.data_ptr(), M, N, K, fmt, 0, kernel, tile, ksplit,
                            ws.data_ptr() if ws is not None else 0,
                            ws.numel() if ws is not None else 0,
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return c


CONFIGS = [
    # kernel, tile, ksplit, scale format, M, N, K, workspace
    (S, 16, 1, FP32, 5, 1000, 1024, False),
    (S, 64, 3, FP32, 37, 1000, 1024, False),
    (S, 128, 8, FP32, 100, 300, 2048, False),
    (S, 32, 2, UE8M0, 20, 700, 1280, False),
    (P, 64, 1, FP32, 300, 1000, 1024, False),
    (P, 128, 1, FP32, 300, 1000, 1024, False),
    (P, 192, 1, FP32, 300, 1000, 1024, False),
    (P, 256, 1, FP32, 300, 1000, 1024, False),
    (P, 64, 3, FP32, 300, 1000, 1024, False),
    (P, 128, 2, FP32, 300, 1000, 1024, False),
    (P, 192, 4, FP32, 300, 1000, 1024, False),
    (P, 256, 8, FP32, 300, 1000, 1024, False),
    (P, 192, 0, FP32, 2560, 2304, 1024, True),      # stream-K: 180 tiles on the SMs
    (P, 128, 2, UE8M0, 300, 1000, 1024, False),     # power-of-two scales on the fp32 kernel
    (B, 64, 1, UE8M0, 300, 1000, 1024, False),
    (B, 128, 1, UE8M0, 300, 1000, 1024, False),
    (B, 192, 1, UE8M0, 300, 1000, 1024, False),
    (B, 256, 1, UE8M0, 300, 1000, 1024, False),
    (B, 64, 4, UE8M0, 300, 1000, 1024, False),
    (B, 128, 3, UE8M0, 300, 1000, 1024, False),
    (B, 192, 2, UE8M0, 300, 1000, 1024, False),
    (B, 256, 8, UE8M0, 300, 1000, 1024, False),
    (B, 128, 0, UE8M0, 1100, 2500, 2048, True),     # stream-K: 180 tiles, ragged both ways
    (B, 192, 1, UE8M0, 300, 1003, 1024, False),    # N % 8 != 0: element stores, two issuers
    (B, 192, 3, UE8M0, 300, 1003, 1024, False),
    (B, 256, 1, UE8M0, 300, 1003, 1024, False),
    (PAIR, 128, 1, UE8M0, 600, 1000, 640, False),   # the last pair's second CTA past M
    (PAIR, 192, 1, UE8M0, 600, 1000, 640, False),
    (PAIR, 256, 1, UE8M0, 600, 1000, 640, False),
    (PAIR, 256, 1, UE8M0, 2560, 4096, 256, False),  # more tiles than pairs: persistent
]


@pytest.mark.parametrize("kernel,tile,ksplit,fmt,M,N,K,with_ws", CONFIGS)
def test_every_configuration_against_oracle(kernel, tile, ksplit, fmt, M, N, K, with_ws):
    a, a_s, b, b_s = inputs(M, N, K, fmt, seed=M + N + K + tile + ksplit)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda") \
        if with_ws else None
    c1 = run_config(a, a_s, b, b_s, fmt, kernel, tile, ksplit, ws)
    c2 = run_config(a, a_s, b, b_s, fmt, kernel, tile, ksplit, ws)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16)), "two calls differ"
    assert_gemm_close(host_bf16_f64(c1), oracle.gemm(a, a_s, b, b_s),
                      f"kernel {kernel} tile {tile} ksplit {ksplit} {M}x{N}x{K}")


def random_codes(rng, rows, cols):
    c = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x00                        # no NaN codes
    return c


@pytest.mark.parametrize("kernel,tile", [(PAIR, 128), (PAIR, 192), (PAIR, 256), (B, 192),
                                         (B, 256)])
def test_block_scaled_per_row_and_block_exponents(kernel, tile):
    """Every row of A and every 128-row block of B carries its own exponent in every K block:
    on CTA pairs each CTA writes the scale factors of its own 128 rows of A and of all the
    tile's rows of B into its own TMEM, a wrong lane, column, chunk slot or CTA moves whole
    regions out of tolerance."""
    M, N, K = 600, 1000, 1280
    rng = np.random.default_rng(tile + kernel)
    a, b = random_codes(rng, M, K), random_codes(rng, N, K)
    m = np.arange(M)[:, None]
    kb = np.arange(K // 128)[None, :]
    a_s = np.ldexp(1.0, ((m * 7 + kb * 3) % 9) - 12).astype(np.float32)
    nb = np.arange(-(-N // 128))[:, None]
    b_s = np.ldexp(1.0, ((nb * 5 + kb * 2) % 7) - 11).astype(np.float32)
    c = run_config(a, a_s, b, b_s, UE8M0, kernel, tile, 1)
    assert_gemm_close(host_bf16_f64(c), oracle.gemm(a, a_s, b, b_s),
                      f"exponent pattern kernel {kernel} tile {tile}")


@pytest.mark.parametrize("kernel,tile,ksplit,fmt,M,with_ws", [
    (S, 16, 1, FP32, 17, False),        # more rows than the tile
    (S, 48, 1, FP32, 8, False),         # not a tile of this kernel
    (P, 96, 1, FP32, 300, False),
    (B, 128, 1, FP32, 300, False),      # block-scaled MMA needs power-of-two scales
    (PAIR, 256, 2, UE8M0, 600, False),  # pairs do not split K
    (PAIR, 64, 1, UE8M0, 600, False),
    (P, 128, 0, FP32, 2560, False),     # stream-K without a workspace
    (B, 256, 0, UE8M0, 2560, True),     # block-scaled stream-K only at 128 wide
    (P, 128, 0, FP32, 256, True),       # stream-K with fewer tiles than SMs
    (P, 128, 9, FP32, 300, False),      # more than a portable cluster
    (P, 128, 5, FP32, 300, False),      # more CTAs than K blocks (K = 512)
])
def test_unsupported_configurations_are_rejected(kernel, tile, ksplit, fmt, M, with_ws):
    N, K = 1000, 512
    A = torch.zeros((M, K), dtype=torch.float8_e4m3fn, device="cuda")
    AS = torch.ones((M, K // 128), dtype=torch.float32, device="cuda")
    Bd = torch.zeros((N, K), dtype=torch.float8_e4m3fn, device="cuda")
    BS = torch.ones((-(-N // 128), K // 128), dtype=torch.float32, device="cuda")
    c = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda") \
        if with_ws else None
    with pytest.raises(fp8bs.Fp8bsError) as err:
        fp8bs.fp8bs_gemm_config(A.data_ptr(), AS.data_ptr(), Bd.data_ptr(), BS.data_ptr(),
                                c.data_ptr(), M, N, K, fmt, 0, kernel, tile, ksplit,
                                ws.data_ptr() if ws is not None else 0,
                                ws.numel() if ws is not None else 0)
    assert err.value.status == 1
    torch.cuda.synchronize()
    assert bool((c == 7.0).all()), "a rejected configuration wrote the output"


def test_plans_are_valid_configurations():
    """Whatever fp8bs_gemm_plan reports for a shape, fp8bs_gemm_config accepts and computes."""
    for (M, N, K, fmt) in [(1, 2048, 7168, FP32), (300, 2048, 2048, FP32),
                           (2048, 576, 1024, UE8M0), (2048, 1536, 1024, UE8M0)]:
        p = fp8bs.fp8bs_gemm_plan(M, N, K, fmt, False)
        a, a_s, b, b_s = inputs(M, N, K, fmt, seed=M + N)
        c = run_config(a, a_s, b, b_s, fmt, p["kernel"], p["tile"], p["ksplit"])
        assert_gemm_close(host_bf16_f64(c), oracle.gemm(a, a_s, b, b_s), f"plan {p}")
