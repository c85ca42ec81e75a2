"""GPU parity of the split-K schedule: the K loop of each output tile (or 128-row weight slab)
shared by the CTAs of one thread-block cluster, whose fp32 partials are added in rank order
through distributed shared memory ("DeepSeek-V3 Administrator & Developer Guide", §8.5.3: the
sum over K blocks, here cut into consecutive ranges; the Note there says M is not an autotune
key, and decode-sized M leaves the weight slabs too few to fill the SMs).

Every case checks first, through fp8bs_gemm_plan, that the call really takes the schedule it is
meant to test, then compares the output with the oracle: every element where the oracle
finishes in seconds, else whole rows and whole columns (every lane and every column of every
tile they cross) plus samples in every tile. Two calls in a row must agree bit for bit.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import assert_gemm_close, dev_e4m3, dev_f32, host_bf16_f64, lines_and_tiles

pytestmark = pytest.mark.gpu

FMTS = {"fp32": oracle.SCALE_FP32, "ue8m0": oracle.SCALE_UE8M0}
KERNEL = {"swapped": fp8bs.KERNEL_SWAPPED, "promoted": fp8bs.KERNEL_PROMOTED,
          "block_scaled": fp8bs.KERNEL_BLOCK_SCALED}


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"


def case(M, N, K, fmt, seed):
    x = synth.activations(M, K, seed=seed, name="splitA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x, FMTS[fmt])
    b, b_s = synth.weights(N, K, seed=seed + 1, name="splitB", pow2=fmt == "ue8m0")
    return a, a_s, b, b_s


def run(a, a_s, b, b_s, fmt, workspace=None):
    c = fp8bs.fp8_gemm(dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s), fmt,
                       workspace=workspace)
    torch.cuda.synchronize()
    return c


def check_plan(M, N, K, fmt, kernel, tile=None, min_split=2):
    p = fp8bs.fp8bs_gemm_plan(M, N, K, fp8bs._fmt(fmt), with_workspace=False)
    assert p["kernel"] == KERNEL[kernel], p
    if tile is not None:
        assert p["tile"] == tile, p
    assert p["ksplit"] >= min_split, p
    return p


# ------------------------------------------------------------------ decode orientation (M <= 128)

@pytest.mark.parametrize("N", [576, 1536, 2048, 7168])
@pytest.mark.parametrize("M", [1, 8, 32, 64, 128])
def test_decode_split_k_full_compare(M, N):
    """Decode-sized M with few weight slabs (the kv latent, q down-projection, one expert's
    up-projection, the down-projection's output width) at the model's K = 7168: every output
    against the oracle, and a second call bit-identical."""
    K = synth.DIM
    check_plan(M, N, K, "fp32", "swapped")
    a, a_s, b, b_s = case(M, N, K, "fp32", seed=M * 7 + N)
    c1, c2 = run(a, a_s, b, b_s, "fp32"), run(a, a_s, b, b_s, "fp32")
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert_gemm_close(host_bf16_f64(c1), oracle.gemm(a, a_s, b, b_s), f"decode split {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 8, 32, 64, 128])
def test_decode_split_k_down_projection_long_k(M):
    """N = 7168 with K = 18432 (the MLP down-projection at decode): 144 K blocks per slab."""
    N, K = synth.DIM, synth.INTER
    check_plan(M, N, K, "fp32", "swapped")
    a, a_s, b, b_s = case(M, N, K, "fp32", seed=M + 3)
    assert_gemm_close(host_bf16_f64(run(a, a_s, b, b_s, "fp32")), oracle.gemm(a, a_s, b, b_s),
                      f"decode split {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (3, 200, 1024),       # one slab, ragged rows and columns
    (50, 1000, 2048),     # eight slabs, the last one 104 rows
    (100, 333, 4096),     # odd N: element stores
    (17, 2048, 1152),     # nine K blocks: ranges of four and five
])
def test_decode_split_k_ragged(M, N, K):
    check_plan(M, N, K, "fp32", "swapped")
    a, a_s, b, b_s = case(M, N, K, "fp32", seed=M + N + K)
    assert_gemm_close(host_bf16_f64(run(a, a_s, b, b_s, "fp32")), oracle.gemm(a, a_s, b, b_s),
                      f"decode split {M}x{N}x{K}")


def test_decode_split_k_ue8m0_scales():
    M, N, K = 64, 576, 7168
    check_plan(M, N, K, "ue8m0", "swapped")
    a, a_s, b, b_s = case(M, N, K, "ue8m0", seed=5)
    assert_gemm_close(host_bf16_f64(run(a, a_s, b, b_s, "ue8m0")), oracle.gemm(a, a_s, b, b_s),
                      "decode split ue8m0")


def test_decode_without_split_unchanged_at_full_width():
    """N = 18432 fills the SMs with slabs: no split."""
    p = fp8bs.fp8bs_gemm_plan(64, synth.INTER, synth.DIM, fp8bs.SCALE_FP32, True)
    assert p["kernel"] == fp8bs.KERNEL_SWAPPED and p["ksplit"] == 1, p


# ------------------------------------------------------------------ normal orientation (M > 128)

@pytest.mark.parametrize("M,N,K", [
    (300, 2048, 7168),     # one MoE expert's rows: 24 tiles 256 wide on 152 SMs
    (129, 2048, 4096),     # two row tiles, the second one row high
    (257, 1000, 4096),     # ragged columns, three row tiles
    (200, 97, 4096),       # one tile narrower than the narrowest width
    (300, 1536, 4096),
])
def test_fp32_split_k_full_compare(M, N, K):
    check_plan(M, N, K, "fp32", "promoted")
    a, a_s, b, b_s = case(M, N, K, "fp32", seed=M + N)
    c1, c2 = run(a, a_s, b, b_s, "fp32"), run(a, a_s, b, b_s, "fp32")
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert_gemm_close(host_bf16_f64(c1), oracle.gemm(a, a_s, b, b_s), f"fp32 split {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (512, 576, 7168),      # twelve 192-wide tiles, eight CTAs each
    (300, 576, 2048),
    (129, 1000, 4096),
    (1000, 64, 4096),      # eight 64-wide tiles (two MMA issuers per CTA)
])
def test_ue8m0_split_k_full_compare(M, N, K):
    check_plan(M, N, K, "ue8m0", "block_scaled")
    a, a_s, b, b_s = case(M, N, K, "ue8m0", seed=M + N + 1)
    c1, c2 = run(a, a_s, b, b_s, "ue8m0"), run(a, a_s, b, b_s, "ue8m0")
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert_gemm_close(host_bf16_f64(c1), oracle.gemm(a, a_s, b, b_s), f"ue8m0 split {M}x{N}x{K}")


def test_mla_projection_plans():
    """The ue8m0 MLA projections (M=2048, K=7168) fill the SMs with whole tiles, with or without
    a workspace: the kv projection (N=576) as 144 tiles 64 wide, the q projection (N=1536) as
    128 tiles 192 wide (1536 = 8 x 192)."""
    for ws in (False, True):
        for N, tile in ((576, 64), (1536, 192)):
            p = fp8bs.fp8bs_gemm_plan(2048, N, synth.DIM, fp8bs.SCALE_UE8M0, ws)
            assert p == {"kernel": fp8bs.KERNEL_BLOCK_SCALED, "tile": tile, "ksplit": 1,
                         "stream_k": False}, (N, ws, p)


def random_codes(rng, rows, cols):
    c = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x00                        # no NaN codes
    return c


@pytest.mark.parametrize("M,N,K,split", [
    (512, 576, 7168, True),      # 192-wide tiles at n0 = 0, 192, 384, split K
    (2048, 1536, 640, False),    # 192-wide whole tiles at every n0 up to 1344
    (2560, 1152, 768, False),
])
def test_ue8m0_192_wide_tiles_per_row_and_block_exponents(M, N, K, split):
    """Every row of A and every 128-row block of B carries its own exponent in every K block. A
    192-wide tile at an odd multiple of 64 meets its second block of B at tile row 64, at an
    even one at row 128: a scale factor taken from the wrong block, row or K block moves whole
    regions out of tolerance."""
    p = fp8bs.fp8bs_gemm_plan(M, N, K, fp8bs.SCALE_UE8M0, False)
    assert p["kernel"] == fp8bs.KERNEL_BLOCK_SCALED and p["tile"] == 192, p
    assert (p["ksplit"] > 1) == split, p
    rng = np.random.default_rng(13)
    a, b = random_codes(rng, M, K), random_codes(rng, N, K)
    m = np.arange(M)[:, None]
    kb = np.arange(K // 128)[None, :]
    a_s = np.ldexp(1.0, ((m * 7 + kb * 3) % 9) - 4 - 8).astype(np.float32)
    nb = np.arange(-(-N // 128))[:, None]
    b_s = np.ldexp(1.0, ((nb * 5 + kb * 2) % 7) - 3 - 8).astype(np.float32)
    c = host_bf16_f64(run(a, a_s, b, b_s, "ue8m0"))
    assert_gemm_close(c, oracle.gemm(a, a_s, b, b_s), f"ue8m0 192-wide exponents {M}x{N}x{K}")


@pytest.mark.parametrize("N", [synth.Q_LORA, synth.KV_LORA_ROPE])
def test_mla_full_size_rows_and_columns(N):
    """The MLA projections at full size (M=2048, K=7168, ue8m0) in the benchmark's call (with a
    workspace): whole rows, whole columns and samples in every tile against the oracle."""
    M, K = 2048, synth.DIM
    x = synth.mla_acts()
    a, a_s = oracle.act_quant(x, oracle.SCALE_UE8M0)
    b, b_s = synth.weights(N, K, seed=0, name=f"mla/B{N}", pow2=True)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    c_dev = run(a, a_s, b, b_s, "ue8m0", workspace=ws)
    c = host_bf16_f64(c_dev)
    mi, ni = lines_and_tiles(M, N, 2, seed=N)
    assert_gemm_close(c[mi, ni], oracle.gemm_at(a, a_s, b, b_s, mi, ni), f"MLA N={N}",
                      c_full=c_dev)
