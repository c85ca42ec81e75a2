"""GPU parity: the CUDA library (called through its C ABI) against the CPU oracle on seeded
synthetic inputs. act_quant codes and scales and weight_dequant outputs must be bit-exact;
fp8_gemm must lie within |C - C_ref| <= 2^-7 |C_ref| + 1e-3 rms(C_ref).

Small shapes compare every element and span several tiles with ragged tails; the full-size
workloads (decode, prefill, MoE experts, ue8m0 MLA projections) run the kernels in the same
launch configuration as the benchmark and compare sampled rows/positions, with every output
tile sampled. Oracle inputs always come from synth or the oracle itself, never from the GPU.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import (assert_gemm_close, dev_bf16, dev_e4m3, dev_f32, host_bf16_bits,
                         host_bf16_f64, host_codes, lines_and_tiles)

pytestmark = pytest.mark.gpu

FMTS = {"fp32": oracle.SCALE_FP32, "ue8m0": oracle.SCALE_UE8M0}


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"


def gpu_act_quant(x_bits, fmt):
    y, s = fp8bs.act_quant(dev_bf16(x_bits), fmt)
    torch.cuda.synchronize()
    return host_codes(y), s.cpu().numpy()


def assert_quant_equal(y, s, y_ref, s_ref, what):
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32)), f"{what}: scales differ"
    bad = np.argwhere(y != y_ref)
    assert bad.size == 0, f"{what}: {len(bad)} codes differ, first at {bad[:3].tolist()}"


# ------------------------------------------------------------------------------ act_quant

@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
@pytest.mark.parametrize("M,K", [(1, 128), (16, 512), (3, 640), (37, 1024), (300, 7168),
                                 (129, 18432)])
def test_act_quant_bit_exact_small(fmt, M, K):
    x = synth.activations(M, K, seed=M * 7 + K, name="pq", outlier_frac=0.01)
    y, s = gpu_act_quant(x, fmt)
    y_ref, s_ref = oracle.act_quant(x, FMTS[fmt])
    assert_quant_equal(y, s, y_ref, s_ref, f"{M}x{K} {fmt}")


@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
def test_act_quant_special_blocks(fmt):
    rng = np.random.default_rng(5)
    blocks = [np.zeros(128), -np.zeros(128), np.full(128, 448.0), np.full(128, -1e-30),
              np.r_[1.0, np.zeros(127)], np.r_[-2.0, 1.0, 0.5, -0.25, np.zeros(124)],
              rng.standard_normal(128) * 1e-6,           # amax below the 1e-4 clamp
              rng.standard_normal(128) * 3e4,            # large magnitudes
              np.ldexp(1.0, rng.integers(-133, -120, 128)) * rng.choice([-1, 1], 128),  # tiny
              rng.standard_normal(128) * np.exp2(rng.uniform(-20, 20, 128)),  # wide range
              np.linspace(-448, 448, 128),
              # every value a midpoint-ish neighbour of e4m3 grid points after scaling
              (np.arange(128) + 0.5) / 128 * 448.0]
    x = synth.to_bf16_bits(np.stack(blocks).astype(np.float32).reshape(3, -1))
    y, s = gpu_act_quant(x, fmt)
    y_ref, s_ref = oracle.act_quant(x, FMTS[fmt])
    assert_quant_equal(y, s, y_ref, s_ref, f"special {fmt}")


def test_act_quant_every_bf16_value_against_every_scale_exponent():
    """All 65536 bf16 bit patterns (minus NaN/inf) as x, placed in blocks whose amax sets
    scales across the whole exponent range, so that each x meets many scales."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(pats)
    pats = pats[np.isfinite(f)]
    f = np.abs(synth.bf16_bits_to_f32(pats))
    rng = np.random.default_rng(17)
    rows = []
    for amax_exp in range(-20, 128, 3):
        amax = np.float32(np.ldexp(1.0 + rng.integers(0, 128) / 128.0, amax_exp))
        cand = pats[f <= amax]
        cand = cand[rng.permutation(cand.size)][: 127 * 64]
        n = cand.size // 127 * 127
        blk = cand[:n].reshape(-1, 127)
        lead = np.full((blk.shape[0], 1), synth.to_bf16_bits(np.array([amax]))[0], np.uint16)
        rows.append(np.concatenate([lead, blk], axis=1))
    x = np.concatenate(rows).reshape(-1, 128)
    for fmt in ("fp32", "ue8m0"):
        y, s = gpu_act_quant(x, fmt)
        y_ref, s_ref = oracle.act_quant(x, FMTS[fmt])
        assert_quant_equal(y, s, y_ref, s_ref, f"sweep {fmt}")


@pytest.mark.parametrize("name,M,K,fmt", [("decode", 64, 7168, "fp32"),
                                          ("moe_gathered", 8192, 7168, "fp32"),
                                          ("prefill_down", 4096, 18432, "fp32"),
                                          ("mla", 2048, 7168, "ue8m0")])
def test_act_quant_full_size_sampled_rows(name, M, K, fmt):
    x = synth.activations(M, K, seed=0, name=f"full/{name}",
                          outlier_frac=0.0 if name == "mla" else 0.01)
    y, s = gpu_act_quant(x, fmt)
    rows = np.unique(np.r_[0, M - 1, np.random.default_rng(1).integers(0, M, 48)])
    y_ref, s_ref = oracle.act_quant(x[rows], FMTS[fmt])
    assert_quant_equal(y[rows], s[rows], y_ref, s_ref, name)


@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
@pytest.mark.parametrize("M,K", [
    (333, 128 * 121),     # 40293 blocks
    (1000, 128 * 56),     # 56000 blocks
])
def test_act_quant_large_ragged_bit_exact(fmt, M, K):
    """Inputs large enough that every thread takes several grid-stride steps, with a ragged
    last step; every code and scale against the oracle."""
    x = synth.activations(M, K, seed=M + K, name="large", outlier_frac=0.01)
    y, s = gpu_act_quant(x, fmt)
    y_ref, s_ref = oracle.act_quant(x, FMTS[fmt])
    assert_quant_equal(y, s, y_ref, s_ref, f"large {M}x{K} {fmt}")


# ------------------------------------------------------------------------------ weight_dequant

@pytest.mark.parametrize("N,K", [(1, 1), (5, 33), (128, 128), (300, 272), (333, 391),
                                 (576, 7168), (1000, 1040)])
def test_weight_dequant_bit_exact_small(N, K):
    b, s = synth.weights(N, K, seed=N + K, name="pd")
    y = fp8bs.weight_dequant(dev_e4m3(b), dev_f32(s))
    torch.cuda.synchronize()
    assert np.array_equal(host_bf16_bits(y), oracle.weight_dequant(b, s))


def test_weight_dequant_full_size_sampled_rows():
    N, K = synth.INTER, synth.DIM
    b, s = synth.weights(N, K, seed=0, name="full/dequant")
    y = host_bf16_bits(fp8bs.weight_dequant(dev_e4m3(b), dev_f32(s)))
    rows = np.unique(np.r_[0, N - 1, np.random.default_rng(2).integers(0, N, 200)])
    for r in rows:  # per row: the oracle on one row with its scale row
        ref = oracle.weight_dequant(b[r:r + 1], s[r // 128:r // 128 + 1])
        assert np.array_equal(y[r], ref[0]), f"row {r}"


# ------------------------------------------------------------------------------ fp8_gemm

def run_gemm(a_codes, a_s, b_codes, b_s, fmt="fp32"):
    c = fp8bs.fp8_gemm(dev_e4m3(a_codes), dev_f32(a_s), dev_e4m3(b_codes), dev_f32(b_s), fmt)
    torch.cuda.synchronize()
    return host_bf16_f64(c)


def test_gemm_tiny_config():
    t = synth.tiny(0)
    a, a_s = oracle.act_quant(t["x"])
    b, b_s = t["b"]
    assert b_s.shape == (2, 4)
    assert_gemm_close(run_gemm(a, a_s, b, b_s), oracle.gemm(a, a_s, b, b_s), "tiny")


@pytest.mark.parametrize("M,N,K", [
    (1, 256, 512), (8, 576, 1024), (16, 384, 128), (33, 1000, 640), (64, 1536, 1024),
    (100, 130, 256), (128, 2048, 512),                  # swapped-orientation kernel
    (129, 256, 512), (200, 640, 1024), (300, 576, 384), (256, 2304, 256), (513, 97, 256),
    (1200, 4608, 256), (1100, 4736, 256), (1024, 4800, 384), (768, 5120, 1280),
    (1024, 2048, 256), (2048, 1536, 512), (700, 1000, 256), (2048, 1300, 256),
                                                        # normal kernel: 64/128/192/256-wide
                                                        # tiles (192: a thread's columns may
                                                        # span two blocks of b_s), several
                                                        # tiles, ragged tails
])
def test_gemm_shapes_full_compare(M, N, K):
    x = synth.activations(M, K, seed=M + N + K, name="pgA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(N, K, seed=M * N + K, name="pgB")
    assert_gemm_close(run_gemm(a, a_s, b, b_s), oracle.gemm(a, a_s, b, b_s), f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (1, 300, 384), (20, 500, 384), (50, 700, 384), (120, 900, 384),   # three K blocks, each MT
    (7, 9800, 1152), (64, 9800, 2176), (128, 9800, 1408),            # 9, 17, 11: buffers wrap
])                                                  # (77 slabs: too many to split K)
def test_decode_two_issuers_odd_k_blocks(M, N, K):
    """The decode kernel's two MMA issuers take alternate K blocks, each into its own pair of
    TMEM buffers: an odd count leaves one issuer a block more, and more than four blocks wrap
    the buffers. Every element against the oracle, two calls bit-identical."""
    p = fp8bs.fp8bs_gemm_plan(M, N, K, fp8bs.SCALE_FP32, False)
    assert p["kernel"] == fp8bs.KERNEL_SWAPPED and p["ksplit"] == 1, p
    x = synth.activations(M, K, seed=M + N + K, name="issA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(N, K, seed=M + 2 * N + K, name="issB")
    args = (dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s), "fp32")
    c1 = fp8bs.fp8_gemm(*args, workspace=None)
    c2 = fp8bs.fp8_gemm(*args, workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert_gemm_close(host_bf16_f64(c1), oracle.gemm(a, a_s, b, b_s), f"decode {M}x{N}x{K}")


def test_gemm_fp32_stream_k_against_oracle():
    """fp32 scales with a workspace: 180 tiles of 128 x 192 on the SMs share their K loops
    (each owner starts from the next CTA's partial); every element matches the oracle, and two
    calls agree bit for bit."""
    M, N, K = 2560, 2304, 1024
    x = synth.activations(M, K, seed=21, name="skA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(N, K, seed=22, name="skB")
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    args = (dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s), "fp32")
    c1 = fp8bs.fp8_gemm(*args, workspace=ws)
    c2 = fp8bs.fp8_gemm(*args, workspace=ws)
    c0 = fp8bs.fp8_gemm(*args, workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    ref = oracle.gemm(a, a_s, b, b_s)
    assert_gemm_close(host_bf16_f64(c1), ref, "fp32 stream-K")
    assert_gemm_close(host_bf16_f64(c0), ref, "fp32 no workspace")


def test_gemm_k_zero_writes_zeros():
    c = torch.full((5, 24), 3.0, dtype=torch.bfloat16, device="cuda")
    a = torch.empty((5, 0), dtype=torch.float8_e4m3fn, device="cuda")
    b = torch.empty((24, 0), dtype=torch.float8_e4m3fn, device="cuda")
    e = torch.empty((5, 0), dtype=torch.float32, device="cuda")
    f = torch.empty((1, 0), dtype=torch.float32, device="cuda")
    fp8bs.fp8_gemm(a, e, b, f, out=c)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0


def test_gemm_deterministic():
    x = synth.activations(256, 1024, seed=3, name="detA")
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(4096, 1024, seed=3, name="detB")
    c1 = run_gemm(a, a_s, b, b_s)
    c2 = run_gemm(a, a_s, b, b_s)
    assert np.array_equal(c1, c2)


def pipeline_check(x_bits, b, b_s, fmt, what, per_tile=2, weights_constant=False):
    """The whole path on the GPU (act_quant then fp8_gemm, as the benchmark runs it); the
    oracle recomputes act_quant on the sampled rows from the same bf16 input, checks those rows
    bit-exactly, and evaluates the GEMM at sampled positions from its own codes."""
    M, K = x_bits.shape
    N = b.shape[0]
    bt, bst, xt = dev_e4m3(b), dev_f32(b_s), dev_bf16(x_bits)
    torch.cuda.synchronize()
    y, s = fp8bs.act_quant(xt, fmt)          # the GEMM may start while this one finishes
    c = fp8bs.fp8_gemm(y, s, bt, bst, fmt, weights_constant=weights_constant)
    torch.cuda.synchronize()
    mi, ni = lines_and_tiles(M, N, per_tile, seed=M + N)
    rows = np.unique(mi)
    a_ref, as_ref = oracle.act_quant(x_bits[rows], FMTS[fmt])
    assert_quant_equal(host_codes(y)[rows], s.cpu().numpy()[rows], a_ref, as_ref, what)
    # the oracle's GEMM on its own codes of the sampled rows
    local = np.searchsorted(rows, mi).astype(np.int64)
    ref = oracle.gemm_at(a_ref, as_ref, b, b_s, local, ni)
    got = host_bf16_f64(c[torch.from_numpy(mi).cuda(), torch.from_numpy(ni).cuda()])
    return assert_gemm_close(got, ref, what, c_full=c)


@pytest.mark.parametrize("weights_constant", [False, True])
@pytest.mark.parametrize("M", synth.DECODE_MS)
def test_pipeline_decode_full_size(M, weights_constant):
    b, b_s = synth.weights(synth.INTER, synth.DIM, seed=0, name="decode/B")
    pipeline_check(synth.decode(M), b, b_s, "fp32", f"decode M={M}", per_tile=4,
                   weights_constant=weights_constant)


def test_back_to_back_layers_share_buffers():
    """Several act_quant -> GEMM pairs on one stream reusing the same activation and output
    buffers, as consecutive layers do: each kernel may start while the previous one finishes,
    and must still see its inputs complete."""
    K, N, M = synth.DIM, 2048, 32
    ws = [synth.weights(N, K, seed=40 + i, name="layers/B") for i in range(3)]
    xs = [synth.activations(M, K, seed=50 + i, name="layers/A") for i in range(3)]
    y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
    s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    outs = []
    dev_w = [(dev_e4m3(b), dev_f32(bs)) for b, bs in ws]
    dev_x = [dev_bf16(x) for x in xs]
    torch.cuda.synchronize()
    st = torch.cuda.current_stream().cuda_stream
    for i in range(3):
        fp8bs.fp8bs_act_quant(dev_x[i].data_ptr(), y.data_ptr(), s.data_ptr(), M, K, 0, st)
        fp8bs.fp8bs_gemm_ex(y.data_ptr(), s.data_ptr(), dev_w[i][0].data_ptr(),
                            dev_w[i][1].data_ptr(), c.data_ptr(), M, N, K, 0,
                            fp8bs.GEMM_WEIGHTS_CONSTANT, st)
        outs.append(c.clone())
    torch.cuda.synchronize()
    for i in range(3):
        a_ref, as_ref = oracle.act_quant(xs[i])
        assert_gemm_close(host_bf16_f64(outs[i]), oracle.gemm(a_ref, as_ref, *ws[i]), f"layer {i}")


@pytest.mark.parametrize("which", ["up", "down"])
def test_pipeline_prefill_full_size(which):
    if which == "up":
        x, (b, b_s) = synth.prefill_up(), synth.weights(synth.INTER, synth.DIM, 0, "prefill/B_up")
    else:
        x, (b, b_s) = synth.prefill_down(), synth.weights(synth.DIM, synth.INTER, 0, "prefill/B_down")
    pipeline_check(x, b, b_s, "fp32", f"prefill {which}", per_tile=1)


@pytest.mark.parametrize("N", [synth.Q_LORA, synth.KV_LORA_ROPE])
def test_pipeline_mla_ue8m0_full_size(N):
    b, b_s = synth.weights(N, synth.DIM, seed=0, name=f"mla/B{N}", pow2=True)
    pipeline_check(synth.mla_acts(), b, b_s, "ue8m0", f"mla N={N}", per_tile=2)


def test_moe_experts_full_size():
    rows, counts = synth.moe_routing(0)
    assert counts.sum() == 8192 and counts.size == 32
    tokens = synth.activations(1024, synth.DIM, seed=0, name="moe/tokens", outlier_frac=0.01)
    x = tokens[rows]
    y, s = fp8bs.act_quant(dev_bf16(x), "fp32")
    offsets = np.r_[0, np.cumsum(counts)]
    outs = []
    weights = [synth.weights(synth.MOE_INTER, synth.DIM, seed=0, name=f"moe/B{e}") for e in range(32)]
    for e in range(32):
        lo, hi = offsets[e], offsets[e + 1]
        b, b_s = weights[e]
        outs.append(fp8bs.fp8_gemm(y[lo:hi], s[lo:hi], dev_e4m3(b), dev_f32(b_s)))
    torch.cuda.synchronize()
    y_h, s_h = host_codes(y), s.cpu().numpy()
    for e in range(32):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        b, b_s = weights[e]
        mi, ni = lines_and_tiles(hi - lo, synth.MOE_INTER, 1, seed=e, n_rows=1, n_cols=1)
        rows_e = np.unique(mi)
        a_ref, as_ref = oracle.act_quant(x[lo + rows_e])
        assert_quant_equal(y_h[lo + rows_e], s_h[lo + rows_e], a_ref, as_ref, f"expert {e}")
        ref = oracle.gemm_at(a_ref, as_ref, b, b_s, np.searchsorted(rows_e, mi), ni)
        got = host_bf16_f64(outs[e])[mi, ni]
        assert_gemm_close(got, ref, f"expert {e} (M_e={hi - lo})", c_full=outs[e])


def grouped_check(counts, N, K, seed, what, per_tile=None, fmt="fp32"):
    """Grouped GEMM of stacked experts against the oracle, group by group. With fmt="ue8m0"
    every scale is a power of two (act_quant's ue8m0 scales, 2^e weight scales)."""
    counts = np.asarray(counts, dtype=np.int64)
    offs = np.r_[0, np.cumsum(counts)]
    T = int(offs[-1])
    x = synth.activations(max(T, 1), K, seed=seed, name="grpA", outlier_frac=0.01)[:T]
    a, a_s = oracle.act_quant(x, FMTS[fmt]) if T else \
        (np.zeros((0, K), np.uint8), np.zeros((0, K // 128), np.float32))
    ws = [synth.weights(N, K, seed=seed + 1 + e, name="grpB", pow2=fmt == "ue8m0")
          for e in range(len(counts))]
    b = np.stack([w for w, _ in ws])
    b_s = np.stack([s for _, s in ws])
    c_dev = fp8bs.fp8_gemm_grouped(dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s), offs,
                                   fmt)
    torch.cuda.synchronize()
    c = host_bf16_f64(c_dev)
    for e in range(len(counts)):
        lo, hi = offs[e], offs[e + 1]
        if hi == lo:
            continue
        if per_tile is None:
            ref = oracle.gemm(a[lo:hi], a_s[lo:hi], b[e], b_s[e])
            assert_gemm_close(c[lo:hi], ref, f"{what} group {e}")
        else:
            mi, ni = lines_and_tiles(hi - lo, N, per_tile, seed=e, n_rows=1, n_cols=1)
            ref = oracle.gemm_at(a[lo:hi], a_s[lo:hi], b[e], b_s[e], mi, ni)
            assert_gemm_close(c[lo:hi][mi, ni], ref, f"{what} group {e}", c_full=c[lo:hi])


@pytest.mark.parametrize("counts,N,K", [
    ([37], 256, 256),                          # one group
    ([0, 130, 5, 0, 257, 1], 384, 256),        # empty groups, ragged counts, N tail vs BN
    ([64] * 8, 576, 512),                      # N not a multiple of the tile width
    ([300, 0, 200], 2048, 256),
])
def test_gemm_grouped_against_oracle(counts, N, K):
    grouped_check(counts, N, K, seed=sum(counts) + N, what=f"grouped {counts}")


@pytest.mark.parametrize("counts,N,K,fmt", [
    ([1, 8, 32, 64], 2048, 7168, "fp32"),      # decode-sized groups: one swapped launch
    ([3, 17, 40], 1000, 2048, "fp32"),         # ragged N, the K loop split in clusters
    ([0, 5, 0, 64, 2], 576, 1024, "ue8m0"),
    ([200, 3, 0, 64, 130, 1], 384, 512, "fp32"),  # both launches: tiles, then swapped groups
    # ten small groups x 16 weight slabs would be 160 CTAs on 152 SMs: the largest small group
    # (64 rows) joins the tiles as one padded tile, the other nine stay in the swapped launch
    ([300, 40, 3, 17, 64, 1, 9, 33, 50, 12, 28], 2048, 256, "fp32"),
    ([300, 40, 3, 17, 64, 1, 9, 33, 50, 12, 28], 2048, 256, "ue8m0"),
])
def test_gemm_grouped_small_groups(counts, N, K, fmt):
    """Groups of at most 64 rows run in the swapped orientation (with other groups: as a
    second launch that starts without waiting for the first); every element against the
    oracle."""
    grouped_check(counts, N, K, seed=sum(counts) + N + 3, what=f"grouped small {counts}", fmt=fmt)


def test_gemm_grouped_moe_full_size():
    """The MoE workload (1024 tokens x 8 slots over 32 experts, N=2048, K=7168) in one call."""
    rows, counts = synth.moe_routing(0)
    grouped_check(counts, synth.MOE_INTER, synth.DIM, seed=7, what="moe", per_tile=1)


def test_gemm_grouped_k_zero_and_no_rows():
    c = torch.full((6, 16), 2.0, dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8bs_gemm_grouped(0, 0, 0, 0, c.data_ptr(), [0, 2, 6], 2, 16, 0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0
    fp8bs.fp8bs_gemm_grouped(0, 0, 0, 0, 0, [0, 0, 0], 2, 16, 128)   # no rows: nothing runs


# ------------------------------------------------------------------------------ ue8m0 block-scaled MMA
# With FP8BS_SCALE_UE8M0 and more than 128 rows the tensor cores apply the power-of-two scales
# themselves (block-scaled MMA); the oracle is the same fp64 GEMM on the same codes and scales.

def pow2_case(M, N, K, seed):
    x = synth.activations(M, K, seed=seed, name="bsA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x, oracle.SCALE_UE8M0)
    b, b_s = synth.weights(N, K, seed=seed + 1, name="bsB", pow2=True)
    return a, a_s, b, b_s


@pytest.mark.parametrize("M,N,K", [
    (64, 1536, 1024),                                   # few rows: swapped kernel, ue8m0 scales
    (129, 256, 512), (200, 640, 1024), (300, 576, 384), (513, 97, 256), (1024, 2048, 256),
    (2048, 1536, 512), (700, 1000, 256), (1100, 4736, 256), (256, 128, 7168), (384, 200, 2048),
    (300, 576, 128),        # 64-wide tiles, one K block: the second MMA issuer has none
])
def test_gemm_ue8m0_block_scaled_full_compare(M, N, K):
    a, a_s, b, b_s = pow2_case(M, N, K, M + N + K)
    assert_gemm_close(run_gemm(a, a_s, b, b_s, "ue8m0"), oracle.gemm(a, a_s, b, b_s),
                      f"ue8m0 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (2560, 4096, 256),     # 320 tiles of 128 x 256: the 256-wide block-scaled kernel
    (2600, 3900, 384),     # ragged rows; the last tile holds one 128-row block of B, half past N
])
def test_gemm_ue8m0_256_wide_tiles(M, N, K):
    a, a_s, b, b_s = pow2_case(M, N, K, M + N + K)
    assert_gemm_close(run_gemm(a, a_s, b, b_s, "ue8m0"), oracle.gemm(a, a_s, b, b_s),
                      f"ue8m0 {M}x{N}x{K}")


def random_codes(rng, rows, cols):
    c = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x00                        # no NaN codes
    return c


@pytest.mark.parametrize("M,N,K", [
    (384, 384, 1152),      # 128-wide tiles
    (2560, 4096, 640),     # 256-wide tiles: two blocks of B, two exponents per tile
])
def test_gemm_ue8m0_per_row_and_block_exponents(M, N, K):
    """Every row of A and every 128-row block of B carries its own exponent in every K block,
    so a scale factor taken from the wrong row, column block, K block or pipeline stage moves
    whole output regions out of tolerance."""
    rng = np.random.default_rng(11)
    a, b = random_codes(rng, M, K), random_codes(rng, N, K)
    m = np.arange(M)[:, None]
    kb = np.arange(K // 128)[None, :]
    a_s = np.ldexp(1.0, ((m * 7 + kb * 3) % 9) - 4 - 8).astype(np.float32)
    nb = np.arange(N // 128)[:, None]
    b_s = np.ldexp(1.0, ((nb * 5 + kb * 2) % 7) - 3 - 8).astype(np.float32)
    c = run_gemm(a, a_s, b, b_s, "ue8m0")
    if M * N <= 384 * 384:
        assert_gemm_close(c, oracle.gemm(a, a_s, b, b_s), "ue8m0 exponent pattern")
    else:
        mi, ni = lines_and_tiles(M, N, 2, seed=K)
        assert_gemm_close(c[mi, ni], oracle.gemm_at(a, a_s, b, b_s, mi, ni),
                          "ue8m0 exponent pattern (sampled)", c_full=c)


def test_gemm_ue8m0_extreme_exponents():
    """Scales at the ends of the ue8m0 range that act_quant and the weights can produce."""
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(12)
    a, b = random_codes(rng, M, K), random_codes(rng, N, K)
    a_s = np.ldexp(1.0, rng.integers(-22, 0, size=(M, K // 128))).astype(np.float32)
    b_s = np.ldexp(1.0, rng.integers(-10, 30, size=(N // 128, K // 128))).astype(np.float32)
    assert_gemm_close(run_gemm(a, a_s, b, b_s, "ue8m0"), oracle.gemm(a, a_s, b, b_s),
                      "ue8m0 extreme exponents")


def test_gemm_ue8m0_reports_a_scale_that_is_not_a_power_of_two():
    a, a_s, b, b_s = pow2_case(256, 256, 256, 5)
    b_s = b_s.copy()
    b_s[1, 1] *= np.float32(1.5)
    run_gemm(a, a_s, b, b_s, "ue8m0")
    assert fp8bs.fp8bs_device_error(clear=True) & fp8bs.DEVERR_SCALE_NOT_POW2


@pytest.mark.parametrize("counts,N,K", [
    ([0, 130, 5, 0, 257, 1], 384, 256),
    ([64] * 8, 576, 512),
    ([300, 0, 200], 2048, 256),
    ([600, 0, 700, 650, 100], 1536, 256),    # 192-wide tiles (two issuers, one buffer); the
                                             # coalesced stores stop at each group's last row
])
def test_gemm_grouped_ue8m0_block_scaled(counts, N, K):
    grouped_check(counts, N, K, seed=sum(counts) + N + 1, what=f"grouped ue8m0 {counts}",
                  fmt="ue8m0")


def run_gemm_ws(a_codes, a_s, b_codes, b_s, ws, fmt="ue8m0"):
    """With a workspace and at least as many 128 x 128 tiles as SMs: the block-scaled kernel's
    stream-K schedule, selected explicitly (the automatic plan prefers wider whole tiles for
    these shapes); otherwise the automatic plan."""
    M, K = a_codes.shape
    N = b_codes.shape[0]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if ws is not None and fmt == "ue8m0" and -(-M // 128) * -(-N // 128) >= sms:
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        A, AS, B, BS = dev_e4m3(a_codes), dev_f32(a_s), dev_e4m3(b_codes), dev_f32(b_s)
        fp8bs.fp8bs_gemm_config(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(),
                                c.data_ptr(), M, N, K, fp8bs.SCALE_UE8M0, 0,
                                fp8bs.KERNEL_BLOCK_SCALED, 128, 0, ws.data_ptr(), ws.numel(),
                                torch.cuda.current_stream().cuda_stream)
    else:
        c = fp8bs.fp8_gemm(dev_e4m3(a_codes), dev_f32(a_s), dev_e4m3(b_codes), dev_f32(b_s),
                           fmt, workspace=ws)
    torch.cuda.synchronize()
    return host_bf16_f64(c)


@pytest.mark.parametrize("M,N,K,full", [
    (1100, 2500, 2048, True),    # 180 tiles, ragged rows and columns, each shared by two CTAs
    (1024, 2560, 2048, True),    # 160 tiles
    (256, 256, 1024, True),      # 4 tiles: too few to share, computed whole
    (2048, 1536, 7168, False),   # the MLA q projection, 192 tiles of 56 K blocks
])
def test_gemm_ue8m0_stream_k_against_oracle(M, N, K, full):
    """With a workspace the block-scaled GEMM shares tiles' K loops between CTAs; every output
    element (or a sample hitting every tile) must still match the oracle, and repeated calls on
    the same workspace agree bit for bit (the partials are added in a fixed order, and the
    workspace's counters return to zero after each call)."""
    a, a_s, b, b_s = pow2_case(M, N, K, M * 3 + N + K)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    c1 = run_gemm_ws(a, a_s, b, b_s, ws)
    c2 = run_gemm_ws(a, a_s, b, b_s, ws)
    c0 = run_gemm_ws(a, a_s, b, b_s, None)
    assert np.array_equal(c1, c2)
    if full:
        ref = oracle.gemm(a, a_s, b, b_s)
        assert_gemm_close(c1, ref, f"stream-K {M}x{N}x{K}")
        assert_gemm_close(c0, ref, f"no workspace {M}x{N}x{K}")
    else:
        mi, ni = lines_and_tiles(M, N, 1, seed=M + N)
        ref = oracle.gemm_at(a, a_s, b, b_s, mi, ni)
        assert_gemm_close(c1[mi, ni], ref, f"stream-K {M}x{N}x{K}", c_full=c1)
        assert_gemm_close(c0[mi, ni], ref, f"no workspace {M}x{N}x{K}", c_full=c0)


def test_gemm_ue8m0_stream_k_after_whole_tiles():
    """320 tiles: the first 152 are computed whole, the last 168 share their K loops."""
    M, N, K = 2560, 2048, 2048
    a, a_s, b, b_s = pow2_case(M, N, K, 23)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    c = run_gemm_ws(a, a_s, b, b_s, ws)
    mi, ni = lines_and_tiles(M, N, 2, seed=5)
    assert_gemm_close(c[mi, ni], oracle.gemm_at(a, a_s, b, b_s, mi, ni), "ue8m0 hybrid stream-K",
                      c_full=c)


def test_gemm_ue8m0_stream_k_workspace_reused_across_shapes():
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    for M, N, K in [(1024, 2560, 2048), (1100, 2500, 2048), (256, 256, 1024), (1024, 2560, 2048)]:
        a, a_s, b, b_s = pow2_case(M, N, K, M + N)
        assert_gemm_close(run_gemm_ws(a, a_s, b, b_s, ws), oracle.gemm(a, a_s, b, b_s),
                          f"reused workspace {M}x{N}x{K}")


def test_gemm_ws_rejects_a_short_workspace():
    a, a_s, b, b_s = pow2_case(256, 256, 256, 3)
    need = fp8bs.fp8bs_gemm_workspace_size()
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    c = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
    A, AS, B, BS = dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s)
    with pytest.raises(fp8bs.Fp8bsError):
        fp8bs.fp8bs_gemm_ws(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(), c.data_ptr(),
                            256, 256, 256, 1, 0, ws.data_ptr(), need - 1)


def test_gemm_ue8m0_deterministic():
    a, a_s, b, b_s = pow2_case(512, 1024, 1024, 9)
    assert np.array_equal(run_gemm(a, a_s, b, b_s, "ue8m0"), run_gemm(a, a_s, b, b_s, "ue8m0"))


# ------------------------------------------------------------------------------ act_quant + GEMM
# fp8bs_act_quant_gemm: act_quant then the GEMM in one call, or (FP8BS_GEMM_QUANT_IN_KERNEL,
# M <= 16) one kernel that quantises the activations itself; y, s and C must equal those of the
# two separate calls bit for bit.

def separate_act_quant_gemm(xt, bt, bst, fmt, ws):
    y, s = fp8bs.act_quant(xt, fmt)
    c = fp8bs.fp8_gemm(y, s, bt, bst, fmt, workspace=ws)
    return c, y, s


@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
@pytest.mark.parametrize("M,N,K", [
    # M <= 16: the one-kernel form applies where the separate GEMM would not split K (more
    # than 76 weight slabs, or too few K blocks to split)
    (1, 18432, 7168), (3, 20480, 256), (16, 10000, 2048), (5, 12000, 4096), (9, 1000, 128),
    (8, 2048, 7168),       # 16 slabs: the separate GEMM splits K, so two launches
    (7, 1000, 18432),      # K too long for the resident activations: two launches
    (17, 1000, 18432), (32, 576, 1024), (64, 18432, 7168),   # M > 16: two launches
    (100, 1536, 2048), (128, 4096, 512),   # two launches whatever the flag (swapped)
    (300, 1024, 512),      # two launches, normal orientation
])
def test_act_quant_gemm_matches_separate_calls(fmt, M, N, K):
    x = synth.activations(M, K, seed=M + N + K, name="aqgA", outlier_frac=0.01)
    b, b_s = synth.weights(N, K, seed=N + K, name="aqgB", pow2=fmt == "ue8m0")
    xt, bt, bst = dev_bf16(x), dev_e4m3(b), dev_f32(b_s)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    c0, y0, s0 = separate_act_quant_gemm(xt, bt, bst, fmt, ws)
    for in_kernel in (False, True, True):                 # default, then the one-kernel form
        c1, y1, s1 = fp8bs.act_quant_gemm(xt, bt, bst, fmt, weights_constant=True, workspace=ws,
                                          quant_in_kernel=in_kernel)
        torch.cuda.synchronize()
        assert torch.equal(y1.view(torch.uint8), y0.view(torch.uint8))
        assert torch.equal(s1.view(torch.int32), s0.view(torch.int32))
        assert torch.equal(c1.view(torch.int16), c0.view(torch.int16))
    # and against the oracle on the codes it produced itself
    a_ref, as_ref = oracle.act_quant(x, FMTS[fmt])
    assert_quant_equal(host_codes(y1), s1.cpu().numpy(), a_ref, as_ref, f"aqg {M}x{K}")
    mi, ni = lines_and_tiles(M, N, 2, seed=K)
    ref = oracle.gemm_at(a_ref, as_ref, b, b_s, mi, ni)
    assert_gemm_close(host_bf16_f64(c1)[mi, ni], ref, f"aqg {M}x{N}x{K}", c_full=c1)


def test_act_quant_gemm_without_workspace():
    x = synth.activations(16, 1024, seed=4, name="aqgA")
    b, b_s = synth.weights(512, 1024, seed=5, name="aqgB")
    xt, bt, bst = dev_bf16(x), dev_e4m3(b), dev_f32(b_s)
    c0, y0, s0 = separate_act_quant_gemm(xt, bt, bst, "fp32", None)
    c1, y1, s1 = fp8bs.act_quant_gemm(xt, bt, bst, "fp32", workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c0.view(torch.int16))
    assert torch.equal(y1.view(torch.uint8), y0.view(torch.uint8))


# ------------------------------------------------------------------------------ bf16 path
# fp8bs_linear_bf16: x . bf16(dequant(W))^T with the weight dequantised tile by tile on chip;
# the oracle dequantises with weight_dequant's arithmetic and multiplies in binary64.

@pytest.mark.parametrize("M,N,K", [
    (1, 256, 128), (5, 576, 512), (16, 1000, 1024), (17, 384, 256), (40, 2048, 2048),
    (64, 1536, 7168),
    (40, 128, 384),       # three K blocks: the two accumulators and dequantiser groups unequal
    (64, 128, 640),       # five K blocks
    (3, 256, 896),        # seven K blocks
    (65, 256, 512),       # 128 rows of x per CTA from here on
    (128, 384, 1024),
    (200, 1000, 768),     # ragged in M and N
    (1000, 640, 384),     # eight tiles of x share each slab
])
def test_linear_bf16_against_oracle(M, N, K):
    x = synth.activations(M, K, seed=M + N, name="linA", outlier_frac=0.01)
    w, w_s = synth.weights(N, K, seed=N + K, name="linB")
    y = fp8bs.linear_bf16(dev_bf16(x), dev_e4m3(w), dev_f32(w_s))
    torch.cuda.synchronize()
    assert_gemm_close(host_bf16_f64(y), oracle.linear_bf16(x, w, w_s), f"bf16 path {M}x{N}x{K}")


@pytest.mark.parametrize("M", synth.DECODE_MS)
def test_linear_bf16_decode_full_size(M):
    w, w_s = synth.weights(synth.INTER, synth.DIM, seed=0, name="decode/B")
    x = synth.decode(M)
    y = fp8bs.linear_bf16(dev_bf16(x), dev_e4m3(w), dev_f32(w_s), weights_constant=True)
    torch.cuda.synchronize()
    assert_gemm_close(host_bf16_f64(y), oracle.linear_bf16(x, w, w_s), f"bf16 path decode M={M}")


def test_linear_bf16_prefill_sampled_rows():
    """Prefill size (4096 x 18432 x 7168, 32 tiles of x per weight slab): sixteen rows,
    first and last rows of tiles among them, against the oracle."""
    x = synth.prefill_up()
    w, w_s = synth.weights(synth.INTER, synth.DIM, seed=0, name="prefill/B_up")
    y = fp8bs.linear_bf16(dev_bf16(x), dev_e4m3(w), dev_f32(w_s), weights_constant=True)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 1000, 2047, 2048, 2049, 3071, 3200, 3968, 4000, 4094,
                     4095, 255, 513])
    got = host_bf16_f64(y[torch.from_numpy(rows).to(y.device)])
    assert_gemm_close(got, oracle.linear_bf16(x[rows], w, w_s), "bf16 path prefill rows")


def test_linear_bf16_phases_with_a_partial_last_phase():
    """4352 rows of x at K = 7168 make 17 pairs of 128-row tiles, which the kernel runs in
    phases of 8 (a quarter of L2 each): 8, 8 and 1. Whole rows from every tile pair (first and
    last of each) and whole columns across all rows, against the oracle."""
    M, N, K = 4352, 1000, synth.DIM
    x = synth.activations(M, K, seed=11, name="phaseX", outlier_frac=0.01)
    w, w_s = synth.weights(N, K, seed=12, name="phaseW")
    y = fp8bs.linear_bf16(dev_bf16(x), dev_e4m3(w), dev_f32(w_s))
    torch.cuda.synchronize()
    rows = np.unique(np.r_[np.arange(0, M, 256), np.arange(255, M, 256), 4096, 4351])
    got = host_bf16_f64(y[torch.from_numpy(rows).to(y.device)])
    assert_gemm_close(got, oracle.linear_bf16(x[rows], w, w_s), "bf16 phases: rows")
    cols = np.array([0, 127, 128, 511, 999])
    got = host_bf16_f64(y[:, torch.from_numpy(cols).to(y.device)])
    # one weight row at a time, with the scale row of its 128-row block
    ref = np.concatenate([oracle.linear_bf16(x, w[c:c + 1], w_s[c // 128:c // 128 + 1])
                          for c in cols], axis=1)
    assert_gemm_close(got, ref, "bf16 phases: cols")


def test_linear_bf16_large_block_scales():
    """Block scales of 2^8 and above, mixed with small ones in one weight: the dequantisers'
    fp32 product and bf16 rounding must hold at any finite scale."""
    M, N, K = 8, 384, 768
    x = synth.activations(M, K, seed=6, name="linA")
    w, w_s = synth.weights(N, K, seed=7, name="linB")
    w_s = w_s.copy()
    w_s[::2, ::2] = np.float32(300.0)
    w_s[1, 1] = np.float32(2.0 ** 20)
    y = fp8bs.linear_bf16(dev_bf16(x), dev_e4m3(w), dev_f32(w_s))
    torch.cuda.synchronize()
    assert_gemm_close(host_bf16_f64(y), oracle.linear_bf16(x, w, w_s), "large scales")


def test_linear_bf16_deterministic_and_k_zero():
    x = synth.activations(9, 1024, seed=2, name="linA")
    w, w_s = synth.weights(640, 1024, seed=3, name="linB")
    args = (dev_bf16(x), dev_e4m3(w), dev_f32(w_s))
    y1, y2 = fp8bs.linear_bf16(*args), fp8bs.linear_bf16(*args)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    y = torch.full((4, 32), 1.0, dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8bs_linear_bf16(0, 0, 0, y.data_ptr(), 4, 32, 0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0


# ------------------------------------------------------------------------------ bounded waits

def test_bounded_wait_reports_instead_of_hanging():
    fp8bs.fp8bs_probe_wait_timeout(5_000_000)  # 5 ms on a barrier nothing signals
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) & fp8bs.DEVERR_PROBE
    # the context is still usable
    t = synth.tiny(0)
    a, a_s = oracle.act_quant(t["x"])
    b, b_s = t["b"]
    assert_gemm_close(run_gemm(a, a_s, b, b_s), oracle.gemm(a, a_s, b, b_s), "after probe")


def test_stream_k_while_another_stream_holds_sms():
    """A stream-K GEMM launched while a kernel on another stream holds half the SMs for longer
    than any wait inside the library may last (2.2 s against 2 s): the stream-K grid is a
    cooperative launch, so its CTAs are placed together once the SMs are free, and no tile's
    owner waits on a contributor that has no SM. C is bit-identical to an uncontended call and
    no wait runs out."""
    M, N, K = 2560, 2304, 1024          # 220 tiles 192 wide, all shared (fp32 scales)
    assert fp8bs.fp8bs_gemm_plan(M, N, K, fp8bs.SCALE_FP32, True)["stream_k"]
    x = synth.activations(M, K, seed=31, name="occA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x)
    b, b_s = synth.weights(N, K, seed=32, name="occB")
    A, AS, B, BS = dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    ref = fp8bs.fp8_gemm(A, AS, B, BS, "fp32", workspace=ws)
    whole = torch.empty_like(ref)
    fp8bs.fp8bs_gemm_config(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(),
                            whole.data_ptr(), M, N, K, fp8bs.SCALE_FP32, 0,
                            fp8bs.KERNEL_PROMOTED, 192, 1, 0, 0,
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    # the shared tiles add their partials in another order than whole tiles: the reference
    # really ran the stream-K schedule
    assert not torch.equal(whole.view(torch.int16), ref.view(torch.int16))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    other = torch.cuda.Stream()
    fp8bs.fp8bs_probe_occupy(sms // 2, 2_200_000_000, other.cuda_stream)
    c = fp8bs.fp8_gemm(A, AS, B, BS, "fp32", workspace=ws)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=False) == 0
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))
    assert_gemm_close(host_bf16_f64(c), oracle.gemm(a, a_s, b, b_s), "stream-K under contention")
