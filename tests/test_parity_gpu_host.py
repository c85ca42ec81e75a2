"""Host buffers used in place. On GB300 the GPU reaches pinned (page-locked) host memory over
NVLink-C2C, and the C ABI lets act_quant read its input x there and the GEMMs (and the bf16
path) write their output there. Every case runs twice through the C ABI, once with device
buffers and once with pinned host buffers, and the results must agree bit for bit; act_quant's
codes and scales, and the GEMM results, are also checked against the oracle.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import assert_gemm_close, dev_bf16, dev_e4m3, dev_f32, host_bf16_f64

pytestmark = pytest.mark.gpu

WC = fp8bs.GEMM_WEIGHTS_CONSTANT
QIK = fp8bs.GEMM_QUANT_IN_KERNEL
FMTS = {"fp32": fp8bs.SCALE_FP32, "ue8m0": fp8bs.SCALE_UE8M0}
ORACLE_FMTS = {"fp32": oracle.SCALE_FP32, "ue8m0": oracle.SCALE_UE8M0}


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"


def pinned_like(t: torch.Tensor) -> torch.Tensor:
    """A pinned host tensor of t's shape and dtype, filled with NaN bytes (0xFF)."""
    h = torch.empty(t.shape, dtype=t.dtype).pin_memory()
    h.view(torch.uint8).fill_(0xFF)
    return h


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.uint8).cpu()


def stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("M,K,fmt", [(1, 7168, "fp32"), (64, 7168, "ue8m0"), (300, 1024, "fp32")])
def test_act_quant_reads_x_from_host_memory(M, K, fmt):
    x = synth.activations(M, K, seed=M, name="hostX", outlier_frac=0.01)
    xd = dev_bf16(x)
    xh = xd.cpu().pin_memory()
    out = []
    for src in (xd, xh):
        y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
        fp8bs.fp8bs_act_quant(src.data_ptr(), y.data_ptr(), s.data_ptr(), M, K, FMTS[fmt],
                              stream())
        out.append((y, s))
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.act_quant(x, ORACLE_FMTS[fmt])
    assert torch.equal(bits(out[0][0]), bits(out[1][0]))
    assert torch.equal(bits(out[0][1]), bits(out[1][1]))
    assert np.array_equal(out[1][0].view(torch.uint8).cpu().numpy(), y_ref)
    assert np.array_equal(out[1][1].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("M,N,K,fmt,flags", [
    (1, 18432, 7168, "fp32", WC),          # swapped orientation, 144 weight slabs
    (8, 18432, 7168, "ue8m0", WC | QIK),   # the in-kernel quantisation reads x itself
    (64, 2048, 7168, "fp32", WC),          # few slabs: K split in clusters
    (300, 1000, 1024, "ue8m0", 0),         # block-scaled MMA
    (300, 1000, 1024, "fp32", 0),          # fp32 scale promotion
])
def test_act_quant_gemm_with_x_and_c_in_host_memory(M, N, K, fmt, flags):
    x = synth.activations(M, K, seed=M + N, name="hostAQ", outlier_frac=0.01)
    b, b_s = synth.weights(N, K, seed=K, name="hostAQB", pow2=fmt == "ue8m0")
    xd, B, BS = dev_bf16(x), dev_e4m3(b), dev_f32(b_s)
    xh = xd.cpu().pin_memory()
    ws = fp8bs.gemm_workspace()
    res = []
    for src, host_c in ((xd, False), (xh, True)):
        y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        if host_c:
            c = pinned_like(c)
        fp8bs.fp8bs_act_quant_gemm(src.data_ptr(), y.data_ptr(), s.data_ptr(), B.data_ptr(),
                                   BS.data_ptr(), c.data_ptr(), M, N, K, FMTS[fmt], flags,
                                   ws.data_ptr(), ws.numel(), stream())
        res.append((c, y, s))
    torch.cuda.synchronize()
    for (t_dev, t_host, name) in zip(res[0], res[1], ("C", "y", "s")):
        assert torch.equal(bits(t_dev), bits(t_host)), f"{name} differs with host buffers"
    a, a_s = oracle.act_quant(x, ORACLE_FMTS[fmt])
    assert np.array_equal(res[1][1].view(torch.uint8).cpu().numpy(), a)
    rows = np.unique(np.r_[0, M - 1, np.arange(0, M, max(1, M // 8))])
    assert_gemm_close(host_bf16_f64(res[1][0])[rows], oracle.gemm(a[rows], a_s[rows], b, b_s),
                      f"{M}x{N}x{K} {fmt} C in host memory", c_full=res[1][0])


@pytest.mark.parametrize("M,N,K,fmt,how", [
    (2560, 2048, 2048, "fp32", "workspace"),   # the plan takes stream-K: owners add partials
    (1100, 2500, 2048, "ue8m0", "stream-K"),   # block-scaled stream-K, chosen explicitly
    (2048, 1536, 1024, "ue8m0", "plan"),       # block-scaled whole tiles
    (120, 1000, 2048, "fp32", "plan"),         # swapped orientation, several M rows per tile
])
def test_gemm_writes_c_to_host_memory(M, N, K, fmt, how):
    if how == "workspace":
        assert fp8bs.fp8bs_gemm_plan(M, N, K, FMTS[fmt], True)["stream_k"]
    x = synth.activations(M, K, seed=N, name="hostG", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x, ORACLE_FMTS[fmt])
    b, b_s = synth.weights(N, K, seed=M, name="hostGB", pow2=fmt == "ue8m0")
    A, AS, B, BS = dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ch = pinned_like(cd)
    for c in (cd, ch):
        ptrs = (A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(), c.data_ptr())
        if how == "stream-K":
            fp8bs.fp8bs_gemm_config(*ptrs, M, N, K, FMTS[fmt], 0, fp8bs.KERNEL_BLOCK_SCALED, 128,
                                    0, ws.data_ptr(), ws.numel(), stream())
        else:
            use_ws = how == "workspace"
            fp8bs.fp8bs_gemm_ws(*ptrs, M, N, K, FMTS[fmt], 0, ws.data_ptr() if use_ws else 0,
                                ws.numel() if use_ws else 0, stream())
    torch.cuda.synchronize()
    assert torch.equal(bits(cd), bits(ch))
    rows = np.unique(np.r_[0, M - 1, np.arange(0, M, max(1, M // 16))])
    assert_gemm_close(host_bf16_f64(ch)[rows], oracle.gemm(a[rows], a_s[rows], b, b_s),
                      f"{M}x{N}x{K} {fmt} C in host memory", c_full=ch)


def test_grouped_and_bf16_path_write_to_host_memory():
    K, N = 1024, 1000
    counts = [0, 5, 300, 40, 129]
    offs = np.r_[0, np.cumsum(counts)]
    T, G = int(offs[-1]), len(counts)
    x = synth.activations(T, K, seed=1, name="hostGr", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x, oracle.SCALE_FP32)
    w = [synth.weights(N, K, seed=10 + e, name="hostGrB") for e in range(G)]
    b, b_s = np.stack([v for v, _ in w]), np.stack([s for _, s in w])
    A, AS, B, BS = dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s)
    cd = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    ch = pinned_like(cd)
    offs_list = [int(v) for v in offs]
    for c in (cd, ch):
        fp8bs.fp8bs_gemm_grouped(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(),
                                 c.data_ptr(), offs_list, G, N, K, fp8bs.SCALE_FP32, stream())
    torch.cuda.synchronize()
    assert torch.equal(bits(cd), bits(ch))
    for e in range(G):
        lo, hi = offs[e], offs[e + 1]
        if hi > lo:
            assert_gemm_close(host_bf16_f64(ch)[lo:hi], oracle.gemm(a[lo:hi], a_s[lo:hi], b[e], b_s[e]),
                              f"grouped C in host memory, group {e}")
    # the bf16 path: y in host memory (x and the weight stay on the device)
    for M in (1, 300):
        xb = synth.activations(M, K, seed=M, name="hostL", outlier_frac=0.01)
        X, W, WS = dev_bf16(xb), dev_e4m3(b[0]), dev_f32(b_s[0])
        yd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        yh = pinned_like(yd)
        for y in (yd, yh):
            fp8bs.fp8bs_linear_bf16(X.data_ptr(), W.data_ptr(), WS.data_ptr(), y.data_ptr(),
                                    M, N, K, WC, stream())
        torch.cuda.synchronize()
        assert torch.equal(bits(yd), bits(yh))
        assert_gemm_close(host_bf16_f64(yh), oracle.linear_bf16(xb, b[0], b_s[0]),
                          f"bf16 path y in host memory, M={M}")


def test_tensor_helpers_take_pinned_host_x_and_out():
    """The binding's helpers with host tensors: act_quant and act_quant_gemm on a pinned x,
    fp8_gemm, act_quant_gemm, linear_bf16 and fp8_gemm_grouped into a pinned `out`; each equal
    bit for bit to the same helper on device tensors."""
    M, N, K = 8, 1000, 1024
    x = synth.activations(M, K, seed=3, name="hostHx", outlier_frac=0.01)
    b, b_s = synth.weights(N, K, seed=4, name="hostHb")
    xd, B, BS = dev_bf16(x), dev_e4m3(b), dev_f32(b_s)
    xh = xd.cpu().pin_memory()
    yd, sd = fp8bs.act_quant(xd)
    yh, sh = fp8bs.act_quant(xh)
    assert yh.is_cuda and torch.equal(bits(yd), bits(yh)) and torch.equal(bits(sd), bits(sh))
    cd, _, _ = fp8bs.act_quant_gemm(xd, B, BS, weights_constant=True)
    out = pinned_like(cd)
    ch, _, _ = fp8bs.act_quant_gemm(xh, B, BS, weights_constant=True, out=out)
    torch.cuda.synchronize()
    assert ch is out and torch.equal(bits(cd), bits(ch))
    out = pinned_like(cd)
    fp8bs.fp8_gemm(yd, sd, B, BS, out=out)
    torch.cuda.synchronize()
    assert torch.equal(bits(out), bits(cd))
    out = pinned_like(cd)
    fp8bs.linear_bf16(xd, B, BS, out=out)
    torch.cuda.synchronize()
    assert torch.equal(bits(out), bits(fp8bs.linear_bf16(xd, B, BS)))
    offs = [0, 3, 8]
    stack_b, stack_s = torch.stack([B, B]), torch.stack([BS, BS])
    gd = fp8bs.fp8_gemm_grouped(yd, sd, stack_b, stack_s, offs)
    out = pinned_like(gd)
    fp8bs.fp8_gemm_grouped(yd, sd, stack_b, stack_s, offs, out=out)
    torch.cuda.synchronize()
    assert torch.equal(bits(out), bits(gd))


def test_tensor_helpers_reject_a_wrong_out_before_launching():
    M, N, K = 8, 1000, 1024
    x = synth.activations(M, K, seed=5, name="hostBad", outlier_frac=0.01)
    b, b_s = synth.weights(N, K, seed=6, name="hostBadB")
    xd, B, BS = dev_bf16(x), dev_e4m3(b), dev_f32(b_s)
    y, s = fp8bs.act_quant(xd)
    torch.cuda.synchronize()
    guard = torch.full((M * N + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda")
    short = guard[:M * N - 1].view(-1)                 # one element short of C
    with pytest.raises(ValueError):
        fp8bs.fp8_gemm(y, s, B, BS, out=short.view(1, -1))
    with pytest.raises(ValueError):
        fp8bs.fp8_gemm(y, s, B, BS, out=guard[:M * (N - 8)].view(M, N - 8))
    with pytest.raises(ValueError):
        fp8bs.linear_bf16(xd, B, BS, out=guard[:(M - 1) * N].view(M - 1, N))
    with pytest.raises(ValueError):
        fp8bs.act_quant_gemm(xd, B, BS, out=guard[:M * N].view(N, M))
    with pytest.raises(TypeError):
        fp8bs.fp8_gemm(y, s, B, BS, out=torch.empty((M, N), dtype=torch.float32, device="cuda"))
    with pytest.raises(TypeError):
        fp8bs.fp8_gemm(y, s, B, BS, out=torch.empty((M, N), dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        fp8bs.fp8_gemm(y, s, B, BS, workspace=torch.zeros(1 << 20, dtype=torch.uint8))
    torch.cuda.synchronize()
    assert bool(torch.isnan(guard.float()).all()), "a rejected call wrote to the buffer"
