"""Guard bands around every output buffer: each kernel must write every element of its output
and nothing outside it. compute-sanitizer is not available on this machine, and a full compare
against the oracle catches a wrong value inside an output but not a store past its end; TMA
boxes overhang ragged M and N, grouped tiles straddle groups, split and stream-K tiles are
stored by a CTA other than the one that computed them, and 16-byte stores sit at the N tail.

Each output is a view into a larger device buffer: the bytes before and after it are filled
with a sentinel (0xA5) and the output itself with 0xFF (a NaN in bf16, e4m3 and fp32). After
the call the sentinel must be intact and no NaN may be left in the output.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import dev_bf16, dev_e4m3, dev_f32

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side (a multiple of 256: the output stays aligned)
SENTINEL = 0xA5


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"


class Guarded:
    """An output tensor of `shape` and `dtype` inside a buffer with guard bands."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.buf[GUARD:GUARD + n] = 0xFF
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)

    def ptr(self):
        return self.t.data_ptr()

    def check(self, what):
        torch.cuda.synchronize()
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        assert bool((head == SENTINEL).all()), f"{what}: bytes written before the output"
        bad = (tail != SENTINEL).nonzero()
        assert bad.numel() == 0, f"{what}: {bad.numel()} bytes written after the output, " \
                                 f"first at +{int(bad[0])}"
        out = self.t
        if out.dtype == torch.float8_e4m3fn:
            unwritten = int(((out.view(torch.uint8) & 0x7F) == 0x7F).sum())
        else:
            unwritten = int(torch.isnan(out.float()).sum())
        assert unwritten == 0, f"{what}: {unwritten} output elements not written"


def st():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("M,K", [(3, 640), (129, 18432), (1000, 7168)])
def test_act_quant_guard_bands(M, K, fmt):
    x = dev_bf16(synth.activations(M, K, seed=M + K, name="guardA", outlier_frac=0.01))
    y, s = Guarded((M, K), torch.float8_e4m3fn), Guarded((M, K // 128), torch.float32)
    fp8bs.fp8bs_act_quant(x.data_ptr(), y.ptr(), s.ptr(), M, K, fmt, st())
    y.check(f"act_quant y {M}x{K}")
    s.check(f"act_quant s {M}x{K}")


@pytest.mark.parametrize("N,K", [(333, 391), (300, 272), (129, 7168), (5, 33)])
def test_weight_dequant_guard_bands(N, K):
    b, b_s = synth.weights(N, K, seed=N + K, name="guardW")
    y = Guarded((N, K), torch.bfloat16)
    B, S = dev_e4m3(b), dev_f32(b_s)
    fp8bs.fp8bs_weight_dequant(B.data_ptr(), S.data_ptr(), y.ptr(), N, K, st())
    y.check(f"weight_dequant {N}x{K}")


def gemm_inputs(M, N, K, fmt, seed):
    x = synth.activations(M, K, seed=seed, name="guardA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x, fmt)
    b, b_s = synth.weights(N, K, seed=seed + 1, name="guardB", pow2=fmt == 1)
    return dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s)


# Every schedule of every GEMM kernel, on ragged shapes: (M, N, K, scale_fmt, workspace).
GEMM_CASES = [
    (5, 200, 1024, 0, False),       # swapped, K split in a cluster
    (100, 130, 256, 0, False),      # swapped, one slab per CTA
    (64, 18432, 512, 0, False),     # swapped, every SM a slab
    (513, 97, 256, 0, False),       # promoted, 64-wide tiles
    (300, 1000, 2048, 0, False),    # promoted, split K
    (2560, 2304, 1024, 0, True),    # promoted, stream-K (192-wide tiles)
    (1100, 4736, 256, 0, False),    # promoted, 256-wide tiles
    (2600, 3900, 384, 1, False),    # block-scaled, 256-wide tiles, ragged both ways
    (2600, 4096, 384, 1, False),    # block-scaled, 256-wide tiles, stores through the scratch
    (2000, 1536, 640, 1, False),    # block-scaled, 192-wide tiles (two issuers), scratch stores
    (1100, 2500, 2048, 1, True),    # block-scaled, stream-K
    (512, 576, 7168, 1, False),     # block-scaled, 192-wide tiles, split K
    (2048, 1300, 640, 1, False),    # block-scaled, 192-wide whole tiles, N tail
    (300, 576, 128, 1, False),      # block-scaled, 64-wide tiles, two issuers
]


@pytest.mark.parametrize("M,N,K,fmt,with_ws", GEMM_CASES)
def test_gemm_guard_bands(M, N, K, fmt, with_ws):
    A, AS, B, BS = gemm_inputs(M, N, K, fmt, seed=M + N + K)
    c = Guarded((M, N), torch.bfloat16)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda") \
        if with_ws else None
    fp8bs.fp8bs_gemm_ws(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(), c.ptr(),
                        M, N, K, fmt, 0, ws.data_ptr() if ws is not None else 0,
                        ws.numel() if ws is not None else 0, st())
    c.check(f"gemm {M}x{N}x{K} fmt={fmt} workspace={with_ws}")


@pytest.mark.parametrize("fmt,counts,N", [
    (0, [0, 130, 5, 0, 257, 1], 384),
    (1, [0, 130, 5, 0, 257, 1], 384),
    (1, [600, 0, 700, 650, 100], 1536),      # 192-wide tiles, stores through the scratch
])
def test_grouped_gemm_guard_bands(fmt, counts, N):
    K = 256
    offs = np.r_[0, np.cumsum(counts)]
    T = int(offs[-1])
    A, AS, _, _ = gemm_inputs(T, N, K, fmt, seed=3)
    ws = [synth.weights(N, K, seed=10 + e, name="guardG", pow2=fmt == 1)
          for e in range(len(counts))]
    B = dev_e4m3(np.stack([w for w, _ in ws]))
    BS = dev_f32(np.stack([s for _, s in ws]))
    c = Guarded((T, N), torch.bfloat16)
    fp8bs.fp8bs_gemm_grouped(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(), c.ptr(),
                             offs, len(counts), N, K, fmt, st())
    c.check(f"grouped gemm fmt={fmt}")


@pytest.mark.parametrize("M,N,K,flags", [(17, 1000, 512, 2), (40, 2048, 7168, 3),
                                         (300, 1000, 512, 1),
                                         (13, 10000, 1024, 2),    # one kernel (M <= 16)
                                         (16, 18432, 2048, 3)])
def test_act_quant_gemm_guard_bands(M, N, K, flags):
    x = dev_bf16(synth.activations(M, K, seed=M, name="guardX", outlier_frac=0.01))
    b, b_s = synth.weights(N, K, seed=N, name="guardB")
    B, BS = dev_e4m3(b), dev_f32(b_s)
    y, s = Guarded((M, K), torch.float8_e4m3fn), Guarded((M, K // 128), torch.float32)
    c = Guarded((M, N), torch.bfloat16)
    fp8bs.fp8bs_act_quant_gemm(x.data_ptr(), y.ptr(), s.ptr(), B.data_ptr(), BS.data_ptr(),
                               c.ptr(), M, N, K, 0, flags, 0, 0, st())
    for g, what in ((y, "y"), (s, "s"), (c, "c")):
        g.check(f"act_quant_gemm {what} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (40, 128, 384), (200, 1000, 768),
                                   (1000, 640, 384)])
def test_linear_bf16_guard_bands(M, N, K):
    x = dev_bf16(synth.activations(M, K, seed=M + N, name="guardL"))
    w, w_s = synth.weights(N, K, seed=N + K, name="guardL")
    W, WS = dev_e4m3(w), dev_f32(w_s)
    y = Guarded((M, N), torch.bfloat16)
    fp8bs.fp8bs_linear_bf16(x.data_ptr(), W.data_ptr(), WS.data_ptr(), y.ptr(), M, N, K, 0, st())
    y.check(f"linear_bf16 {M}x{N}x{K}")
