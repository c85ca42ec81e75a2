"""fp8bs_gemm_noalloc (the stream-K GEMM on the library's static workspace) against
fp8bs_gemm_ws (the same GEMM on a caller workspace): two calls in a row on the same inputs
must both give the caller-workspace result bit for bit (the partials are added in a fixed
order, and the first call must leave the static workspace's counters at zero for the second).
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import assert_gemm_close, dev_e4m3, dev_f32, host_bf16_f64, lines_and_tiles

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"


@pytest.mark.parametrize("M,N,K,fmt", [
    (1100, 2500, 2048, fp8bs.SCALE_UE8M0),  # 180 tiles shared between neighbouring CTAs
    (2560, 2048, 2048, fp8bs.SCALE_UE8M0),  # 152 tiles computed whole, then 168 shared
    (2048, 1536, 7168, fp8bs.SCALE_UE8M0),  # the MLA q projection
    (2560, 2048, 2048, fp8bs.SCALE_FP32),   # fp32 scales: 220 tiles 192 wide, all shared
])
def test_noalloc_matches_caller_workspace_on_two_calls_in_a_row(M, N, K, fmt):
    ue8m0 = fmt == fp8bs.SCALE_UE8M0
    if not ue8m0:   # the fp32-scale shape shares tiles through the workspace
        assert fp8bs.fp8bs_gemm_plan(M, N, K, fmt, True)["stream_k"]
    x = synth.activations(M, K, seed=M + N, name="noallocA", outlier_frac=0.01)
    a, a_s = oracle.act_quant(x, oracle.SCALE_UE8M0 if ue8m0 else oracle.SCALE_FP32)
    b, b_s = synth.weights(N, K, seed=N + K, name="noallocB", pow2=ue8m0)
    A, AS, B, BS = dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream

    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8bs_gemm_ws(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(), ref.data_ptr(),
                        M, N, K, fmt, 0, ws.data_ptr(), ws.numel(), st)
    outs = []
    for _ in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        fp8bs.fp8bs_gemm_noalloc(A.data_ptr(), AS.data_ptr(), B.data_ptr(), BS.data_ptr(),
                                 c.data_ptr(), M, N, K, fmt, 0, st)
        outs.append(c)
    torch.cuda.synchronize()
    for i, c in enumerate(outs):
        assert torch.equal(c.view(torch.int16), ref.view(torch.int16)), f"call {i + 1} differs"
    mi, ni = lines_and_tiles(M, N, 1, seed=K)
    got = host_bf16_f64(outs[1])[mi, ni]
    assert_gemm_close(got, oracle.gemm_at(a, a_s, b, b_s, mi, ni), f"{M}x{N}x{K}",
                      c_full=outs[1])
