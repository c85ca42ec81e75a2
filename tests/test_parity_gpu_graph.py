"""Library calls captured in a CUDA graph and replayed with new inputs, against the oracle.

Every entry point takes a stream and launches with programmatic dependent launch, and the
stream-K schedule keeps counters in a caller's workspace that each call leaves at zero: a graph
of several calls (act_quant feeding a GEMM, GEMMs on each kernel and schedule, a grouped call)
must give the oracle's results on every replay, with the inputs rewritten between replays.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_fp8bs_gb300 as fp8bs
import oracle
import synth
from parity_util import assert_gemm_close, host_bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_device_error():
    fp8bs.fp8bs_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_error(clear=True) == 0, "a kernel wait ran out"


def u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def put(dev, host):
    """Rewrite a device buffer in place (its address stays the one the graph captured)."""
    dev.copy_(torch.from_numpy(np.ascontiguousarray(host)).view(dev.dtype).view(dev.shape))


GEMMS = [
    # M, N, K, scale format, workspace: the decode kernel with split K, the promotion kernel
    # with stream-K over the workspace, the block-scaled kernel
    (8, 2048, 2048, 0, False),
    (2560, 2048, 2048, 0, True),
    (600, 1000, 640, 1, False),
]
SAMPLED_ROWS = np.array([0, 1, 127, 128, 640, 1279, 1280, 1919, 2047, 2048, 2431, 2559])


def test_graph_replay_with_new_inputs_matches_oracle():
    assert fp8bs.fp8bs_gemm_plan(2560, 2048, 2048, fp8bs.SCALE_FP32, True)["stream_k"]
    st = torch.cuda.Stream()
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    # act_quant -> GEMM (decode orientation) on its output
    Mq, Nq, Kq = 16, 640, 1024
    xq = torch.zeros((Mq, Kq), dtype=torch.bfloat16, device="cuda")
    yq = torch.empty((Mq, Kq), dtype=torch.float8_e4m3fn, device="cuda")
    sq = torch.empty((Mq, Kq // 128), dtype=torch.float32, device="cuda")
    bq_codes, bq_s = synth.weights(Nq, Kq, seed=1, name="graphBq")
    Bq, BSq = u8(bq_codes).view(torch.float8_e4m3fn), u8(bq_s)
    cq = torch.empty((Mq, Nq), dtype=torch.bfloat16, device="cuda")
    # plain GEMMs
    bufs = []
    for (M, N, K, fmt, with_ws) in GEMMS:
        b, b_s = synth.weights(N, K, seed=N + K, name="graphB", pow2=fmt == 1)
        bufs.append(dict(M=M, N=N, K=K, fmt=fmt, ws=with_ws, b=b, b_s=b_s,
                         A=torch.zeros((M, K), dtype=torch.uint8, device="cuda"),
                         AS=torch.ones((M, K // 128), dtype=torch.float32, device="cuda"),
                         B=u8(b), BS=u8(b_s),
                         C=torch.empty((M, N), dtype=torch.bfloat16, device="cuda")))
    # grouped: one large group, two small ones (both of its launches)
    counts = [200, 5, 0, 40]
    offs = np.r_[0, np.cumsum(counts)]
    T, Ng, Kg = int(offs[-1]), 384, 512
    wg = [synth.weights(Ng, Kg, seed=30 + e, name="graphG") for e in range(len(counts))]
    Ag = torch.zeros((T, Kg), dtype=torch.uint8, device="cuda")
    ASg = torch.ones((T, Kg // 128), dtype=torch.float32, device="cuda")
    Bg = u8(np.stack([w for w, _ in wg]))
    BSg = u8(np.stack([s for _, s in wg]))
    Cg = torch.empty((T, Ng), dtype=torch.bfloat16, device="cuda")

    def calls(stream):
        h = stream.cuda_stream
        fp8bs.fp8bs_act_quant(xq.data_ptr(), yq.data_ptr(), sq.data_ptr(), Mq, Kq, 0, h)
        fp8bs.fp8bs_gemm(yq.data_ptr(), sq.data_ptr(), Bq.data_ptr(), BSq.data_ptr(),
                         cq.data_ptr(), Mq, Nq, Kq, 0, h)
        for d in bufs:
            fp8bs.fp8bs_gemm_ws(d["A"].data_ptr(), d["AS"].data_ptr(), d["B"].data_ptr(),
                                d["BS"].data_ptr(), d["C"].data_ptr(), d["M"], d["N"], d["K"],
                                d["fmt"], 0, ws.data_ptr() if d["ws"] else 0,
                                ws.numel() if d["ws"] else 0, h)
        fp8bs.fp8bs_gemm_grouped(Ag.data_ptr(), ASg.data_ptr(), Bg.data_ptr(), BSg.data_ptr(),
                                 Cg.data_ptr(), offs, len(counts), Ng, Kg, 0, h)

    with torch.cuda.stream(st):
        calls(st)                       # eager first: kernel attributes set, plans cached
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        calls(st)
    torch.cuda.synchronize()

    for r in range(2):
        xh = synth.activations(Mq, Kq, seed=100 + r, name="graphX", outlier_frac=0.01)
        put(xq, xh.view(np.int16))
        refs = []
        for d in bufs:
            x = synth.activations(d["M"], d["K"], seed=200 + r + d["M"], name="graphA",
                                  outlier_frac=0.01)
            a, a_s = oracle.act_quant(x, d["fmt"])
            put(d["A"], a)
            put(d["AS"], a_s)
            refs.append((a, a_s))
        xg = synth.activations(T, Kg, seed=300 + r, name="graphAg", outlier_frac=0.01)
        ag, ag_s = oracle.act_quant(xg, oracle.SCALE_FP32)
        put(Ag, ag)
        put(ASg, ag_s)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()

        yq_ref, sq_ref = oracle.act_quant(xh, oracle.SCALE_FP32)
        assert np.array_equal(yq.view(torch.uint8).cpu().numpy(), yq_ref), f"replay {r}: codes"
        assert_gemm_close(host_bf16_f64(cq), oracle.gemm(yq_ref, sq_ref, bq_codes, bq_s),
                          f"replay {r}: act_quant -> gemm")
        for d, (a, a_s) in zip(bufs, refs):
            c_dev, what = d["C"], f"replay {r}: gemm {d['M']}x{d['N']}x{d['K']} fmt {d['fmt']}"
            if d["M"] >= 2048:      # rows in every row tile, whole-matrix rms from the output
                rows = SAMPLED_ROWS
                assert_gemm_close(host_bf16_f64(c_dev)[rows],
                                  oracle.gemm(a[rows], a_s[rows], d["b"], d["b_s"]), what,
                                  c_full=c_dev)
            else:
                assert_gemm_close(host_bf16_f64(c_dev), oracle.gemm(a, a_s, d["b"], d["b_s"]),
                                  what)
        c = host_bf16_f64(Cg)
        for e in range(len(counts)):
            lo, hi = offs[e], offs[e + 1]
            if hi > lo:
                assert_gemm_close(c[lo:hi], oracle.gemm(ag[lo:hi], ag_s[lo:hi], *wg[e]),
                                  f"replay {r}: grouped group {e}")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert bool((ws[:4 * sms] == 0).all()), "stream-K counters not back at zero after the replays"
