"""Benchmark of the FP8 block-scaled linear path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}] [--quick]

Headline workload (one JSON line on rank 0): the decode configuration -- for each
M in {1, 8, 32, 64}: act_quant of a bf16 [M, 7168] activation, then fp8_gemm against an e4m3
[18432, 7168] weight with 128x128 fp32 block scales. One step runs the four (act_quant, gemm)
pairs; each M uses its own weight matrix, so a step streams 4 x 132 MB of weights and no
weight is resident in L2 (129 MB) when it is read again. The timed steps replay CUDA graphs of
ten steps each (the same launches; the steps launched one by one are timed too and reported as
eager_ms_per_step). The metric is algorithmic bytes moved per second (GB/s): weights, weight
scales, activations, codes, scales and outputs.

Also reported (rank 0, N=1): prefill GEMM TFLOPS, weight_dequant / act_quant GB/s, the MoE
expert GEMMs and the ue8m0 MLA projections, each against its roofline; the CPU oracle on a
bounded sample of the decode workload (cpu_baseline); clocks sampled during the timed region.

--impl reference times the CPU oracle instead (the pages publish no runnable reference), on a
bounded sample of the same workload, and prints the same metric with "impl": "reference".

Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas; the path
has no exchange step): weak scaling, value = bytes of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("fp8_gemm TFLOPS & % FP8 peak (prefill M); GB/s & % HBM (quant, decode M)")
K_DIM, N_DIM = synth.DIM, synth.INTER
DECODE_MS = synth.DECODE_MS
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 vs 2.25 PFLOP/s)

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the decode GEMM
# kernel (gemm_swapab_kernel), from ncu captures of its M=1 and M=64 launches (their mean),
# valid only for the kernel sources they were taken on (DECODE_KERNEL_SOURCES, first 16 hex
# digits of their SHA-256); for any other source the bench reports traffic as null.
DECODE_TRAFFIC_MB = {"kernel_sha": "ef1125afebf8d989", "per_launch_mb": (134.93 + 135.32) / 2}


# ----------------------------------------------------------------------------- accounting

def act_quant_bytes(M, K):
    """read bf16 x, write e4m3 y and fp32 scales."""
    return 2 * M * K + M * K + 4 * M * (K // 128)


def gemm_bytes(M, N, K):
    """read A codes + a_s, B codes + b_s once, write bf16 C."""
    return M * K + 4 * M * (K // 128) + N * K + 4 * (-(-N // 128)) * (K // 128) + 2 * M * N


def dequant_bytes(N, K):
    return N * K + 4 * (-(-N // 128)) * (-(-K // 128)) + 2 * N * K


def linear_bf16_bytes(M, N, K):
    """bf16 path: x bf16 + the e4m3 weight and its block scales + y bf16."""
    return 2 * M * K + N * K + 4 * (-(-N // 128)) * (K // 128) + 2 * M * N


def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def decode_step_bytes():
    return sum(act_quant_bytes(M, K_DIM) + gemm_bytes(M, N_DIM, K_DIM) for M in DECODE_MS)


DECODE_KERNEL_SOURCES = ("gemm_swapab.cu", "gemm_common.cuh", "quant_math.cuh", "ptx.cuh",
                         "kernels.h")


def decode_kernel_sha():
    """Hash of the sources the decode GEMM kernel is compiled from."""
    import hashlib
    h = hashlib.sha256()
    try:
        for f in DECODE_KERNEL_SOURCES:
            h.update(open(os.path.join(ROOT, "fp8_block_scaled_fp8bs_gb300", "csrc", f), "rb").read())
    except OSError:
        return None
    return h.hexdigest()[:16]


def decode_traffic():
    """Measured DRAM bytes per decode-GEMM launch, if the kernel's sources are unchanged."""
    sha = decode_kernel_sha()
    if sha is None or sha != DECODE_TRAFFIC_MB["kernel_sha"]:
        return None
    return round(DECODE_TRAFFIC_MB["per_launch_mb"] * 1e6)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path: str | None = None):
        self.index = index
        self.path = path
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
            if self.path:
                with open(self.path, "w") as fh:
                    fh.write(self.QUERY + "\n" + "\n".join(self.lines) + "\n")
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

class Gpu:
    def __init__(self):
        import torch
        import fp8_block_scaled_fp8bs_gb300 as fp8bs
        self.torch = torch
        self.fp8bs = fp8bs
        fp8bs.load()
        self.stream = torch.cuda.current_stream()
        self.sh = self.stream.cuda_stream
        self._flush_buf = None
        self._ws = None

    def bf16(self, bits):
        return self.torch.from_numpy(np.ascontiguousarray(bits)).view(self.torch.bfloat16).cuda()

    def e4m3(self, codes):
        return self.torch.from_numpy(np.ascontiguousarray(codes)).view(
            self.torch.float8_e4m3fn).cuda()

    def f32(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()

    def flush_l2(self):
        """Evict L2 by reading 256 MB: the cache then holds clean lines, so the next kernel
        pays no write-back of the flush (a write-based flush would leave ~129 MB dirty)."""
        if self._flush_buf is None:
            self._flush_buf = self.torch.ones(32 * 1024 * 1024, dtype=self.torch.int64,
                                              device="cuda")
        self._flush_buf.sum()

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)

    # raw C-ABI calls on the benchmark stream
    def act_quant(self, x, y, s, M, K, fmt=0):
        self.fp8bs.fp8bs_act_quant(x.data_ptr(), y.data_ptr(), s.data_ptr(), M, K, fmt, self.sh)

    def gemm(self, a, a_s, b, b_s, c, M, N, K, fmt=0):
        self.fp8bs.fp8bs_gemm(a.data_ptr(), a_s.data_ptr(), b.data_ptr(), b_s.data_ptr(),
                              c.data_ptr(), M, N, K, fmt, self.sh)

    def gemm_ex(self, a, a_s, b, b_s, c, M, N, K, fmt=0, flags=0):
        self.fp8bs.fp8bs_gemm_ex(a.data_ptr(), a_s.data_ptr(), b.data_ptr(), b_s.data_ptr(),
                                 c.data_ptr(), M, N, K, fmt, flags, self.sh)

    def workspace(self):
        if self._ws is None:
            self._ws = self.torch.zeros(self.fp8bs.fp8bs_gemm_workspace_size(),
                                        dtype=self.torch.uint8, device="cuda")
        return self._ws

    def act_quant_gemm(self, x, y, s, b, b_s, c, M, N, K, fmt=0, flags=0):
        """act_quant + fp8_gemm through fp8bs_act_quant_gemm: two launches (the GEMM starting
        under act_quant), or one with FP8BS_GEMM_QUANT_IN_KERNEL in flags."""
        ws = self.workspace()
        self.fp8bs.fp8bs_act_quant_gemm(x.data_ptr(), y.data_ptr(), s.data_ptr(), b.data_ptr(),
                                        b_s.data_ptr(), c.data_ptr(), M, N, K, fmt, flags,
                                        ws.data_ptr(), ws.numel(), self.sh)

    def gemm_ws(self, a, a_s, b, b_s, c, M, N, K, fmt=0):
        """fp8bs_gemm_ws with the benchmark's workspace (stream-K where it pays)."""
        self.workspace()
        self.fp8bs.fp8bs_gemm_ws(a.data_ptr(), a_s.data_ptr(), b.data_ptr(), b_s.data_ptr(),
                                 c.data_ptr(), M, N, K, fmt, 0, self._ws.data_ptr(),
                                 self._ws.numel(), self.sh)

    def dequant(self, w, s, y, N, K):
        self.fp8bs.fp8bs_weight_dequant(w.data_ptr(), s.data_ptr(), y.data_ptr(), N, K, self.sh)

    def linear_bf16(self, x, w, s, y, M, N, K, flags=0):
        self.fp8bs.fp8bs_linear_bf16(x.data_ptr(), w.data_ptr(), s.data_ptr(), y.data_ptr(), M, N,
                                     K, flags, self.sh)

    def time_cycle(self, fn, items, rounds):
        """Average device time (ms) of one fn(item) launch: `rounds` passes over `items`, all
        launched back to back as one region between two events on the benchmark stream (behind
        a GPU sleep, so that no launch waits on the host)."""
        torch = self.torch
        for it in items:
            fn(it)
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e6 + rounds * len(items) * 1e5))
        t0, t1 = self.event(), self.event()
        t0.record()
        for _ in range(rounds):
            for it in items:
                fn(it)
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / (rounds * len(items))

    def time_each(self, fn, reps, flush=True):
        """Device time (ms) of one fn() launch with a cold L2: `reps` launches back to back,
        each after an L2 flush, timed as one region between two events, minus a region of the
        flushes alone. (An event pair around every single launch would add the GPU's launch
        latency, ~5 us here, to each sample.) Everything is enqueued behind a GPU sleep so that
        no launch waits on the host."""
        torch = self.torch
        e = [self.event() for _ in range(3)]
        fn()
        if flush:
            self.flush_l2()          # allocates the flush buffer outside the timed region
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e6 + reps * 2e5))       # ~1 ms + 0.1 ms per launch at 2 GHz
        e[0].record()
        for _ in range(reps):
            if flush:
                self.flush_l2()
            fn()
        e[1].record()
        if flush:
            for _ in range(reps):
                self.flush_l2()
        e[2].record()
        torch.cuda.synchronize()
        return (e[0].elapsed_time(e[1]) - e[1].elapsed_time(e[2])) / reps


def copy_of_bytes(g: Gpu, total_bytes):
    """A device-to-device copy that reads and writes total_bytes / 2 each (the same bytes in
    total as the kernel it stands beside)."""
    n = total_bytes // 2 // 16 * 16
    src = g.torch.empty(n, dtype=g.torch.uint8, device="cuda")
    dst = g.torch.empty(n, dtype=g.torch.uint8, device="cuda")
    return lambda: dst.copy_(src)


def decode_setup(g: Gpu, seed=0):
    torch = g.torch
    b_codes, b_s = synth.weights(N_DIM, K_DIM, seed, "decode/B")
    B0, S0 = g.e4m3(b_codes), g.f32(b_s)
    del b_codes
    state = []
    for i, M in enumerate(DECODE_MS):
        # one distinct weight matrix per M (a perturbed copy of the first: same distribution)
        B = B0 if i == 0 else torch.roll(B0.view(torch.uint8), shifts=i * 4096, dims=0) \
            .contiguous().view(torch.float8_e4m3fn)
        S = S0 if i == 0 else torch.roll(S0, shifts=i * 32, dims=0).contiguous()
        x = g.bf16(synth.decode(M, seed))
        state.append(dict(M=M, x=x, B=B, S=S,
                          y=torch.empty((M, K_DIM), dtype=torch.float8_e4m3fn, device="cuda"),
                          s=torch.empty((M, K_DIM // 128), dtype=torch.float32, device="cuda"),
                          c=torch.empty((M, N_DIM), dtype=torch.bfloat16, device="cuda")))
    return state


WEIGHTS_CONSTANT = 1   # fp8bs_gemm_ex flag: model weights are not written during the step


def decode_step(g: Gpu, state):
    """act_quant + fp8_gemm for every M, back to back, through fp8bs_act_quant_gemm (two
    kernels per M): each kernel may start while the previous one finishes (the GEMM starts its
    weight stream early)."""
    for st in state:
        g.act_quant_gemm(st["x"], st["y"], st["s"], st["B"], st["S"], st["c"], st["M"], N_DIM,
                         K_DIM, 0, WEIGHTS_CONSTANT)


GRAPH_STEPS = 10   # decode steps per captured CUDA graph


def capture_steps(g: Gpu, state, n):
    """A CUDA graph of n decode steps, captured on a side stream (the launches keep their
    programmatic-dependent-launch attributes inside the graph)."""
    torch = g.torch
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    main_stream, main_sh = g.stream, g.sh
    g.stream, g.sh = side, side.cuda_stream
    try:
        with torch.cuda.stream(side):
            decode_step(g, state)                   # kernel attributes set outside the capture
            side.synchronize()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(n):
                    decode_step(g, state)
    finally:
        g.stream, g.sh = main_stream, main_sh
    torch.cuda.synchronize()
    return graph


def run_decode(g: Gpu, steps, warmup, rank, world, clocks_path):
    """The timed decode steps, replayed from CUDA graphs of GRAPH_STEPS steps (plus one graph for
    the remainder): exactly `steps` steps, the same launches as decode_step, without the host's
    launch overhead between them -- the way a serving loop runs decode. Also returns the same
    number of steps launched one by one (eager), for comparison."""
    torch = g.torch
    state = decode_setup(g)
    for _ in range(warmup):
        decode_step(g, state)
    torch.cuda.synchronize()
    full, rest = divmod(steps, GRAPH_STEPS)
    graph = capture_steps(g, state, GRAPH_STEPS) if full else None
    tail = capture_steps(g, state, rest) if rest else None
    for _ in range(2):
        if graph is not None:
            graph.replay()
        if tail is not None:
            tail.replay()
    torch.cuda.synchronize()
    # eager, for comparison (not the reported value)
    e0, e1 = g.event(), g.event()
    e0.record()
    for _ in range(steps):
        decode_step(g, state)
    e1.record()
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1)
    sampler = ClockSampler(torch.cuda.current_device(), clocks_path)
    with sampler:
        time.sleep(0.25)
        barrier(world)
        torch.cuda.synchronize()
        t0, t1 = g.event(), g.event()
        t0.record()
        for _ in range(full):
            graph.replay()
        if tail is not None:
            tail.replay()
        t1.record()
        torch.cuda.synchronize()
        barrier(world)
        time.sleep(0.25)
    ms_total = t0.elapsed_time(t1)
    return (ms_total, eager_ms, decode_gemm_launch_ms(g, state, max(3, min(steps, 100))),
            sampler.summary())


def decode_gemm_launch_ms(g: Gpu, state, rounds):
    """Average duration of one decode-GEMM launch per M: `rounds` x 4 launches back to back,
    cycling through the four distinct 132 MB weights (so that no launch finds its weight in
    L2), timed as one region between two events on the launching stream."""
    torch = g.torch
    per_m = []
    for st in state:
        M = st["M"]

        def launch(w):
            g.gemm_ex(st["y"], st["s"], w["B"], w["S"], st["c"], M, N_DIM, K_DIM, 0,
                      WEIGHTS_CONSTANT)
        for w in state:
            launch(w)
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e6 + rounds * 4e5))
        t0, t1 = g.event(), g.event()
        t0.record()
        for _ in range(rounds):
            for w in state:
                launch(w)
        t1.record()
        torch.cuda.synchronize()
        per_m.append((M, t0.elapsed_time(t1) / (rounds * len(state))))
    return per_m


def run_decode_e2e(g: Gpu, steps, warmup, world):
    """The same step through the C ABI with host buffers: every step moves its activations from
    pinned host memory to the GPU and its outputs back, and steps stay ordered (a step starts
    only once the previous step's outputs are on the host, as when the next input depends on
    them). On GB300 the GPU reaches pinned host memory over NVLink-C2C, so the host buffers are
    used in place where that is cheapest:
      - act_quant reads each activation straight from pinned host memory (the same bytes cross
        the link as with a copy, without a copy's fixed cost of ~6 us and its wait);
      - the GEMMs of the problems with small outputs (M <= E2E_DIRECT_MAX_M) write C straight
        into pinned host memory;
      - the larger outputs go out by copy on a second stream while the next problems compute.
    The problems run largest first, so the outputs written in place come last. Measured on one
    box: 126.2 us per step with one packed input copy and four output copies, 119.3 us with the
    activations read in place, 108.5 us with the two small outputs also written in place; with
    every output written in place 121.0 us (a 2.4 MB output written over the link holds its
    GEMM's tail)."""
    torch = g.torch
    state = decode_setup(g, seed=1)
    n = len(state)
    order = sorted(range(n), key=lambda i: -state[i]["M"])
    direct = [i for i in order if state[i]["M"] <= E2E_DIRECT_MAX_M]
    copied = [i for i in order if i not in direct]
    hx = [state[i]["x"].cpu().pin_memory() for i in range(n)]
    hc = [torch.empty(st["c"].shape, dtype=torch.bfloat16).pin_memory() for st in state]
    comp = g.stream
    copy = torch.cuda.Stream()
    c_done = [torch.cuda.Event() for _ in range(n)]      # c_i is computed
    c_out = [torch.cuda.Event() for _ in range(n)]       # c_i is on the host
    for i in range(n):
        c_out[i].record(comp)

    def step():
        for i in copied:
            comp.wait_event(c_out[i])     # the previous step's outputs are on the host
        for i in order:
            st = state[i]
            g.act_quant_gemm(hx[i], st["y"], st["s"], st["B"], st["S"],
                             hc[i] if i in direct else st["c"], st["M"], N_DIM, K_DIM, 0,
                             WEIGHTS_CONSTANT)
            if i in direct:
                c_out[i].record(comp)
            else:
                c_done[i].record(comp)
        with torch.cuda.stream(copy):
            for i in copied:
                copy.wait_event(c_done[i])
                hc[i].copy_(state[i]["c"], non_blocking=True)
                c_out[i].record(copy)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = g.event(), g.event()
    t0.record(comp)
    for _ in range(steps):
        step()
    for i in range(n):
        comp.wait_event(c_out[i])     # the region ends with the last outputs on the host
    t1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    h2d = sum(2 * st["M"] * K_DIM for st in state)
    d2h = sum(2 * st["M"] * N_DIM for st in state)
    return t0.elapsed_time(t1), h2d, d2h


E2E_DIRECT_MAX_M = 8   # decode problems whose output the GEMM writes into host memory in place


def secondary(g: Gpu, peaks, reps=20):
    """Other workloads of the path, each kernel timed alone with L2 flushed before every
    launch; reported against its roofline."""
    torch = g.torch
    out = {}
    hbm = peaks["hbm_gbs"]
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16

    def gemm_entry(name, M, N, K, fmt, x_bits, b_codes, b_s):
        x = g.bf16(x_bits)
        y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
        g.act_quant(x, y, s, M, K, fmt)
        B, S = g.e4m3(b_codes), g.f32(b_s)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            g.gemm_ws(y, s, B, S, c, M, N, K, fmt)
        ms = g.time_each(lambda: g.gemm_ws(y, s, B, S, c, M, N, K, fmt), reps)
        tf = gemm_flops(M, N, K) / ms / 1e9
        gb = gemm_bytes(M, N, K) / ms / 1e6
        bound_ms = max(gemm_flops(M, N, K) / (fp8_peak * 1e9), gemm_bytes(M, N, K) / (hbm * 1e6))
        out[name] = {"M": M, "N": N, "K": K, "us": round(ms * 1e3, 2), "TFLOP/s": round(tf, 1),
                     "GB/s": round(gb, 1), "frac_fp8_peak": round(tf / fp8_peak, 4),
                     "frac_roofline": round(bound_ms / ms, 4)}
        del x, y, s, B, S, c

    xb = synth.prefill_up()
    bc, bs = synth.weights(N_DIM, K_DIM, 0, "prefill/B_up")
    gemm_entry("prefill_up", 4096, N_DIM, K_DIM, 0, xb, bc, bs)
    # weight_dequant of the same [18432, 7168] matrix
    W, WS = g.e4m3(bc), g.f32(bs)
    Y = torch.empty((N_DIM, K_DIM), dtype=torch.bfloat16, device="cuda")
    ms = g.time_each(lambda: g.dequant(W, WS, Y, N_DIM, K_DIM), reps)
    gbs = dequant_bytes(N_DIM, K_DIM) / ms / 1e6
    out["weight_dequant"] = {"N": N_DIM, "K": K_DIM, "us": round(ms * 1e3, 2),
                             "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}
    del Y
    # the bf16 path (weight dequantised on chip inside the GEMM) on the same weight: decode rows
    # against HBM, the prefill rows against the bf16 tensor peak
    bf16_peak = peaks["bf16_tflops"]
    for M, bits in ((1, synth.decode(1)), (64, synth.decode(64)), (4096, synth.prefill_up())):
        x = g.bf16(bits)
        y = torch.empty((M, N_DIM), dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            g.linear_bf16(x, W, WS, y, M, N_DIM, K_DIM)
        ms = g.time_each(lambda: g.linear_bf16(x, W, WS, y, M, N_DIM, K_DIM), reps)
        gbs = linear_bf16_bytes(M, N_DIM, K_DIM) / ms / 1e6
        tf = 2 * M * N_DIM * K_DIM / ms / 1e9
        out[f"linear_bf16_M{M}"] = {"M": M, "N": N_DIM, "K": K_DIM, "us": round(ms * 1e3, 2),
                                    "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                                    "TFLOP/s": round(tf, 1),
                                    "frac_bf16_peak": round(tf / bf16_peak, 4)}
        del x, y
    del W, WS, bc
    xb = synth.prefill_down()
    bc, bs = synth.weights(K_DIM, N_DIM, 0, "prefill/B_down")
    gemm_entry("prefill_down", 4096, K_DIM, N_DIM, 0, xb, bc, bs)
    del bc

    # act_quant at large row counts (MoE gathered rows; ue8m0 MLA input)
    for name, M, K, fmt, bits in (("act_quant_moe", 8192, K_DIM, 0, None),
                                  ("act_quant_mla_ue8m0", 2048, K_DIM, 1, synth.mla_acts()),
                                  ("act_quant_prefill_up", 4096, K_DIM, 0, synth.prefill_up()),
                                  ("act_quant_prefill_down", 4096, N_DIM, 0, synth.prefill_down())):
        if bits is None:
            rows, _ = synth.moe_routing(0)
            bits = synth.activations(1024, K_DIM, 0, "moe/tokens", outlier_frac=0.01)[rows]
        x = g.bf16(bits)
        y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
        ms = g.time_each(lambda: g.act_quant(x, y, s, M, K, fmt), reps)
        gbs = act_quant_bytes(M, K) / ms / 1e6
        # A device copy moving the same number of bytes (half read, half written), timed the
        # same way: what any kernel moving these bytes achieves at this size.
        copy_ms = g.time_each(copy_of_bytes(g, act_quant_bytes(M, K)), reps)
        # The same launches back to back, as in a model step where act_quant follows another
        # kernel (its launch and the memory system's ramp overlap the previous launch), over
        # distinct inputs and outputs that together exceed L2, so none is found in L2.
        n_in = max(4, -(-300_000_000 // act_quant_bytes(M, K)))
        xs = [x] + [torch.roll(x, shifts=64 * i, dims=0) for i in range(1, n_in)]
        ys = [y] + [torch.empty_like(y) for _ in range(1, n_in)]
        ss = [s] + [torch.empty_like(s) for _ in range(1, n_in)]
        b2b_ms = g.time_cycle(lambda i: g.act_quant(xs[i], ys[i], ss[i], M, K, fmt),
                              list(range(n_in)), max(3, 200 // n_in))
        b2b_gbs = act_quant_bytes(M, K) / b2b_ms / 1e6
        out[name] = {"M": M, "K": K, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / hbm, 4), "copy_us": round(copy_ms * 1e3, 2),
                     "frac_of_copy": round(copy_ms / ms, 4),
                     "back_to_back": {"inputs": n_in, "us": round(b2b_ms * 1e3, 2),
                                      "GB/s": round(b2b_gbs, 1),
                                      "frac_hbm": round(b2b_gbs / hbm, 4)}}
        del x, y, s, xs, ys, ss

    # act_quant at the decode sizes: one row block per M, each launch timed alone (cold L2)
    for M in DECODE_MS:
        x = g.bf16(synth.decode(M))
        y = torch.empty((M, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K_DIM // 128), dtype=torch.float32, device="cuda")
        ms = g.time_each(lambda: g.act_quant(x, y, s, M, K_DIM, 0), reps)
        out[f"act_quant_decode_M{M}"] = {"M": M, "K": K_DIM, "us": round(ms * 1e3, 2),
                                         "GB/s": round(act_quant_bytes(M, K_DIM) / ms / 1e6, 1)}
        del x, y, s

    # decode GEMMs with few weight slabs (each slab's K loop split between the CTAs of a
    # cluster): the MLP down-projection (N=7168, K=18432; four distinct 132 MB weights) and one
    # MoE expert's up-projection (N=2048, K=7168; 32 distinct 14.7 MB weights). Launches cycle
    # through the weights back to back, so no weight is in L2 when it is read again.
    for name, N, K, n_w in (("decode_down_N7168_K18432", K_DIM, N_DIM, 4),
                            ("decode_expert_N2048_K7168", synth.MOE_INTER, K_DIM, 32)):
        b0, bs0 = synth.weights(N, K, 0, f"decode/{name}")
        B0, S0 = g.e4m3(b0), g.f32(bs0)
        del b0
        ws = [(B0, S0)] + [
            (torch.roll(B0.view(torch.uint8), shifts=i * 8, dims=0).contiguous()
             .view(torch.float8_e4m3fn), torch.roll(S0, shifts=i, dims=0).contiguous())
            for i in range(1, n_w)]
        per_m = []
        for M in DECODE_MS:
            x = g.bf16(synth.activations(M, K, 0, f"decode/{name}/x", outlier_frac=0.01))
            y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
            s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
            c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            g.act_quant(x, y, s, M, K)
            plan = g.fp8bs.fp8bs_gemm_plan(M, N, K, 0, False)
            ms = g.time_cycle(lambda w: g.gemm_ex(y, s, w[0], w[1], c, M, N, K, 0,
                                                  WEIGHTS_CONSTANT), ws, max(3, 400 // n_w))
            gbs = gemm_bytes(M, N, K) / ms / 1e6
            per_m.append({"M": M, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                          "frac_hbm": round(gbs / hbm, 4), "ksplit": plan["ksplit"]})
            del x, y, s, c
        out[name] = {"N": N, "K": K, "weights": n_w, "per_M": per_m}
        del ws, B0, S0

    # the decode step's four GEMMs (M = 1, 8, 32, 64 against four distinct 132 MB weights) as
    # one grouped launch in the swapped orientation, after the four act_quant launches
    st4 = decode_setup(g)
    B4 = torch.stack([st["B"] for st in st4]).contiguous()
    S4 = torch.stack([st["S"] for st in st4]).contiguous()
    Ms = [st["M"] for st in st4]
    offs4 = np.r_[0, np.cumsum(Ms)]
    x4 = torch.cat([st["x"] for st in st4]).contiguous()
    y4 = torch.empty((int(offs4[-1]), K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
    s4 = torch.empty((int(offs4[-1]), K_DIM // 128), dtype=torch.float32, device="cuda")
    c4 = torch.empty((int(offs4[-1]), N_DIM), dtype=torch.bfloat16, device="cuda")

    def step_grouped():
        for i, st in enumerate(st4):
            lo, hi = int(offs4[i]), int(offs4[i + 1])
            g.act_quant(x4[lo:hi], y4[lo:hi], s4[lo:hi], hi - lo, K_DIM)
        g.fp8bs.fp8bs_gemm_grouped(y4.data_ptr(), s4.data_ptr(), B4.data_ptr(), S4.data_ptr(),
                                   c4.data_ptr(), offs4, 4, N_DIM, K_DIM, 0, g.sh)
    for _ in range(3):
        step_grouped()
    ms = g.time_cycle(lambda _: step_grouped(), [0], 50)
    gbs = decode_step_bytes() / ms / 1e6
    out["decode_step_grouped"] = {"M": Ms, "N": N_DIM, "K": K_DIM, "us": round(ms * 1e3, 2),
                                  "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                                  "launches": len(Ms) + 1}
    del B4, S4, st4, x4, y4, s4, c4

    # ue8m0 MLA projections (block-scaled MMA: the tensor cores apply the power-of-two scales)
    xa = synth.mla_acts()
    for N in (synth.Q_LORA, synth.KV_LORA_ROPE):
        bc, bs = synth.weights(N, K_DIM, 0, f"mla/B{N}", pow2=True)
        gemm_entry(f"mla_ue8m0_N{N}", 2048, N, K_DIM, 1, xa, bc, bs)
    # the prefill up-projection shape with ue8m0 scales, on the same block-scaled kernel
    bc, bs = synth.weights(N_DIM, K_DIM, 0, "prefill/B_up", pow2=True)
    gemm_entry("prefill_up_ue8m0", 4096, N_DIM, K_DIM, 1, synth.prefill_up(), bc, bs)
    del bc

    # MoE: 32 expert GEMMs back to back on one stream, timed as a group
    rows, counts = synth.moe_routing(0)
    tokens = synth.activations(1024, K_DIM, 0, "moe/tokens", outlier_frac=0.01)
    x = g.bf16(tokens[rows])
    y = torch.empty((8192, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
    s = torch.empty((8192, K_DIM // 128), dtype=torch.float32, device="cuda")
    g.act_quant(x, y, s, 8192, K_DIM)
    Bs = []
    for e in range(32):
        bc, bs = synth.weights(synth.MOE_INTER, K_DIM, 0, f"moe/B{e}")
        Bs.append((g.e4m3(bc), g.f32(bs)))
    Bstack = torch.stack([w for w, _ in Bs]).contiguous()
    Sstack = torch.stack([sc for _, sc in Bs]).contiguous()
    offs = np.r_[0, np.cumsum(counts)]
    cs = [torch.empty((int(counts[e]), synth.MOE_INTER), dtype=torch.bfloat16, device="cuda")
          for e in range(32)]

    def moe():
        for e in range(32):
            lo, hi = int(offs[e]), int(offs[e + 1])
            if hi > lo:
                g.gemm(y[lo:hi], s[lo:hi], Bs[e][0], Bs[e][1], cs[e], hi - lo,
                       synth.MOE_INTER, K_DIM)
    c_all = torch.empty((8192, synth.MOE_INTER), dtype=torch.bfloat16, device="cuda")

    def moe_grouped():
        g.fp8bs.fp8bs_gemm_grouped(y.data_ptr(), s.data_ptr(), Bstack.data_ptr(),
                                   Sstack.data_ptr(), c_all.data_ptr(), offs, 32,
                                   synth.MOE_INTER, K_DIM, 0, g.sh)
    flops = sum(gemm_flops(int(m), synth.MOE_INTER, K_DIM) for m in counts)
    # one launch: max(total FLOPs / peak, total bytes / bandwidth)
    total_bytes = sum(gemm_bytes(int(m), synth.MOE_INTER, K_DIM) for m in counts if m > 0)
    bound = max(flops / (fp8_peak * 1e9), total_bytes / (hbm * 1e6))
    # The per-expert loop captured once in a CUDA graph (the host's per-call work, argument
    # checks and tensor maps, is then paid at capture, not per replay).
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()

    def moe_on(stream_handle):
        for e in range(32):
            lo, hi = int(offs[e]), int(offs[e + 1])
            if hi > lo:
                g.fp8bs.fp8bs_gemm(y[lo:hi].data_ptr(), s[lo:hi].data_ptr(), Bs[e][0].data_ptr(),
                                   Bs[e][1].data_ptr(), cs[e].data_ptr(), hi - lo,
                                   synth.MOE_INTER, K_DIM, 0, stream_handle)
    variants = [("moe_32_experts_grouped", moe_grouped), ("moe_32_experts_loop", moe)]
    try:
        with torch.cuda.stream(cap):
            moe_on(cap.cuda_stream)                   # warm-up: one-time kernel attributes
        cap.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            moe_on(cap.cuda_stream)
        variants.append(("moe_32_experts_loop_graph", graph.replay))
    except RuntimeError as err:                       # reported, not fatal to the benchmark
        out["moe_32_experts_loop_graph"] = {"unavailable": str(err).splitlines()[0][:200]}

    for name, fn in variants:
        fn()
        ms = g.time_each(fn, reps)
        out[name] = {"M_e_min": int(counts.min()), "M_e_max": int(counts.max()),
                     "N": synth.MOE_INTER, "K": K_DIM, "us": round(ms * 1e3, 2),
                     "TFLOP/s": round(flops / ms / 1e9, 1),
                     "frac_roofline": round(bound / ms, 4),
                     "launches": 1 if name == "moe_32_experts_grouped" else int((counts > 0).sum())}
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(n_rows: int = 256, seed: int = 0):
    """Inputs of the bounded decode sample: all four activations, the first n_rows of the
    weight matrix (2 scale rows)."""
    b_codes, b_s = synth.weights(N_DIM, K_DIM, seed, "decode/B")
    b = np.ascontiguousarray(b_codes[:n_rows])
    bs = np.ascontiguousarray(b_s[: -(-n_rows // 128)])
    xs = [synth.decode(M, seed) for M in DECODE_MS]
    return xs, b, bs


def oracle_step(xs, b, bs):
    import oracle
    for x in xs:
        y, s = oracle.act_quant(x)
        oracle.gemm(y, s, b, bs)


def oracle_sample_bytes(n_rows):
    return sum(act_quant_bytes(M, K_DIM) + gemm_bytes(M, n_rows, K_DIM) for M in DECODE_MS)


def cpu_baseline(target_s: float = 12.0):
    n_rows = 256
    xs, b, bs = oracle_sample(n_rows)
    t0 = time.perf_counter()
    oracle_step(xs, b, bs)
    one = time.perf_counter() - t0
    reps = max(1, int(target_s / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(xs, b, bs)
    dt = (time.perf_counter() - t0) / reps
    return {"value": round(oracle_sample_bytes(n_rows) / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"decode workload with N cut to the first {n_rows} of {N_DIM} weight rows: "
                       f"act_quant of all M in {list(DECODE_MS)} rows x {K_DIM} and fp8_gemm "
                       f"[M x {n_rows} x {K_DIM}]; single-threaded C, {reps} repetitions, "
                       f"{dt * 1e3:.1f} ms each")}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


_pg = None


def init_dist(world, backend):
    global _pg
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
        _pg = dist


def barrier(world):
    if world > 1 and _pg is not None:
        _pg.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1 or _pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    _pg.all_reduce(t, op=_pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- main

def run_profile(case: str, launches: int, warmup: int):
    """One kernel of the path on its full-size workload, `warmup` + `launches` times, with no
    other work: the command profiled by ncu (one kernel name per case)."""
    import torch
    g = Gpu()
    if case.startswith("decode"):
        M = int(case[len("decode"):] or 64)
        b, bs = synth.weights(N_DIM, K_DIM, 0, "decode/B")
        B, S = g.e4m3(b), g.f32(bs)
        x = g.bf16(synth.decode(M))
        y = torch.empty((M, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K_DIM // 128), dtype=torch.float32, device="cuda")
        c = torch.empty((M, N_DIM), dtype=torch.bfloat16, device="cuda")
        g.act_quant(x, y, s, M, K_DIM)
        fn = lambda: g.gemm_ex(y, s, B, S, c, M, N_DIM, K_DIM, 0,  # noqa: E731
                               WEIGHTS_CONSTANT)
    elif case.startswith("expert") or case.startswith("down"):
        # decode GEMMs with few weight slabs (split K): expert1..expert64 (N=2048, K=7168),
        # down1..down64 (N=7168, K=18432)
        expert = case.startswith("expert")
        M = int(case[len("expert" if expert else "down"):] or 1)
        N, K = (synth.MOE_INTER, K_DIM) if expert else (K_DIM, N_DIM)
        b, bs = synth.weights(N, K, 0, "decode/profile")
        B, S = g.e4m3(b), g.f32(bs)
        x = g.bf16(synth.activations(M, K, 0, "decode/profile/x", outlier_frac=0.01))
        y = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        g.act_quant(x, y, s, M, K)
        fn = lambda: g.gemm_ex(y, s, B, S, c, M, N, K, 0,  # noqa: E731
                               WEIGHTS_CONSTANT)
    elif case in ("prefill_up", "prefill_down"):
        up = case == "prefill_up"
        N, K = (N_DIM, K_DIM) if up else (K_DIM, N_DIM)
        b, bs = synth.weights(N, K, 0, "prefill/B_up" if up else "prefill/B_down")
        B, S = g.e4m3(b), g.f32(bs)
        x = g.bf16(synth.prefill_up() if up else synth.prefill_down())
        y = torch.empty((4096, K), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((4096, K // 128), dtype=torch.float32, device="cuda")
        c = torch.empty((4096, N), dtype=torch.bfloat16, device="cuda")
        g.act_quant(x, y, s, 4096, K)
        fn = lambda: g.gemm_ws(y, s, B, S, c, 4096, N, K)  # noqa: E731
    elif case == "prefill_up_ue8m0":
        # the prefill up-projection with ue8m0 scales, on the block-scaled kernel
        b, bs = synth.weights(N_DIM, K_DIM, 0, "prefill/B_up", pow2=True)
        B, S = g.e4m3(b), g.f32(bs)
        x = g.bf16(synth.prefill_up())
        y = torch.empty((4096, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((4096, K_DIM // 128), dtype=torch.float32, device="cuda")
        c = torch.empty((4096, N_DIM), dtype=torch.bfloat16, device="cuda")
        g.act_quant(x, y, s, 4096, K_DIM, 1)
        fn = lambda: g.gemm_ws(y, s, B, S, c, 4096, N_DIM, K_DIM, 1)  # noqa: E731
    elif case.startswith("mla"):
        # ue8m0 MLA projection on the block-scaled kernel: mla1536 or mla576
        N = int(case[len("mla"):] or synth.Q_LORA)
        b, bs = synth.weights(N, K_DIM, 0, f"mla/B{N}", pow2=True)
        B, S = g.e4m3(b), g.f32(bs)
        x = g.bf16(synth.mla_acts())
        y = torch.empty((2048, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((2048, K_DIM // 128), dtype=torch.float32, device="cuda")
        c = torch.empty((2048, N), dtype=torch.bfloat16, device="cuda")
        g.act_quant(x, y, s, 2048, K_DIM, 1)
        fn = lambda: g.gemm_ws(y, s, B, S, c, 2048, N, K_DIM, 1)  # noqa: E731
    elif case == "act_quant_mla":
        # the ue8m0 MLA input, 2048 x 7168
        x = g.bf16(synth.mla_acts())
        y = torch.empty((2048, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((2048, K_DIM // 128), dtype=torch.float32, device="cuda")
        fn = lambda: g.act_quant(x, y, s, 2048, K_DIM, 1)  # noqa: E731
    elif case.startswith("act_quant_decode"):
        # act_quant at a decode size: act_quant_decode1 .. act_quant_decode64 rows of 7168
        M = int(case[len("act_quant_decode"):] or 64)
        x = g.bf16(synth.decode(M))
        y = torch.empty((M, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((M, K_DIM // 128), dtype=torch.float32, device="cuda")
        fn = lambda: g.act_quant(x, y, s, M, K_DIM)  # noqa: E731
    elif case == "act_quant":
        rows, _ = synth.moe_routing(0)
        x = g.bf16(synth.activations(1024, K_DIM, 0, "moe/tokens", outlier_frac=0.01)[rows])
        y = torch.empty((8192, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((8192, K_DIM // 128), dtype=torch.float32, device="cuda")
        fn = lambda: g.act_quant(x, y, s, 8192, K_DIM)  # noqa: E731
    elif case == "moe":
        rows, counts = synth.moe_routing(0)
        x = g.bf16(synth.activations(1024, K_DIM, 0, "moe/tokens", outlier_frac=0.01)[rows])
        y = torch.empty((8192, K_DIM), dtype=torch.float8_e4m3fn, device="cuda")
        s = torch.empty((8192, K_DIM // 128), dtype=torch.float32, device="cuda")
        g.act_quant(x, y, s, 8192, K_DIM)
        ws = [synth.weights(synth.MOE_INTER, K_DIM, 0, f"moe/B{e}") for e in range(32)]
        B = g.e4m3(np.stack([w for w, _ in ws]))
        S = g.f32(np.stack([sc for _, sc in ws]))
        c = torch.empty((8192, synth.MOE_INTER), dtype=torch.bfloat16, device="cuda")
        offs = [int(v) for v in np.r_[0, np.cumsum(counts)]]
        fn = lambda: g.fp8bs.fp8bs_gemm_grouped(  # noqa: E731
            y.data_ptr(), s.data_ptr(), B.data_ptr(), S.data_ptr(), c.data_ptr(), offs, 32,
            synth.MOE_INTER, K_DIM, 0, g.sh)
    elif case.startswith("linear"):
        # the bf16 path: linear1 (decode row), linear64, linear4096 (prefill rows)
        M = int(case[len("linear"):] or 1)
        b, bs = synth.weights(N_DIM, K_DIM, 0, "prefill/B_up")
        W, WS = g.e4m3(b), g.f32(bs)
        x = g.bf16(synth.prefill_up()[:M] if M > 64 else synth.decode(M))
        Y = torch.empty((M, N_DIM), dtype=torch.bfloat16, device="cuda")
        fn = lambda: g.linear_bf16(x, W, WS, Y, M, N_DIM, K_DIM)  # noqa: E731
    elif case == "dequant":
        b, bs = synth.weights(N_DIM, K_DIM, 0, "prefill/B_up")
        W, WS = g.e4m3(b), g.f32(bs)
        Y = torch.empty((N_DIM, K_DIM), dtype=torch.bfloat16, device="cuda")
        fn = lambda: g.dequant(W, WS, Y, N_DIM, K_DIM)  # noqa: E731
    else:
        raise SystemExit(f"unknown profile case {case!r}")
    torch.cuda.synchronize()
    for _ in range(warmup + launches):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"profile": case, "launches": warmup + launches}), flush=True)
    return 0


def workload_config():
    return {"workload": (f"decode: act_quant + fp8_gemm for M in {list(DECODE_MS)}, "
                         f"K={K_DIM}, N={N_DIM}, fp32 block scales"),
            "M": list(DECODE_MS), "K": K_DIM, "N": N_DIM,
            "l2": "inputs larger than L2: each M has its own 132 MB weight (528 MB per step)",
            "parallelism": "replicas"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    n_rows = 256
    xs, b, bs = oracle_sample(n_rows)
    for _ in range(args.warmup):
        oracle_step(xs, b, bs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(xs, b, bs)
    dt = time.perf_counter() - t0
    value = oracle_sample_bytes(n_rows) * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "host_cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"per step: decode workload with N cut to {n_rows} of "
                                       f"{N_DIM} weight rows (all M rows of act_quant)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only: no secondary workloads "
                    "and no CPU baseline")
    ap.add_argument("--out-dir", default=os.path.join(ROOT, "bench_out"),
                    help="where the per-rank clock samples (clocks_rank<r>.csv) are written")
    ap.add_argument("--profile", metavar="CASE", default=None,
                    help="run one kernel only (decode1..decode64, expert1..expert64, down1..down64, prefill_up, prefill_down, prefill_up_ue8m0, mla1536, mla576, linear1..linear4096, "
                         "act_quant, act_quant_mla, dequant, moe): warmup + steps launches, for ncu")
    args = ap.parse_args(argv)
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()

    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.profile:
        return run_profile(args.profile, args.steps, args.warmup)

    import torch
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    g = Gpu()
    peaks = load_peaks()
    os.makedirs(args.out_dir, exist_ok=True)
    clocks_path = os.path.join(args.out_dir, f"clocks_rank{rank}.csv")

    ms_total, eager_ms, per_m, clocks = run_decode(g, args.steps, args.warmup, rank, world,
                                                   clocks_path)
    ms_total = max_over_ranks(ms_total, world, "cuda")
    eager_ms = max_over_ranks(eager_ms, world, "cuda")
    e2e_ms, h2d, d2h = run_decode_e2e(g, args.steps, args.warmup, world)
    e2e_ms = max_over_ranks(e2e_ms, world, "cuda")

    step_bytes = decode_step_bytes()
    ms_per_step = ms_total / args.steps
    value = world * step_bytes / (ms_per_step * 1e6)
    e2e_value = world * step_bytes / (e2e_ms / args.steps * 1e6)

    gemm_bytes_total = sum(gemm_bytes(M, N_DIM, K_DIM) for M in DECODE_MS)
    gemm_ms = sum(d for _, d in per_m)
    achieved = gemm_bytes_total / (gemm_ms * 1e6)
    roofline = {"kernel": "gemm_swapab_kernel (decode fp8_gemm, all four M; per M, 4 x rounds "
                          "launches back to back over four distinct weights, one event pair "
                          "around the region)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": f"{peaks['source']} hbm_gbs (copy bandwidth)",
                "traffic": decode_traffic(),
                "traffic_note": "dram read+write bytes per launch of gemm_swapab_kernel, from an "
                                "ncu capture; null if the kernel's sources changed since",
                "per_launch": [{"M": M, "us": round(d * 1e3, 2),
                                "GB/s": round(gemm_bytes(M, N_DIM, K_DIM) / (d * 1e6), 1)}
                               for M, d in per_m]}

    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "step_launch": f"CUDA graphs of {GRAPH_STEPS} steps",
            "eager_ms_per_step": round(eager_ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic", "config": workload_config(),
            "clocks": clocks, "roofline": roofline,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "transfers": "pinned host buffers every step: act_quant reads each "
                                 "activation from host memory over NVLink-C2C; C of M <= "
                                 f"{E2E_DIRECT_MAX_M} written to host memory by the GEMM, the "
                                 "larger C copied out while later problems compute"},
            "gpu_launches": 2 * len(DECODE_MS) * args.steps}
    if rank == 0 and world == 1 and not args.quick:
        sampler = ClockSampler(torch.cuda.current_device(),
                               os.path.join(args.out_dir, "clocks_secondary.csv"))
        with sampler:
            line["secondary"] = secondary(g, peaks)
        line["secondary"]["clocks"] = sampler.summary()
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        _pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
