"""A larger seeded random campaign through every public GEMM entry point, every output element
against the oracle. It complements test_parity_gpu_fuzz.py (a few dozen fixed draws) with as
many draws as asked for, in five families:

  plan     fp8_gemm with the library's own plan: M from 1 to ~1300, ragged or aligned N,
           K a multiple of 128, both scale formats, with or without a stream-K workspace,
           with or without the weights-constant flag;
  config   fp8bs_gemm_config with a random kernel, tile width and K split (0 = stream-K):
           supported choices must match the oracle, the rest must be rejected without
           writing C;
  grouped  fp8_gemm_grouped with 1-19 groups of 0 to ~700 rows;
  fused    act_quant_gemm (two launches, or the in-kernel quantisation at M <= 16): y and s
           bit for bit, C within the tolerance;
  bf16     linear_bf16 (the weight dequantised on chip, "DeepSeek-V3 Administrator &
           Developer Guide" §6.3, gemm_impl = "bf16").

Every call runs twice and the two results must agree bit for bit; the device error word must
stay zero. GEMM results are held to the accuracy contract of fp8_gemm (§8.5.3: fp32
accumulation of each K block, one rounding to bf16), parity_util.gemm_violations. Shapes are
capped at 2-3e8 multiply-adds so that the oracle (in a pool of processes started before CUDA,
which also builds the inputs) keeps up.

    python tests/fuzz_campaign.py --plan 1500 --config 1500 --grouped 400 --fused 600 \\
        --bf16 500 --base 1000

Exit status 0 when every comparison passed.
"""
import argparse
import multiprocessing as mp
import os
import sys
import time
import traceback

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

# kernel ids of fp8bs_gemm_config (checked against the binding before the first call)
SWAPPED, PROMOTED, BLOCK_SCALED, PAIR = 0, 1, 2, 3
TILES = {SWAPPED: [16, 32, 64, 128], PROMOTED: [64, 128, 192, 256],
         BLOCK_SCALED: [64, 128, 192, 256], PAIR: [128, 192, 256]}
FAMILIES = ("plan", "config", "grouped", "fused", "bf16")
SEED_BASE = {"plan": 50000, "config": 60000, "grouped": 70000, "fused": 80000, "bf16": 90000}


def _fmt(name):
    import oracle
    return oracle.SCALE_UE8M0 if name == "ue8m0" else oracle.SCALE_FP32


def _shrink(M, N, K, cap, k_first=True):
    """Halve K (keeping a multiple of 128), then N, until M*N*K <= cap."""
    while M * N * K > cap:
        if k_first and K > 128:
            K = 128 * max(1, K // 256)
        elif N > 1:
            N = max(1, N // 2)
        else:
            break
    return N, K


def draw(job):
    """Case i of a family: its parameters and inputs (synth draws, the oracle's act_quant)."""
    import oracle
    import synth
    family, i, base = job
    seed = SEED_BASE[family] + base + i
    rng = np.random.default_rng(seed)
    c = {"family": family, "i": i}
    if family == "plan":
        M = int(rng.choice([int(rng.integers(1, 129)), int(rng.integers(129, 1300))]))
        N = int(rng.integers(1, 3000))
        if rng.random() < 0.5:
            N = max(8, N // 8 * 8)
        N, K = _shrink(M, N, 128 * int(rng.integers(1, 40)), 2e8)
        c.update(M=M, N=N, K=K, fmt="ue8m0" if rng.random() < 0.5 else "fp32",
                 use_ws=bool(rng.random() < 0.5), wc=bool(rng.random() < 0.3))
    elif family == "config":
        kernel = [SWAPPED, PROMOTED, BLOCK_SCALED, PAIR][int(rng.integers(0, 4))]
        tile = int(rng.choice(TILES[kernel]))
        ksplit = int(rng.choice([0, 1, 1, 2, 3, 4, 5, 6, 8]))
        M = int(rng.integers(1, tile + 1)) if kernel == SWAPPED else int(rng.integers(129, 2800))
        N = int(rng.integers(1, 3000))
        if rng.random() < 0.6:
            N = max(8, N // 8 * 8)
        N, K = _shrink(M, N, 128 * int(rng.integers(1, 24)), 3e8)
        fmt = "ue8m0" if kernel in (BLOCK_SCALED, PAIR) or rng.random() < 0.3 else "fp32"
        c.update(M=M, N=N, K=K, fmt=fmt, kernel=kernel, tile=tile, ksplit=ksplit)
    elif family == "grouped":
        G = int(rng.integers(1, 20))
        counts = [int(rng.choice([0, 1, int(rng.integers(1, 65)), int(rng.integers(65, 300)),
                                  int(rng.integers(300, 700))])) for _ in range(G)]
        if sum(counts) == 0:
            counts[0] = 1
        N = int(rng.choice([int(rng.integers(1, 1500)), 8 * int(rng.integers(1, 260))]))
        N, K = _shrink(sum(counts), N, 128 * int(rng.integers(1, 10)), 3e8, k_first=False)
        c.update(counts=counts, offs=np.r_[0, np.cumsum(counts)], M=sum(counts), N=N, K=K,
                 fmt="ue8m0" if rng.random() < 0.5 else "fp32")
    elif family == "fused":
        M = int(rng.integers(1, 17)) if rng.random() < 0.7 else int(rng.integers(17, 400))
        N, K = int(rng.integers(1, 20000)), 128 * int(rng.integers(1, 90))
        while (M * N * K > 3e8 or N * K > 4e7) and N > 1:
            N = max(1, N // 2)
        c.update(M=M, N=N, K=K, fmt="ue8m0" if rng.random() < 0.5 else "fp32",
                 qik=bool(rng.random() < 0.7), wc=bool(rng.random() < 0.5),
                 use_ws=bool(rng.random() < 0.5))
    else:  # bf16
        M = int(rng.choice([int(rng.integers(1, 129)), int(rng.integers(129, 1500))]))
        N, K = _shrink(M, int(rng.integers(1, 3000)), 128 * int(rng.integers(1, 30)), 2e8,
                       k_first=False)
        c.update(M=M, N=N, K=K, wc=bool(rng.random() < 0.5))
        c["x"] = synth.activations(M, K, seed=seed, name="campL", outlier_frac=0.01)
        c["w"], c["w_s"] = synth.weights(N, K, seed=seed + 1, name="campLB")
        return c
    pow2 = c["fmt"] == "ue8m0"
    c["x"] = synth.activations(c["M"], c["K"], seed=seed, name=f"camp{family}A",
                               outlier_frac=0.01)
    c["a"], c["a_s"] = oracle.act_quant(c["x"], _fmt(c["fmt"]))
    if family == "grouped":
        ws = [synth.weights(c["N"], c["K"], seed=seed + 1 + e, name="campgroupedB", pow2=pow2)
              for e in range(len(c["counts"]))]
        c["b"], c["b_s"] = np.stack([w for w, _ in ws]), np.stack([s for _, s in ws])
    else:
        c["b"], c["b_s"] = synth.weights(c["N"], c["K"], seed=seed + 1,
                                         name=f"camp{family}B", pow2=pow2)
    return c


def reference(job):
    import oracle
    kind, args = job
    return oracle.gemm(*args) if kind == "gemm" else oracle.linear_bf16(*args)


def run(counts, base, workers):
    pool = mp.get_context("spawn").Pool(workers)    # before the first CUDA call
    jobs = [(f, i, base) for f in FAMILIES for i in range(counts[f])]
    cases = pool.imap(draw, jobs, chunksize=1)

    import torch
    import fp8_block_scaled_fp8bs_gb300 as fp8bs
    from parity_util import dev_bf16, dev_e4m3, dev_f32, gemm_violations
    assert (SWAPPED, PROMOTED, BLOCK_SCALED, PAIR) == (
        fp8bs.KERNEL_SWAPPED, fp8bs.KERNEL_PROMOTED, fp8bs.KERNEL_BLOCK_SCALED,
        fp8bs.KERNEL_BLOCK_SCALED_PAIR)
    ws = torch.zeros(fp8bs.fp8bs_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    fp8bs.fp8bs_device_error(clear=True)
    stats = {"compared": 0, "rejected": 0}
    fails, pending, worst = [], [], [0.0]
    t0 = time.time()

    def host(t):
        return t.float().cpu().numpy()

    def identical(t1, t2):
        return torch.equal(t1.contiguous().view(torch.uint8), t2.contiguous().view(torch.uint8))

    def settle(label):
        torch.cuda.synchronize()
        err = fp8bs.fp8bs_device_error(clear=True)
        if err:
            fails.append(f"{label}: device error word {err:#x}")

    def compare_later(label, kind, args, got):
        pending.append((label, pool.apply_async(reference, ((kind, args),)), got))

    def drain(wait):
        keep = []
        for label, res, got in pending:
            if not wait and not res.ready():
                keep.append((label, res, got))
                continue
            try:
                ref = res.get(timeout=900)
            except Exception:
                fails.append(f"{label}: oracle failed: {traceback.format_exc(limit=1)}")
                continue
            bad, ratio = gemm_violations(got, ref)
            worst[0] = max(worst[0], ratio)
            stats["compared"] += 1
            if bad:
                fails.append(f"{label}: {bad} elements outside tolerance (worst {ratio:.3g})")
        pending[:] = keep

    for n, c in enumerate(cases):
        f, M, N, K = c["family"], c["M"], c["N"], c["K"]
        label = f"{f} {c['i']}: {M}x{N}x{K}"
        if f in ("plan", "config", "fused"):
            A, AS = dev_e4m3(c["a"]), dev_f32(c["a_s"])
            Bd, BS = dev_e4m3(c["b"]), dev_f32(c["b_s"])
        if f == "plan":
            w = ws if c["use_ws"] else None
            plan = fp8bs.fp8bs_gemm_plan(M, N, K, fp8bs._fmt(c["fmt"]), c["use_ws"])
            label += f" {c['fmt']} workspace={c['use_ws']} weights_constant={c['wc']} {plan}"
            out = [fp8bs.fp8_gemm(A, AS, Bd, BS, c["fmt"], weights_constant=c["wc"], workspace=w)
                   for _ in range(2)]
            settle(label)
            compare_later(label, "gemm", (c["a"], c["a_s"], c["b"], c["b_s"]), host(out[0]))
        elif f == "config":
            label += f" {c['fmt']} kernel {c['kernel']} tile {c['tile']} ksplit {c['ksplit']}"
            out = []
            for _ in range(2):
                cc = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
                try:
                    fp8bs.fp8bs_gemm_config(
                        A.data_ptr(), AS.data_ptr(), Bd.data_ptr(), BS.data_ptr(), cc.data_ptr(),
                        M, N, K, fp8bs._fmt(c["fmt"]), 0, c["kernel"], c["tile"], c["ksplit"],
                        ws.data_ptr() if c["ksplit"] == 0 else 0,
                        ws.numel() if c["ksplit"] == 0 else 0, stream)
                except fp8bs.Fp8bsError:
                    torch.cuda.synchronize()
                    if not bool(torch.isnan(cc.float()).all()):
                        fails.append(f"{label}: rejected, but C was written")
                    out = None
                    break
                out.append(cc)
            settle(label)
            if out is None:
                stats["rejected"] += 1
                continue
            compare_later(label, "gemm", (c["a"], c["a_s"], c["b"], c["b_s"]), host(out[0]))
        elif f == "grouped":
            A, AS = dev_e4m3(c["a"]), dev_f32(c["a_s"])
            Bd, BS = dev_e4m3(c["b"]), dev_f32(c["b_s"])
            label = f"grouped {c['i']}: rows {c['counts']} N={N} K={K} {c['fmt']}"
            out = [fp8bs.fp8_gemm_grouped(A, AS, Bd, BS, c["offs"], c["fmt"]) for _ in range(2)]
            settle(label)
            h = host(out[0])
            for e in range(len(c["counts"])):
                lo, hi = int(c["offs"][e]), int(c["offs"][e + 1])
                if hi > lo:
                    compare_later(f"{label} group {e}", "gemm",
                                  (c["a"][lo:hi], c["a_s"][lo:hi], c["b"][e], c["b_s"][e]),
                                  h[lo:hi])
        elif f == "fused":
            label += (f" {c['fmt']} quant_in_kernel={c['qik']} weights_constant={c['wc']} "
                      f"workspace={c['use_ws']}")
            X = dev_bf16(c["x"])
            w = ws if c["use_ws"] else None
            r = [fp8bs.act_quant_gemm(X, Bd, BS, c["fmt"], weights_constant=c["wc"],
                                      workspace=w, quant_in_kernel=c["qik"]) for _ in range(2)]
            settle(label)
            for t1, t2, name in zip(r[0], r[1], ("C", "y", "s")):
                if not identical(t1, t2):
                    fails.append(f"{label}: two calls differ in {name}")
            if not np.array_equal(r[0][1].view(torch.uint8).cpu().numpy(), c["a"]):
                fails.append(f"{label}: y is not the oracle's act_quant codes")
            if not np.array_equal(r[0][2].cpu().numpy().view(np.uint32), c["a_s"].view(np.uint32)):
                fails.append(f"{label}: s is not the oracle's act_quant scales")
            compare_later(label, "gemm", (c["a"], c["a_s"], c["b"], c["b_s"]), host(r[0][0]))
            out = [r[0][0], r[1][0]]
        else:
            label += f" weights_constant={c['wc']}"
            X, W, WS = dev_bf16(c["x"]), dev_e4m3(c["w"]), dev_f32(c["w_s"])
            out = [fp8bs.linear_bf16(X, W, WS, weights_constant=c["wc"]) for _ in range(2)]
            settle(label)
            compare_later(label, "linear", (c["x"], c["w"], c["w_s"]), host(out[0]))
        if not identical(out[0], out[1]):
            fails.append(f"{label}: two calls differ")
        if (n + 1) % 200 == 0:
            drain(False)
            print(f"{n + 1} cases run in {time.time() - t0:.1f} s", flush=True)
    drain(True)
    pool.close()
    pool.join()
    print(f"{len(jobs)} cases in {time.time() - t0:.1f} s: {stats['compared']} outputs compared, "
          f"{stats['rejected']} configurations rejected, worst error/bound {worst[0]:.3g}",
          flush=True)
    for line in fails:
        print("FAIL", line, flush=True)
    print(f"failures: {len(fails)}", flush=True)
    return 0 if not fails else 1


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    for f, n in zip(FAMILIES, (150, 150, 50, 80, 60)):
        p.add_argument(f"--{f}", type=int, default=n, help=f"number of {f} cases")
    p.add_argument("--base", type=int, default=0, help="offset added to every case's seed")
    p.add_argument("--workers", type=int, default=max(2, (os.cpu_count() or 4) - 2))
    a = p.parse_args(argv)
    return run({f: getattr(a, f) for f in FAMILIES}, a.base, a.workers)


if __name__ == "__main__":
    sys.exit(main())
