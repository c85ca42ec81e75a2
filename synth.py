"""Seeded synthetic inputs for the FP8 block-scaled linear path.

This module serves both sides of every check -- the CUDA library and the CPU oracle -- and
therefore holds none of the method's arithmetic: it only draws numbers and stores them in the
input formats (bf16 activations, e4m3fn weight codes with fp32 block scales). Rounding to those
formats uses PyTorch's own casts (RNE); both sides then read the very same bytes.

Workloads (DeepSeek-V3 dimensions: hidden 7168, dense MLP inter 18432, expert inter 2048,
q low-rank 1536, kv low-rank 512 + rope 64):
  tiny     A bf16 [16,512] ~ N(0,1); B [256,512] = e4m3(N(0,1)/s_b), s_b [2,4] log-uniform
           in [2^-10, 2^-6]; fp32 activation scales.
  decode   A bf16 [M,7168], M in {1,8,32,64}, N(0,1) with 1% of elements scaled by 50;
           B [18432,7168] with 128x128 log-uniform scales.
  prefill  A [4096,7168] with B [18432,7168] (up) and A [4096,18432] with B [7168,18432]
           (down); also weight_dequant of the [18432,7168] matrix.
  moe      1024 tokens x 8 slots routed over 32 experts with Categorical(p), p ~ Dirichlet(0.5);
           rows gathered by expert (stable) -> A_g [8192,7168]; experts B_e [2048,7168].
  mla      A [2048,7168] ~ N(0,1) quantised with power-of-two scales; B [1536,7168] and
           [576,7168] with power-of-two block scales 2^e, e uniform in {-10..-6}.

Every tensor draws from its own numpy Generator seeded with (seed, tensor id), so a tensor
does not depend on which other tensors were drawn before it.
"""
from __future__ import annotations

import zlib

import numpy as np
import torch

BLOCK = 128
DIM = 7168
INTER = 18432
MOE_INTER = 2048
Q_LORA = 1536
KV_LORA_ROPE = 576
DECODE_MS = (1, 8, 32, 64)


def _rng(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), zlib.crc32(name.encode())])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), rounded by torch (RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 array with |x| <= 448 -> e4m3fn codes (uint8), rounded by torch (RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def activations(M: int, K: int, seed: int = 0, name: str = "A",
                outlier_frac: float = 0.0, outlier_gain: float = 50.0) -> np.ndarray:
    """bf16 [M,K] ~ N(0,1); a Bernoulli(outlier_frac) subset of elements is multiplied by
    outlier_gain. Returned as uint16 bit patterns."""
    rng = _rng(seed, f"act/{name}/{M}x{K}")
    z = rng.standard_normal((M, K), dtype=np.float32)
    if outlier_frac > 0:
        mask = rng.random((M, K), dtype=np.float32) < outlier_frac
        z[mask] *= np.float32(outlier_gain)
    return to_bf16_bits(z)


def weight_scales(N: int, K: int, seed: int = 0, name: str = "B",
                  pow2: bool = False) -> np.ndarray:
    """fp32 [ceil(N/128), ceil(K/128)]: 2^u with u ~ U(-10,-6) (log-uniform), or with pow2=True
    2^e with e uniform in {-10,...,-6}."""
    rng = _rng(seed, f"wscale/{name}/{N}x{K}/{int(pow2)}")
    shape = (-(-N // BLOCK), -(-K // BLOCK))
    if pow2:
        e = rng.integers(-10, -5, size=shape)
        return np.ldexp(np.float32(1.0), e).astype(np.float32)
    u = rng.uniform(-10.0, -6.0, size=shape)
    return np.exp2(u).astype(np.float32)


def weights(N: int, K: int, seed: int = 0, name: str = "B", pow2: bool = False):
    """e4m3fn codes B [N,K] = e4m3(z / s_b[n/128, k/128]), z ~ N(0,1), saturated at +-448, with
    their fp32 block scales s_b. Returns (codes uint8 [N,K], s_b float32)."""
    s_b = weight_scales(N, K, seed, name, pow2)
    rng = _rng(seed, f"wval/{name}/{N}x{K}")
    z = rng.standard_normal((N, K), dtype=np.float32)
    full = np.repeat(np.repeat(s_b, BLOCK, axis=0)[:N], BLOCK, axis=1)[:, :K]
    t = np.clip(z / full, -448.0, 448.0)
    return to_e4m3_codes(t), s_b


def moe_routing(seed: int = 0, tokens: int = 1024, slots_per_token: int = 8,
                experts: int = 32, alpha: float = 0.5):
    """Synthetic top-k routing: p ~ Dirichlet(alpha * 1), each of tokens*slots_per_token slots
    picks an expert ~ Categorical(p); slot i belongs to token i // slots_per_token.
    Returns (rows, counts): rows[j] is the token of the j-th gathered row, slots grouped by
    expert in a stable order; counts[e] is the number of rows of expert e."""
    rng = _rng(seed, f"moe/{tokens}/{slots_per_token}/{experts}/{alpha}")
    p = rng.dirichlet(np.full(experts, alpha))
    slots = tokens * slots_per_token
    choice = rng.choice(experts, size=slots, p=p)
    order = np.argsort(choice, kind="stable")
    rows = (order // slots_per_token).astype(np.int64)
    counts = np.bincount(choice, minlength=experts).astype(np.int64)
    return rows, counts


# ----------------------------------------------------------------------------- workloads

def tiny(seed: int = 0):
    return {
        "x": activations(16, 512, seed, "tiny/A"),
        "b": weights(256, 512, seed, "tiny/B"),
    }


def decode(M: int, seed: int = 0):
    return activations(M, DIM, seed, f"decode/A{M}", outlier_frac=0.01)


def prefill_up(seed: int = 0):
    return activations(4096, DIM, seed, "prefill/A_up", outlier_frac=0.01)


def prefill_down(seed: int = 0):
    return activations(4096, INTER, seed, "prefill/A_down", outlier_frac=0.01)


def mla_acts(seed: int = 0):
    return activations(2048, DIM, seed, "mla/A")
