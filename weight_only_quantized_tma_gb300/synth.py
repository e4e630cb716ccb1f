"""Seeded synthetic inputs for the weight-only quantized GEMM.

This module draws random arrays and nothing else: it holds none of the GEMM's
arithmetic (no unpacking, no dequantisation, no products).  The same arrays feed
the float64 oracle and the CUDA path.  Every array is returned as raw storage
(uint8 codes, uint16 bit patterns of fp16/bf16, float32 scalars) so that both
sides read exactly the same bits.

Value recipes (one per weight format) follow the workloads the source pages
measure:

* INT4 W4A16 -- activations ~ N(0, 1) rounded to fp16 (or bf16); codes uniform
  over 0..15, two per byte along K (so the packed bytes are uniform over 0..255);
  group scales ~ U[0.005, 0.02] rounded to fp16, laid out [K/G, N].
* FP8 W8A16 -- activations ~ N(0, 1) in bf16; a weight W ~ N(0, 0.02) is encoded
  as e4m3(clamp(W / s, +-448)) with one per-tensor fp32 scale s = max|W| / 448.
* INT4 codebook -- INT4 codes and scales as above; the 16-entry fp16 table is an
  NF4-style normal-quantile codebook or 16 draws from N(0, 1).
* INT2 W2A16 -- codes uniform over 0..3, four per byte along K; scales as INT4.
* BF16 x FP4 -- activations ~ N(0, 1) in bf16; e2m1 codes uniform over all 16
  values, two per byte along K; one e4m3 block scale ~ U[0.25, 2] per 16 values
  along K, laid out [N, K/16]; global alpha = 0.01.

Seeds are ``1000 * config_index + case_index``; numpy's PCG64 draws everything.
Rounding of the random reals to fp16 / bf16 / e4m3 is done by numpy's and torch's
own round-to-nearest-even casts.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np


def seed_for(config_index: int, case_index: int) -> int:
    return 1000 * int(config_index) + int(case_index)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def _to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array -> uint16 bit pattern of its RNE rounding to fp16 / bf16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch
        return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(f"unknown activation dtype {dtype!r}")


def _to_e4m3(x: np.ndarray) -> np.ndarray:
    """float32 array (already inside +-448) -> e4m3 (FN) codes by torch's RNE cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def activations(M: int, K: int, dtype: str, seed: int) -> np.ndarray:
    """A [M, K] ~ N(0, 1), as fp16 or bf16 bits."""
    return _to_bits(_rng(seed).standard_normal((M, K), dtype=np.float32), dtype)


@dataclass
class Int4Weights:
    w: np.ndarray        # uint8 [N, K/2], canonical: even k in the low nibble
    s: np.ndarray        # uint16 fp16 bits [K/G, N]
    N: int
    K: int
    G: int


def int4_weights(N: int, K: int, G: int, seed: int, scale_lo: float = 0.005,
                 scale_hi: float = 0.02) -> Int4Weights:
    rng = _rng(seed)
    w = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = rng.uniform(scale_lo, scale_hi, size=(K // G, N)).astype(np.float32)
    return Int4Weights(w=w, s=_to_bits(s, "f16"), N=N, K=K, G=G)


def int4_zeros(N: int, K: int, G: int, seed: int) -> np.ndarray:
    """Zero points uint8 [K/G, N], uniform over the codes 0..15."""
    return _rng(seed).integers(0, 16, size=(K // G, N), dtype=np.uint8)


def normal_quantile_codebook() -> np.ndarray:
    """An NF4-style 16-entry codebook as fp16 bits, ascending: quantiles of N(0, 1)
    at evenly spaced probabilities (7 below the median, 8 above, offset 0.03 from
    the tails), an exact zero at index 7, scaled so the largest magnitude is 1.
    The pages name NF4 as the non-uniform 4-bit choice but print no table; any 16
    values are valid input to the codebook GEMM."""
    from scipy.special import ndtri
    neg = ndtri(np.linspace(0.03, 0.5, 8)[:-1])
    pos = ndtri(np.linspace(0.5, 0.97, 9)[1:])
    v = np.concatenate([neg / -neg[0], [0.0], pos / pos[-1]]).astype(np.float32)
    return _to_bits(v, "f16")


def random_codebook(seed: int) -> np.ndarray:
    """16 codebook entries ~ N(0, 1) as fp16 bits (an arbitrary table)."""
    return _to_bits(_rng(seed).standard_normal(16, dtype=np.float32), "f16")


@dataclass
class Int2Weights:
    w: np.ndarray        # uint8 [N, K/4], canonical: code k at bits 2 (k % 4)
    s: np.ndarray        # uint16 fp16 bits [K/G, N]
    N: int
    K: int
    G: int


def int2_weights(N: int, K: int, G: int, seed: int, scale_lo: float = 0.005,
                 scale_hi: float = 0.02) -> Int2Weights:
    """Codes uniform over 0..3, four per byte along K (so bytes uniform over 0..255)."""
    rng = _rng(seed)
    w = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    s = rng.uniform(scale_lo, scale_hi, size=(K // G, N)).astype(np.float32)
    return Int2Weights(w=w, s=_to_bits(s, "f16"), N=N, K=K, G=G)


@dataclass
class Fp8Weights:
    w: np.ndarray        # uint8 e4m3 codes [N, K]
    scale: np.float32    # per-tensor fp32 scale s
    N: int
    K: int


def fp8_weights(N: int, K: int, seed: int, std: float = 0.02) -> Fp8Weights:
    rng = _rng(seed)
    W = rng.normal(0.0, std, size=(N, K)).astype(np.float32)
    s = np.float32(np.abs(W).max() / np.float32(448.0))
    codes = _to_e4m3(np.clip(W / s, -448.0, 448.0))
    return Fp8Weights(w=codes, scale=s, N=N, K=K)


@dataclass
class Fp4Weights:
    w: np.ndarray        # uint8 [N, K/2] e2m1 codes, even k in the low nibble
    sf: np.ndarray       # uint8 e4m3 codes [N, K/16]
    alpha: np.float32
    N: int
    K: int


def fp4_weights(N: int, K: int, seed: int, sf_lo: float = 0.25, sf_hi: float = 2.0,
                alpha: float = 0.01) -> Fp4Weights:
    rng = _rng(seed)
    w = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sf = _to_e4m3(rng.uniform(sf_lo, sf_hi, size=(N, K // 16)).astype(np.float32))
    return Fp4Weights(w=w, sf=sf, alpha=np.float32(alpha), N=N, K=K)


def bias(N: int, dtype: str, seed: int) -> np.ndarray:
    return _to_bits(_rng(seed).standard_normal(N, dtype=np.float32), dtype)


def sample_rows(M: int, count: int, seed: int) -> np.ndarray:
    """Sorted sample of row indices, always including the first and the last row."""
    if M <= count:
        return np.arange(M, dtype=np.int64)
    rng = _rng(seed)
    inner = rng.choice(np.arange(1, M - 1), size=count - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], inner]).astype(np.int64))


# The workloads, by name, with their sizes.  Index i of CONFIGS is config i.
@dataclass(frozen=True)
class Case:
    op: str                      # "w4a16" | "fp8" | "fp4"
    M: int
    N: int
    K: int
    G: Optional[int] = None      # INT4 group size
    a_dtype: str = "f16"


SMOKE = [Case("w4a16", 4, 512, 1024, 128, "f16")]
DECODE_SHAPES = [(4096, 4096), (11008, 4096), (4096, 11008), (12288, 4096)]
DECODE = [Case("w4a16", M, N, K, 128, "f16") for M in (1, 16) for (N, K) in DECODE_SHAPES]
PREFILL = [Case("w4a16", 4096, 4096, 4096, G, "f16") for G in (32, 64, 128, 256)]
FP8 = ([Case("fp8", M, N, K, None, "bf16") for (M, N, K) in
        [(32768, 3200, 5120), (16384, 12800, 5120), (8192, 10240, 5120)]]
       + [Case("fp8", M, 10240, 5120, None, "bf16") for M in (1, 16, 64)])
FP4 = [Case("fp4", M, 12800, 5120, None, "bf16") for M in (1, 128, 8192)]
CONFIGS = [SMOKE, DECODE, PREFILL, FP8, FP4]
