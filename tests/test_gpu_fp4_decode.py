"""GPU parity of the BF16 x FP4 decode kernel (M <= 16, K % 256 == 0) against the oracle.

The kernel reads the e2m1 codes straight from W [N, K/2] and the prepacked e4m3 block
scales, forms e2m1 * e4m3 exactly in registers, and sums in fp32 with alpha applied once.
Its lanes hold codes 8c .. 8c + 7 of each 32-code chunk for two k steps; the one-hot tests
pin that reordering, the per-lane block scale and the split-K placement (every position
inside a chunk, chunks across stages and K slices).
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, Fp4Problem, check_close, out_to_f64, to_dev_f16bits

pytestmark = pytest.mark.gpu


def _plan(M, N, K):
    return wq.get_plan(wq.WQ_OP_FP4, wq.WQ_BF16, M, N, K, 0)


def test_fp4_decode_plan():
    for M in (1, 16):
        plan = _plan(M, 12800, 5120)
        assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["ws_bytes"] == 0
    assert _plan(17, 12800, 5120)["kernel"] == wq.WQ_KERNEL_TILE
    assert _plan(4, 1024, 5248)["kernel"] == wq.WQ_KERNEL_TILE   # K % 256 == 128


@pytest.mark.parametrize("shift", [0, 1, 2])
def test_fp4_decode_one_hot_bit_exact(shift):
    # token m selects k_m: over the three shifts the 16 tokens cover all 32 positions of
    # a 32-code chunk (both k steps, every lane, both scale blocks), with chunks spread
    # over stages and K slices; out[m, n] = e2m1(W[n, k_m]) * e4m3(SF[n, k_m / 16])
    # exactly (alpha = 1; every such product is a bf16 value)
    M, N, K = 16, 392, 2048
    ks = [32 * ((5 * m + 3 * shift) % (K // 32)) + (m + 16 * (shift % 2) + shift // 2 * 7) % 32 for m in range(M)]
    p = Fp4Problem(M, N, K, seed=600 + shift)
    plan = _plan(M, N, K)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] > 1
    A = np.zeros((M, K), dtype=np.float32)
    A[np.arange(M), ks] = 1.0
    p.A = synth._to_bits(A, "bf16")
    p.A_d = to_dev_f16bits(p.A, "bf16")
    p.alpha = torch.ones(1, dtype=torch.float32, device=DEV)
    out = p.run()
    torch.cuda.synchronize()
    w = oracle.dequant_fp4(p.wts.w, p.wts.sf, K).astype(np.float64)   # [N, K]
    assert np.array_equal(out_to_f64(out), w[:, ks].T)


@pytest.mark.parametrize("N,K", [(136, 1024), (1000, 4096), (264, 256)])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_fp4_decode_ragged(M, N, K):
    # tail rows in the last 128-row tile; a single stage (K = 256); several K slices
    assert _plan(M, N, K)["kernel"] == wq.WQ_KERNEL_DECODE
    p = Fp4Problem(M, N, K, seed=610 + M)
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what=f"fp4 decode M={M} N={N} K={K}")


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_fp4_decode_every_token_count(M):
    p = Fp4Problem(M, 256, 1024, seed=630 + M)
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what=f"fp4 decode M={M}")


def test_fp4_decode_largest_cluster_deterministic():
    # two weight tiles and 64 stages: K split over the largest cluster the device holds
    M, N, K = 16, 256, 16384
    plan = _plan(M, N, K)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] >= 8
    p = Fp4Problem(M, N, K, seed=650)
    first = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(first), p.ref(), out_dtype="bf16", what=f"fp4 decode S={plan['splits']}")
    for _ in range(5):
        assert torch.equal(p.run(), first)


def test_fp4_decode_nan_scale_propagates():
    # an e4m3 NaN block scale makes its weights NaN: output columns of that row are NaN
    # for every token, the others are unaffected
    M, N, K = 4, 256, 1024
    p = Fp4Problem(M, N, K, seed=660)
    p.wts.sf[77, 9] = 0x7F
    p.sf_d = torch.from_numpy(p.wts.sf).to(DEV)
    p.sfk = wq.wq_pack_fp4_sf(p.sf_d, N, K)
    out = out_to_f64(p.run())
    torch.cuda.synchronize()
    ref = p.ref()
    assert np.isnan(ref[:, 77]).all() and np.isnan(out[:, 77]).all()
    keep = np.setdiff1d(np.arange(N), [77])
    assert not np.isnan(out[:, keep]).any()
    check_close(out[:, keep], ref[:, keep], out_dtype="bf16", what="fp4 NaN scale")
