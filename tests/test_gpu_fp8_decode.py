"""GPU parity of the FP8 decode kernel (M <= 32, K % 64 == 0) against the oracle.

The decode kernel reads the plain e4m3 codes, converts them to the activation type
in registers (exact) and sums in fp32, with alpha and the bias applied once in the
epilogue.  Its lanes hold the codes k = 4c .. 4c + 3 of each 16-wide k step in the
MMA fragment positions 2c, 2c + 1, 2c + 8, 2c + 9; the one-hot tests below pin that
reordering (a wrong pairing of weight and activation positions moves the selected
weight) and the split-K slices (every k step of every stage is selected by some token).
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, Fp8Problem, check_close, out_to_f64, to_dev_f16bits

pytestmark = pytest.mark.gpu


def _dt(a_dtype):
    return wq.WQ_F16 if a_dtype == "f16" else wq.WQ_BF16


def _one_hot(ks, K, a_dtype):
    A = np.zeros((len(ks), K), dtype=np.float32)
    A[np.arange(len(ks)), ks] = 1.0
    return synth._to_bits(A, a_dtype)


def test_fp8_decode_plan():
    for M in (1, 16, 17, 32):
        plan = wq.get_plan(wq.WQ_OP_FP8, wq.WQ_BF16, M, 10240, 5120, 0)
        assert plan["kernel"] == wq.WQ_KERNEL_DECODE
        assert plan["ws_bytes"] == 0 and plan["tiles_m"] == 1
    assert wq.get_plan(wq.WQ_OP_FP8, wq.WQ_BF16, 33, 10240, 5120, 0)["kernel"] == wq.WQ_KERNEL_TILE
    assert wq.get_plan(wq.WQ_OP_FP8, wq.WQ_F16, 4, 1024, 1040, 0)["kernel"] == wq.WQ_KERNEL_TILE


@pytest.mark.parametrize("a_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shift", [0, 5, 11])
def test_fp8_decode_one_hot_bit_exact(a_dtype, shift):
    # token m selects k_m: the 16 tokens cover every position inside a 16-wide k step
    # and steps spread over all stages and K slices; out[m, n] = e4m3(W[n, k_m])
    # exactly (alpha = 1, no bias; every e4m3 value is exact in fp16 and bf16)
    M, N, K = 16, 392, 2048
    ks = [16 * ((7 * m + 3 * shift) % (K // 16)) + (m + shift) % 16 for m in range(M)]
    assert sorted(k % 16 for k in ks) == list(range(16))
    p = Fp8Problem(M, N, K, a_dtype=a_dtype, seed=400 + shift)
    plan = wq.get_plan(wq.WQ_OP_FP8, _dt(a_dtype), M, N, K, 0)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] > 1
    p.A = _one_hot(ks, K, a_dtype)
    p.A_d = to_dev_f16bits(p.A, a_dtype)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    out = p.run(alpha=one)
    torch.cuda.synchronize()
    w = oracle.dequant_fp8(p.wts.w).astype(np.float64)   # [N, K]
    assert np.array_equal(out_to_f64(out), w[:, ks].T)


@pytest.mark.parametrize("M", [1, 4, 24, 40])
def test_fp8_nan_codes_propagate(M):
    # e4m3 S.1111.111 is NaN: a NaN code in weight row n makes column n of the output
    # NaN for every token (0 * NaN = NaN), on the decode kernel (M <= 32) and the tile
    # kernel alike; the other columns are unaffected
    N, K = 256, 1024
    p = Fp8Problem(M, N, K, seed=410)
    bad = {3: [5], 130: [640, 1023], 255: [64]}
    for n, kk in bad.items():
        for i, k in enumerate(kk):
            p.wts.w[n, k] = 0x7F if i % 2 == 0 else 0xFF
    p.w_d = torch.from_numpy(p.wts.w).to(DEV)
    kernel = wq.get_plan(wq.WQ_OP_FP8, wq.WQ_BF16, M, N, K, 0)["kernel"]
    assert kernel == (wq.WQ_KERNEL_DECODE if M <= 32 else wq.WQ_KERNEL_TILE)
    out = out_to_f64(p.run())
    torch.cuda.synchronize()
    ref = p.ref()
    cols = sorted(bad)
    assert np.isnan(ref[:, cols]).all()
    assert np.isnan(out[:, cols]).all()
    keep = np.setdiff1d(np.arange(N), cols)
    assert not np.isnan(out[:, keep]).any()
    check_close(out[:, keep], ref[:, keep], out_dtype="bf16", what=f"fp8 NaN rows M={M}")


@pytest.mark.parametrize("N,K", [(136, 1088), (264, 192), (1000, 4160)])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_fp8_decode_ragged(M, N, K):
    # tail rows in the last 128-row tile; K % 128 == 64 puts the last stage half past
    # K (zero fill); fp16 activations with a bias on odd M
    a_dtype = "f16" if M % 2 else "bf16"
    p = Fp8Problem(M, N, K, a_dtype=a_dtype, seed=420 + M, with_bias=M % 2 == 1)
    assert wq.get_plan(wq.WQ_OP_FP8, _dt(a_dtype), M, N, K, 0)["kernel"] == wq.WQ_KERNEL_DECODE
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype=a_dtype, what=f"fp8 decode M={M} N={N} K={K}")


@pytest.mark.parametrize("a_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shift", [0, 1])
@pytest.mark.parametrize("M", [24, 32])
def test_fp8_decode_one_hot_wide(M, shift, a_dtype):
    # 4 token tiles: every token selects its own k, so a wrong token <-> column or
    # inbox-slot mapping for tiles 2 and 3 moves outputs between rows of the result
    N, K = 392, 2048
    ks = [16 * ((11 * m + 5 * shift) % (K // 16)) + (m + 3 * shift) % 16 for m in range(M)]
    p = Fp8Problem(M, N, K, a_dtype=a_dtype, seed=470 + M + shift)
    plan = wq.get_plan(wq.WQ_OP_FP8, _dt(a_dtype), M, N, K, 0)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] > 1
    p.A = _one_hot(ks, K, a_dtype)
    p.A_d = to_dev_f16bits(p.A, a_dtype)
    out = p.run(alpha=torch.ones(1, dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    w = oracle.dequant_fp8(p.wts.w).astype(np.float64)
    assert np.array_equal(out_to_f64(out), w[:, ks].T)


@pytest.mark.parametrize("M", list(range(17, 33)))
def test_fp8_decode_wide_ragged(M):
    # 17-32 tokens: 4 token tiles; tail rows (N = 1000) and a half-stage K tail
    a_dtype = "f16" if M % 2 else "bf16"
    N, K = 1000, 4160
    p = Fp8Problem(M, N, K, a_dtype=a_dtype, seed=480 + M, with_bias=M % 3 == 0)
    assert wq.get_plan(wq.WQ_OP_FP8, _dt(a_dtype), M, N, K, 0)["kernel"] == wq.WQ_KERNEL_DECODE
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype=a_dtype, what=f"fp8 decode M={M}")


@pytest.mark.parametrize("M", [20, 32])
def test_fp8_decode_wide_deterministic(M):
    p = Fp8Problem(M, 2048, 8192, seed=490 + M)
    first = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(first), p.ref(), out_dtype="bf16", what=f"fp8 decode M={M}")
    for _ in range(3):
        assert torch.equal(p.run(), first)


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_fp8_decode_every_token_count(M):
    p = Fp8Problem(M, 256, 1024, seed=440 + M)
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what=f"fp8 decode M={M}")


def test_fp8_decode_largest_cluster():
    # two weight tiles and 128 k-blocks: the plan splits K over the largest cluster the
    # device holds (up to 16 CTAs), the deepest in-cluster reduction
    M, N, K = 16, 256, 16384
    plan = wq.get_plan(wq.WQ_OP_FP8, wq.WQ_BF16, M, N, K, 0)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] >= 8
    p = Fp8Problem(M, N, K, seed=450, with_bias=True)
    first = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(first), p.ref(), out_dtype="bf16", what=f"fp8 decode S={plan['splits']}")
    for _ in range(5):
        assert torch.equal(p.run(), first)


def test_fp8_decode_back_to_back_calls():
    # consecutive decode GEMMs on one stream overlap their prologues with the
    # predecessor's tail (programmatic dependent launch); each reads its own inputs
    probs = [Fp8Problem(M, N, K, seed=460 + i, with_bias=i % 2 == 1)
             for i, (M, N, K) in enumerate([(1, 10240, 5120), (16, 4096, 1024), (7, 1000, 4160), (16, 512, 512)])]
    outs = [None] * len(probs)
    for _ in range(3):
        for i, p in enumerate(probs):
            outs[i] = p.run()
    torch.cuda.synchronize()
    for p, out in zip(probs, outs):
        check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what=f"chained fp8 M={p.M} N={p.N} K={p.K}")
