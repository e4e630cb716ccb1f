"""GPU parity of the INT2 (W2A16) decode kernel (M <= 16, G >= 64, K % 256 == 0).

The kernel reads the canonical 2-bit codes through TMA, forms q - 2 exactly in
registers and applies each group's scale to the fp32 sums, so an output is one
rounding of sum_g s_g * sum_{k in g} A (q - 2).  Its lanes hold codes 16c .. 16c + 15
of a 64-code chunk and each of the chunk's four MMA k steps takes codes 16c + 4t ..
16c + 4t + 3 from every lane; the one-hot tests pin that reordering (every position of
a chunk, chunks across stages and K slices) and the per-group scales.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import Int2Problem, check_close, out_bits, out_to_f64

pytestmark = pytest.mark.gpu


def _adt(a_dtype):
    return wq.WQ_BF16 if a_dtype == "bf16" else wq.WQ_F16


def _plan(M, N, K, G, a_dtype="f16"):
    return wq.get_plan(wq.WQ_OP_W2A16, _adt(a_dtype), M, N, K, G)


def _one_hot_bits(ks, K, a_dtype):
    A = np.zeros((len(ks), K), dtype=np.float32)
    A[np.arange(len(ks)), ks] = 1.0
    return synth._to_bits(A, a_dtype)


def _rn(w, a_dtype):
    w = w.astype(np.float64)
    return oracle.round_f16_array(w) if a_dtype == "f16" else oracle.round_bf16_array(w)


def test_int2_decode_plan():
    for M in (1, 8, 16):
        for G in (64, 128, 256):
            plan = _plan(M, 4096, 4096, G)
            assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["bk"] == 256 and plan["ws_bytes"] == 0
    assert _plan(16, 4096, 4096, 128, "bf16")["kernel"] == wq.WQ_KERNEL_DECODE
    assert _plan(16, 4096, 4096, 32)["kernel"] == wq.WQ_KERNEL_TILE      # G = 32
    assert _plan(17, 4096, 4096, 128)["kernel"] == wq.WQ_KERNEL_TILE     # M = 17
    assert _plan(4, 4096, 4160, 64)["kernel"] == wq.WQ_KERNEL_TILE       # K % 256 == 64


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [64, 128, 256])
@pytest.mark.parametrize("shift", [0, 1, 2, 3])
def test_int2_decode_one_hot_bit_exact(shift, G, a_dtype):
    # token m selects k_m: over the four shifts the 16 tokens cover all 64 positions of a
    # 64-code chunk (every lane's bytes and every code of a byte), with chunks spread over
    # stages and K slices; out[m, n] = RN((q[n, k_m] - 2) * s) exactly (one product)
    M, N, K = 16, 392, 4096
    ks = [64 * ((7 * m + 3 * shift) % (K // 64)) + (m + 16 * shift) % 64 for m in range(M)]
    p = Int2Problem(M, N, K, G, a_dtype=a_dtype, seed=800 + shift + G, A_bits=_one_hot_bits(ks, K, a_dtype))
    plan = _plan(M, N, K, G, a_dtype)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] > 1
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), _rn(p.dequant_ref()[:, ks].T, a_dtype))


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_int2_decode_every_token_count(M):
    a_dtype = "bf16" if M % 2 else "f16"
    p = Int2Problem(M, 256, 1024, 128, a_dtype=a_dtype, seed=820 + M)
    assert _plan(M, 256, 1024, 128, a_dtype)["kernel"] == wq.WQ_KERNEL_DECODE
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype=a_dtype, what=f"int2 decode M={M}")


@pytest.mark.parametrize("M,N,K,G", [(1, 1000, 4352, 64), (7, 136, 1280, 256), (16, 11008, 4096, 128),
                                     (3, 264, 256, 64), (16, 256, 16384, 128), (9, 4096, 11008 // 43 * 43, 128)])
def test_int2_decode_ragged_and_deterministic(M, N, K, G):
    # tail rows, a single stage, the largest cluster; repeated calls give the same bits
    if K % 256 or K % G:
        pytest.skip("shape outside the decode kernel's range")
    p = Int2Problem(M, N, K, G, seed=840 + M + K)
    assert _plan(M, N, K, G)["kernel"] == wq.WQ_KERNEL_DECODE
    wq.wq_clear_device_status()
    first = p.run()
    torch.cuda.synchronize()
    assert wq.wq_device_status() == 0
    check_close(out_to_f64(first), p.ref(), what=f"int2 decode M={M} N={N} K={K} G={G}")
    for _ in range(3):
        assert torch.equal(p.run(), first)


def test_int2_decode_back_to_back_calls():
    # consecutive decode GEMMs on one stream (programmatic dependent launch): each reads
    # its own inputs after the preceding kernel
    probs = [Int2Problem(M, N, K, G, seed=860 + i) for i, (M, N, K, G) in
             enumerate([(1, 4096, 4096, 128), (16, 1024, 2048, 64), (5, 1000, 4352, 256), (16, 512, 512, 128)])]
    outs = [None] * len(probs)
    for _ in range(3):
        for i, p in enumerate(probs):
            outs[i] = p.run()
    torch.cuda.synchronize()
    for p, out in zip(probs, outs):
        check_close(out_to_f64(out), p.ref(), what=f"chained int2 M={p.M} N={p.N} K={p.K}")
