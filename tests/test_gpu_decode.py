"""GPU parity of the W4A16 decode kernel (M <= 16, K % 64 == 0) against the oracle.

The decode kernel forms s * sum_k A (b + q) - s (b + 8) sum_k A per group in fp32
instead of rounding (q - 8) * s to the activation type, so its checks are the same
tolerance bar as the tile kernel plus exact cases where every sum is exact.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, Int4Problem, check_close, out_bits, out_to_f64

pytestmark = pytest.mark.gpu

# K per group size: the G <= 64 cases end on a half k-block (K % 128 == 64), so the
# last activation copy reads one 64-wide box past K (zero fill)
K_FOR_G = {32: 1088, 64: 1088, 128: 1280, 256: 1536}


def _dt(a_dtype):
    return wq.WQ_F16 if a_dtype == "f16" else wq.WQ_BF16


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
@pytest.mark.parametrize("M", [1, 5, 8, 9, 16])
def test_decode_group_sizes(M, G, a_dtype):
    N, K = 384, K_FOR_G[G]
    plan = wq.get_plan(wq.WQ_OP_W4A16, _dt(a_dtype), M, N, K, G)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE
    p = Int4Problem(M, N, K, G, a_dtype=a_dtype, seed=200 + M + G).pack()
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype=a_dtype, what=f"decode M={M} G={G} {a_dtype}")


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 128, 256])
@pytest.mark.parametrize("M", [1, 7, 16])
def test_decode_identity_rows_bit_exact(M, G, a_dtype):
    # A[m, k] = 1 at one k per token (spread over several groups and k-blocks), else
    # 0: out[m, n] = RN((q[n, k_m] - 8) * s) exactly, whatever the summation order
    N, K = 256, 2048
    ks = [(m * 613 + 37) % K for m in range(M)]
    A = np.zeros((M, K), dtype=np.float32)
    A[np.arange(M), ks] = 1.0
    bits = A.astype(np.float16).view(np.uint16) if a_dtype == "f16" else \
        torch.from_numpy(A).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    p = Int4Problem(M, N, K, G, a_dtype=a_dtype, seed=210, A_bits=bits).pack()
    out = p.run()
    torch.cuda.synchronize()
    w = oracle.dequant_int4(p.wts.w, p.wts.s, K, G).astype(np.float64)   # [N, K]
    want = w[:, ks].T
    rn = oracle.round_f16_array(want) if a_dtype == "f16" else oracle.round_bf16_array(want)
    assert np.array_equal(out_bits(out), rn)


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_decode_every_token_count(M):
    # every M in 1..16: the activation boxes hold exactly M rows, one or two
    # 8-token column tiles
    N, K, G = 256, 1024, 128
    p = Int4Problem(M, N, K, G, seed=220 + M).pack()
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), what=f"M={M}")


def test_decode_integer_problem_is_exact_bf16():
    # bf16 operand: b + q = 128 + q exact; with A in {-1, 0, 1} and s = 0.25 every
    # sum is an exact small multiple of 0.25, exact in bf16 when |out| < 64
    M, N, K, G = 16, 256, 512, 32
    rng = np.random.Generator(np.random.PCG64(230))
    Af = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    Af[:, 8:] = 0.0                                   # 8 non-zero terms: |out| <= 8 * 8 * 0.25
    wts = synth.int4_weights(N, K, G, seed=231)
    wts.s[:] = np.float16(0.25).view(np.uint16)
    bits = torch.from_numpy(Af).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    p = Int4Problem(M, N, K, G, a_dtype="bf16", A_bits=bits, wts=wts).pack()
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_to_f64(out), p.ref())


def test_decode_not_used_when_K_is_not_a_multiple_of_64():
    plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, 4, 512, 1056, 32)
    assert plan["kernel"] == wq.WQ_KERNEL_TILE
    plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, 17, 512, 1024, 128)
    assert plan["kernel"] == wq.WQ_KERNEL_TILE


def test_decode_back_to_back_calls_overlap_safely():
    # consecutive decode GEMMs on one stream start before their predecessor ends
    # (programmatic dependent launch); each must still see its own inputs and leave
    # the shared workspace counters zero
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=DEV)
    probs = [Int4Problem(M, N, K, 128, seed=240 + i).pack()
             for i, (M, N, K) in enumerate([(1, 4096, 4096), (16, 4096, 11008), (4, 11008, 4096), (16, 512, 512)])]
    outs = [None] * len(probs)
    for _ in range(3):
        for i, p in enumerate(probs):
            outs[i] = p.run(ws=ws)
    torch.cuda.synchronize()
    for p, out in zip(probs, outs):
        check_close(out_to_f64(out), p.ref(), what=f"chained M={p.M} N={p.N} K={p.K}")
    assert int(ws[:16384].count_nonzero()) == 0
