"""GPU parity of the FP8 (W8A16) and BF16 x FP4 paths against the float64 oracle.

Besides the absolute bar, both formats must be no less accurate than the cast-copy
path that materialises a 16-bit weight and calls a dense GEMM ("FlashInfer W8A16
GEMM (mm_bf16_fp8) analysis", introduction and §5: the accuracy gate compares the
kernel's error with the cast-copy path's own error against the same reference).
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, Fp4Problem, Fp8Problem, check_close, out_bits, out_to_f64, to_dev_f16bits

pytestmark = pytest.mark.gpu

BF16_ULP_REL = 2.0 ** -8   # one bf16 ulp relative to a value in [1, 2): tie slack for rel_max


def _cast_copy_fp8(A_d, w_codes_d, scale, out_dtype):
    # the cast-copy path: w16 = weight.to(dtype) * scale.to(dtype); out = A . w16^T
    w16 = w_codes_d.view(torch.float8_e4m3fn).to(out_dtype) * torch.tensor(scale, dtype=torch.float32).to(out_dtype)
    return torch.nn.functional.linear(A_d, w16)


def _cast_copy_fp4(A_d, w_h, sf_h, alpha):
    # e2m1 and e4m3 decoded by the library-independent oracle tables, then the same
    # materialise-then-GEMM recipe with alpha folded into the 16-bit weight
    N, K = w_h.shape[0], w_h.shape[1] * 2
    e2m1 = np.array([oracle.e2m1_to_double(c) for c in range(16)], dtype=np.float32)
    lo, hi = w_h & 0xF, w_h >> 4
    codes = np.empty((N, K), dtype=np.uint8)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    wv = torch.from_numpy(e2m1[codes]).to(DEV).to(torch.bfloat16)
    sfv = torch.from_numpy(sf_h).to(DEV).view(torch.float8_e4m3fn).to(torch.bfloat16)
    w16 = (wv * sfv.repeat_interleave(16, dim=1)) * torch.tensor(alpha, dtype=torch.float32).to(torch.bfloat16)
    return torch.nn.functional.linear(A_d, w16)


def _gate_vs_cast_copy(got, cast, ref, what):
    # absolute bar (bf16 outputs: mean error against the correctly rounded reference),
    # then no worse than the cast-copy path against the same float64 reference
    check_close(got, ref, out_dtype="bf16", what=what)
    k_max, k_mean = oracle.rel_errors(got, ref)
    c_max, c_mean = oracle.rel_errors(cast, ref)
    assert k_mean <= c_mean, f"{what}: kernel rel_mean {k_mean:.3e} > cast-copy {c_mean:.3e}"
    assert k_max <= c_max + BF16_ULP_REL * 0.5, f"{what}: kernel rel_max {k_max:.3e} > cast-copy {c_max:.3e}"
    return (k_max, k_mean), (c_max, c_mean)


# ------------------------------------------------------------------ FP8

@pytest.mark.parametrize("bf16", [True, False])
def test_fp8_debug_dequant_bit_exact(bf16):
    codes = np.arange(256, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0       # NaN codes are never produced by the input recipe
    w = np.tile(codes, (64, 4))              # [64, 1024]
    got = wq.wq_debug_dequant_fp8(torch.from_numpy(w).to(DEV), operand_bf16=bf16).cpu().numpy()
    want = oracle.dequant_fp8(w)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("a_dtype", ["bf16", "f16"])
def test_fp8_identity_A_bit_exact(a_dtype):
    K, N = 256, 256
    eye = np.eye(K, dtype=np.float32)
    p = Fp8Problem(K, N, K, a_dtype=a_dtype, seed=201)
    p.A = synth._to_bits(eye, a_dtype)
    p.A_d = to_dev_f16bits(p.A, a_dtype)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    out = p.run(alpha=one)
    torch.cuda.synchronize()
    w = oracle.dequant_fp8(p.wts.w).astype(np.float64)
    rn = oracle.round_bf16_array(w.T) if a_dtype == "bf16" else oracle.round_f16_array(w.T)
    assert np.array_equal(out_bits(out), rn)


@pytest.mark.parametrize("case", synth.FP8, ids=lambda c: f"M{c.M}_N{c.N}_K{c.K}")
def test_fp8_configs(case):
    p = Fp8Problem(case.M, case.N, case.K, seed=synth.seed_for(3, synth.FP8.index(case)))
    out = p.run()
    cast = _cast_copy_fp8(p.A_d, p.w_d, p.wts.scale, torch.bfloat16)
    torch.cuda.synchronize()
    rows = synth.sample_rows(case.M, 256, seed=202)   # every row when M <= 256
    ref = p.ref(rows=rows)
    _gate_vs_cast_copy(out_to_f64(out)[rows], out_to_f64(cast)[rows], ref, f"fp8 {case}")


@pytest.mark.parametrize("M", [1, 5, 16, 40, 128, 300])
def test_fp8_fp16_activations_and_bias(M):
    p = Fp8Problem(M, 1024, 2048, a_dtype="f16", seed=203 + M, with_bias=True)
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="f16", what=f"fp8 f16+bias M={M}")


def test_fp8_alpha_at_odd_word_address():
    # the per-tensor scale needs only 4-byte alignment (address % 16 == 4 accepted)
    p = Fp8Problem(4, 512, 1024, seed=204)
    holder = torch.zeros(8, dtype=torch.float32, device=DEV)
    holder[1] = float(p.wts.scale)
    alpha = holder[1:2]
    assert alpha.data_ptr() % 16 == 4
    out = p.run(alpha=alpha)
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what="fp8 alpha%16==4")


@pytest.mark.parametrize("N,K", [(136, 80), (8, 16), (264, 1040)])
def test_fp8_ragged(N, K):
    p = Fp8Problem(3, N, K, seed=205)
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what=f"fp8 N={N} K={K}")


def test_fp8_split_k_deterministic():
    p = Fp8Problem(16, 10240, 5120, seed=206)
    first = out_bits(p.run())
    for _ in range(10):
        assert np.array_equal(out_bits(p.run()), first)


# ------------------------------------------------------------------ FP4

@pytest.mark.parametrize("N,K", [(128, 512), (200, 160), (256, 5120)])
def test_fp4_debug_dequant_bit_exact(N, K):
    p = Fp4Problem(1, N, K, seed=301)
    got = wq.wq_debug_dequant_fp4(p.w_d, p.sfk, N, K).cpu().numpy()
    want = oracle.dequant_fp4(p.wts.w, p.wts.sf, K)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fp4_identity_A_bit_exact():
    K, N = 256, 384
    p = Fp4Problem(K, N, K, seed=302)
    p.A = synth._to_bits(np.eye(K, dtype=np.float32), "bf16")
    p.A_d = to_dev_f16bits(p.A, "bf16")
    p.alpha = torch.ones(1, dtype=torch.float32, device=DEV)
    out = p.run()
    torch.cuda.synchronize()
    w = oracle.dequant_fp4(p.wts.w, p.wts.sf, K).astype(np.float64)
    # values, not bits: a -0 weight plus +0 products sums to +0
    assert np.array_equal(out_to_f64(out), w.T)


@pytest.mark.parametrize("case", synth.FP4, ids=lambda c: f"M{c.M}")
def test_fp4_configs(case):
    p = Fp4Problem(case.M, case.N, case.K, seed=synth.seed_for(4, synth.FP4.index(case)))
    out = p.run()
    cast = _cast_copy_fp4(p.A_d, p.wts.w, p.wts.sf, float(p.wts.alpha))
    torch.cuda.synchronize()
    rows = synth.sample_rows(case.M, 256, seed=303)   # every row when M <= 256
    ref = p.ref(rows=rows)
    _gate_vs_cast_copy(out_to_f64(out)[rows], out_to_f64(cast)[rows], ref, f"fp4 {case}")


@pytest.mark.parametrize("M,N,K", [(1, 8, 32), (7, 136, 160), (33, 520, 1056), (200, 256, 512)])
def test_fp4_ragged(M, N, K):
    p = Fp4Problem(M, N, K, seed=304)
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what=f"fp4 M={M} N={N} K={K}")


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_gives_up_and_reports():
    # a wait on a barrier nothing arrives on runs out after ~1 ms; the kernel sets a
    # status bit and returns, and the context stays usable
    wq.wq_clear_device_status()
    wq.wq_debug_wait_probe(1_000_000)
    torch.cuda.synchronize()
    assert wq.wq_device_status() & (1 << 5)
    wq.wq_clear_device_status()
    assert wq.wq_device_status() == 0
    p = Fp8Problem(2, 256, 512, seed=305)
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what="after probe")


# ------------------------------------------------------- large M: pair and one-CTA kernels

@pytest.fixture(params=["pair", "one_cta"])
def tile_kernel(request, monkeypatch):
    """The large-M tile kernel under test: two-CTA pair (default) or one CTA per tile."""
    if request.param == "one_cta":
        monkeypatch.setenv("WQ_DISABLE_PAIR", "1")
    else:
        monkeypatch.delenv("WQ_DISABLE_PAIR", raising=False)
    return wq.WQ_KERNEL_TILE_PAIR if request.param == "pair" else wq.WQ_KERNEL_TILE


@pytest.mark.parametrize("a_dtype", ["bf16", "f16"])
def test_fp8_large_M_identity_bit_exact(a_dtype, tile_kernel):
    # M = K = 1024 tokens of identity over 80 weight tiles (40 pair tiles): out = RN(w),
    # through the staged epilogue on the pair kernel.  Compared as values: a weight of
    # e4m3 -0 yields +0 (its product plus the +0 products of the other tokens)
    M = K = 1024
    N = 10240
    plan = wq.get_plan(wq.WQ_OP_FP8, wq.WQ_F16 if a_dtype == "f16" else wq.WQ_BF16, M, N, K, 0)
    assert plan["kernel"] == tile_kernel
    p = Fp8Problem(M, N, K, a_dtype=a_dtype, seed=210)
    p.A = synth._to_bits(np.eye(K, dtype=np.float32), a_dtype)
    p.A_d = to_dev_f16bits(p.A, a_dtype)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    out = p.run(alpha=one)
    torch.cuda.synchronize()
    w = oracle.dequant_fp8(p.wts.w).astype(np.float64).T
    want = oracle.bf16_bits_to_double_array(oracle.round_bf16_array(w)) if a_dtype == "bf16" else \
        oracle.f16_bits_to_double_array(oracle.round_f16_array(w))
    assert np.array_equal(out_to_f64(out), want)


def test_fp8_large_M_fp16_with_bias(tile_kernel):
    M, N, K = 2100, 3200, 2048
    plan = wq.get_plan(wq.WQ_OP_FP8, wq.WQ_F16, M, N, K, 0)
    assert plan["kernel"] == tile_kernel
    p = Fp8Problem(M, N, K, a_dtype="f16", seed=215, with_bias=True)
    out = p.run()
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([synth.sample_rows(M, 64, seed=216), np.arange(M - 20, M)]))
    check_close(out_to_f64(out)[rows], p.ref(rows=rows), out_dtype="f16", what="fp8 f16 + bias, large M")


def test_fp8_large_M_random(tile_kernel):
    M, N, K = 2100, 3200, 5120
    plan = wq.get_plan(wq.WQ_OP_FP8, wq.WQ_BF16, M, N, K, 0)
    assert plan["kernel"] == tile_kernel
    p = Fp8Problem(M, N, K, seed=211)
    out = p.run()
    cast = _cast_copy_fp8(p.A_d, p.w_d, p.wts.scale, torch.bfloat16)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([synth.sample_rows(M, 64, seed=212), np.arange(M - 20, M)]))
    _gate_vs_cast_copy(out_to_f64(out)[rows], out_to_f64(cast)[rows], p.ref(rows=rows), "fp8 large M")


def test_fp4_large_M(tile_kernel):
    M, N, K = 2100, 4224, 2048
    plan = wq.get_plan(wq.WQ_OP_FP4, wq.WQ_BF16, M, N, K, 0)
    assert plan["kernel"] == tile_kernel
    p = Fp4Problem(M, N, K, seed=213)
    out = p.run()
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([synth.sample_rows(M, 64, seed=214), np.arange(M - 20, M)]))
    check_close(out_to_f64(out)[rows], p.ref(rows=rows), out_dtype="bf16", what="fp4 large M")
