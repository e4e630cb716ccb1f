"""Pins for the float64 CPU oracle: checks against things other than itself.

Each test ties one oracle function to the pages' worked meaning, a number-format
definition cross-checked by a library routine, a closed form, an invariant, or a
brute-force loop on tiny inputs.  The selection is made so that a plausible slip
anywhere in the oracle (a nibble order, the -8 offset, a transposed scale index,
a block-scale stride, an exponent bias, a tie rule, a dropped alpha) fails at
least one of them; tests/test_oracle_mutations.py plants such slips and checks.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_tma_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f16_bits(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


# ------------------------------------------------------------- number formats

def test_f16_decode_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_double_array(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zero is kept
    assert math.copysign(1.0, oracle.f16_to_double(0x8000)) == -1.0


def test_bf16_decode_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_bits_to_double_array(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_e4m3_decode_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = np.array([oracle.e4m3_to_double(c) for c in codes])
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # anchors of the OCP definition: max normal, min normal, min subnormal
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9


# OCP MX E2M1 magnitudes for codes 0..7 (sign in bit 3).
_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table():
    for c in range(16):
        mag = _E2M1[c & 7]
        v = oracle.e2m1_to_double(c)
        assert v == (-mag if c & 8 else mag)
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_e2m1_decode_vs_torch_if_available():
    dt = getattr(torch, "float4_e2m1fn_x2", None)
    if dt is None:
        pytest.skip("torch has no float4_e2m1fn_x2")
    packed = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    try:
        # unpack two codes per byte into float via the library's own decoder
        as_f4 = packed.view(dt)
        vals = as_f4.to(torch.float32)
    except Exception as exc:  # conversion not implemented on CPU in this build
        pytest.skip(f"float4_e2m1fn_x2 conversion unavailable: {exc}")
    if vals.numel() != 512:
        pytest.skip("unexpected float4 conversion shape")
    vals = vals.reshape(256, 2).numpy()
    for b in range(256):
        lo, hi = b & 0xF, b >> 4
        assert vals[b, 0] == oracle.e2m1_to_double(lo)
        assert vals[b, 1] == oracle.e2m1_to_double(hi)


def test_round_f16_vs_numpy():
    rng = np.random.Generator(np.random.PCG64(7))
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                  2048.0 + 1.0, 2048.0 + 3.0, 1e-30, -1e-30]),
    ])
    got = oracle.round_f16_array(x)
    want = x.astype(np.float16).view(np.uint16)   # numpy rounds float64 -> fp16 directly (RNE)
    assert np.array_equal(got, want)


def test_round_bf16_vs_torch_on_float32_values():
    # torch rounds float32 -> bf16 with RNE; feeding float32-representable values
    # avoids any double rounding on torch's side.
    rng = np.random.Generator(np.random.PCG64(8))
    x32 = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000)).astype(np.float32),
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 2.0 ** -133, 2.0 ** -134, 3.0e38],
                 dtype=np.float32),
    ])
    got = oracle.round_bf16_array(x32.astype(np.float64))
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_round_ties_to_even():
    # 1 + 2^-11 is the midpoint between 1 and 1 + 2^-10: even mantissa wins (1.0)
    assert oracle.round_f16(1.0 + 2.0 ** -11) == 0x3C00
    # 1 + 3*2^-11 lies between 1+2^-10 (odd) and 1+2^-9 (even): rounds up
    assert oracle.round_f16(1.0 + 3 * 2.0 ** -11) == 0x3C02
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82


# ------------------------------------------------------------- INT4

@pytest.mark.parametrize("name", ["int4_worked_example_1.json", "int4_worked_example_2.json"])
def test_int4_worked_examples(name):
    g = _golden(name)
    M, N, K, G = g["M"], g["N"], g["K"], g["G"]
    q = np.array(g["q"], dtype=np.uint8)
    packed = oracle.pack_int4(q)
    assert packed.tolist() == g["packed"]
    assert np.array_equal(oracle.unpack_int4(packed, K), q)
    s = _f16_bits(g["scales"])
    w = oracle.dequant_int4(packed, s, K, G)
    assert w.tolist() == g["w"]
    A = _f16_bits(g["A"])
    out = oracle.gemm_w4a16(A, False, packed, s, M, N, K, G)
    assert out.tolist() == g["out"]
    # the bf16 path of the oracle reads the same values when they are exact in bf16
    A_bf = torch.tensor(g["A"], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert oracle.gemm_w4a16(A_bf, True, packed, s, M, N, K, G).tolist() == g["out"]


def test_int4_pack_roundtrip_random():
    rng = np.random.Generator(np.random.PCG64(11))
    q = rng.integers(0, 16, size=(37, 256), dtype=np.uint8)
    packed = oracle.pack_int4(q)
    assert np.array_equal(oracle.unpack_int4(packed, 256), q)
    # the canonical layout: low nibble is the even k
    assert np.array_equal(packed & 0xF, q[:, 0::2])
    assert np.array_equal(packed >> 4, q[:, 1::2])


def test_int4_dequant_against_closed_form():
    wts = synth.int4_weights(64, 512, 128, seed=12)
    q = oracle.unpack_int4(wts.w, 512).astype(np.int64)
    s = wts.s.view(np.float16).astype(np.float64)          # numpy decodes the fp16 scales
    g_of_k = np.arange(512) // 128
    want = (q - 8) * s[g_of_k, :].T                          # [N, K]
    got = oracle.dequant_int4(wts.w, wts.s, 512, 128)
    assert np.array_equal(got.astype(np.float64), want)      # exact in fp32


@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_int4_identity_A_returns_dequantized_weight(G):
    K = 256
    wts = synth.int4_weights(24, K, G, seed=13)
    A = _f16_bits(np.eye(K, dtype=np.float32))
    out = oracle.gemm_w4a16(A, False, wts.w, wts.s, K, 24, K, G)
    w = oracle.dequant_int4(wts.w, wts.s, K, G).astype(np.float64)
    assert np.array_equal(out, w.T)


def _brute_force_int4(A16, w_packed, s16, M, N, K, G):
    """Independent pure-Python triple loop (numpy only decodes fp16)."""
    A = A16.view(np.float16).astype(np.float64)
    S = s16.view(np.float16).astype(np.float64)
    out = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                byte = int(w_packed[n, k // 2])
                code = (byte >> 4) if (k & 1) else (byte & 15)
                acc += float(A[m, k]) * ((code - 8) * float(S[k // G, n]))
            out[m][n] = acc
    return np.array(out)


@pytest.mark.parametrize("M,N,K,G", [(1, 8, 64, 32), (3, 5, 128, 64), (4, 8, 256, 128)])
def test_int4_gemm_vs_brute_force(M, N, K, G):
    A = synth.activations(M, K, "f16", seed=14)
    wts = synth.int4_weights(N, K, G, seed=15)
    got = oracle.gemm_w4a16(A, False, wts.w, wts.s, M, N, K, G)
    want = _brute_force_int4(A, wts.w, wts.s, M, N, K, G)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_int4_row_and_column_subsets():
    M, N, K, G = 9, 20, 256, 64
    A = synth.activations(M, K, "f16", seed=16)
    wts = synth.int4_weights(N, K, G, seed=17)
    full = oracle.gemm_w4a16(A, False, wts.w, wts.s, M, N, K, G)
    rows, cols = [0, 4, 8], [19, 3, 0, 7]
    sub = oracle.gemm_w4a16(A, False, wts.w, wts.s, M, N, K, G, rows=rows, cols=cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])


def test_int4_statistical_magnitude():
    # E[w^2] = E[(q-8)^2] E[s^2] with q uniform on 0..15 and s ~ U[0.005, 0.02];
    # with A ~ N(0,1) the outputs have std sqrt(K E[w^2]).
    M, N, K, G = 8, 256, 4096, 128
    A = synth.activations(M, K, "f16", seed=18)
    wts = synth.int4_weights(N, K, G, seed=19)
    out = oracle.gemm_w4a16(A, False, wts.w, wts.s, M, N, K, G)
    e_q2 = np.mean((np.arange(16) - 8.0) ** 2)
    e_s2 = (0.005 ** 2 + 0.005 * 0.02 + 0.02 ** 2) / 3.0
    expect = math.sqrt(K * e_q2 * e_s2)
    assert 0.9 * expect < out.std() < 1.1 * expect


# ------------------------------------------------------------- FP8

def test_fp8_worked_example():
    g = _golden("fp8_worked_example.json")
    codes = np.array(g["codes"], dtype=np.uint8)
    assert oracle.dequant_fp8(codes).tolist() == g["w"]
    A = _f16_bits(g["A"])
    out = oracle.gemm_w8a16_fp8(A, False, codes, g["alpha"], g["M"], g["N"], g["K"])
    assert out.tolist() == g["out"]
    bias = _f16_bits(g["bias"])
    out_b = oracle.gemm_w8a16_fp8(A, False, codes, g["alpha"], g["M"], g["N"], g["K"], bias_bits=bias)
    assert out_b.tolist() == g["out_with_bias"]


def test_fp8_scale_applies_to_accumulator_linearly():
    M, N, K = 3, 16, 512
    A = synth.activations(M, K, "bf16", seed=20)
    wts = synth.fp8_weights(N, K, seed=21)
    one = oracle.gemm_w8a16_fp8(A, True, wts.w, 1.0, M, N, K)
    scaled = oracle.gemm_w8a16_fp8(A, True, wts.w, 0.25, M, N, K)
    assert np.array_equal(scaled, 0.25 * one)


def test_fp8_small_integer_exact():
    # with s = 1 and small-integer A the float64 sums are exact integers / dyadics
    M, N, K = 4, 8, 64
    rng = np.random.Generator(np.random.PCG64(22))
    Aint = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38          # no NaN codes
    wv = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    A = torch.from_numpy(Aint).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.gemm_w8a16_fp8(A, True, codes, 1.0, M, N, K)
    want = Aint.astype(np.float64) @ wv.T
    assert np.array_equal(got, want)


def test_fp8_weight_recipe_roundtrip():
    wts = synth.fp8_weights(32, 256, seed=23)
    w = oracle.dequant_fp8(wts.w).astype(np.float64)
    assert np.abs(w).max() <= 448.0
    assert np.abs(w).max() >= 256.0         # amax lands near the top of the e4m3 range


# ------------------------------------------------------------- FP4

def _fp4_golden_arrays(g):
    K = g["K"]
    A = np.full((1, K), g["A_default"], dtype=np.float32)
    for k, v in g["A_nonunit"].items():
        A[0, int(k)] = v
    return torch.from_numpy(A).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_fp4_worked_example():
    g = _golden("fp4_worked_example.json")
    K = g["K"]
    packed = np.array(g["packed"], dtype=np.uint8)
    sf = np.array(g["sf_codes"], dtype=np.uint8)
    assert [oracle.e4m3_to_double(c) for c in sf[0]] == g["sf"][0]
    w = oracle.dequant_fp4(packed, sf, K)
    want = np.zeros(K)
    for k, v in g["w_nonzero"].items():
        want[int(k)] = v
    assert w[0].tolist() == want.tolist()
    A = _fp4_golden_arrays(g)
    out = oracle.gemm_bf16_fp4(A, packed, sf, g["alpha"], 1, 1, K)
    assert out.tolist() == g["out"]


def _brute_force_fp4(A16, w_packed, sf, alpha, M, N, K):
    A = torch.from_numpy(A16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    SF = torch.from_numpy(sf).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                byte = int(w_packed[n, k // 2])
                code = (byte >> 4) if (k & 1) else (byte & 15)
                mag = _E2M1[code & 7]
                val = -mag if code & 8 else mag
                acc += float(A[m, k]) * val * float(SF[n, k // 16])
            out[m, n] = alpha * acc
    return out


def test_fp4_gemm_vs_brute_force():
    M, N, K = 2, 6, 96
    A = synth.activations(M, K, "bf16", seed=24)
    wts = synth.fp4_weights(N, K, seed=25)
    got = oracle.gemm_bf16_fp4(A, wts.w, wts.sf, float(wts.alpha), M, N, K)
    want = _brute_force_fp4(A, wts.w, wts.sf, float(wts.alpha), M, N, K)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-15)


def test_fp4_identity_A():
    K = 64
    wts = synth.fp4_weights(10, K, seed=26)
    A = torch.eye(K).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out = oracle.gemm_bf16_fp4(A, wts.w, wts.sf, 1.0, K, 10, K)
    w = oracle.dequant_fp4(wts.w, wts.sf, K).astype(np.float64)
    assert np.array_equal(out, w.T)


def test_fp4_weights_exact_in_bf16():
    # e2m1 (2 significant bits) times e4m3 (4 bits) fits the 8-bit bf16 significand,
    # so RN_bf of the dequantized weight is the weight itself.
    wts = synth.fp4_weights(16, 512, seed=27)
    w = oracle.dequant_fp4(wts.w, wts.sf, 512).astype(np.float64)
    back = oracle.bf16_bits_to_double_array(oracle.round_bf16_array(w))
    assert np.array_equal(back, w)


def test_int4_weights_exact_in_fp32_not_always_in_fp16():
    wts = synth.int4_weights(64, 256, 128, seed=28)
    w = oracle.dequant_int4(wts.w, wts.s, 256, 128).astype(np.float64)
    rn16 = oracle.f16_bits_to_double_array(oracle.round_f16_array(w))
    rel = np.abs(rn16 - w) / np.maximum(np.abs(w), 1e-30)
    assert rel.max() <= 2.0 ** -11          # RN16 relative error bound
    assert (rn16 != w).any()                 # the operand rounding is real


def test_metrics_definition():
    ref = np.array([[1.0, -2.0], [4.0, 0.5]])
    out = ref + np.array([[0.01, 0.0], [-0.02, 0.0]])
    rmax, rmean = oracle.rel_errors(out, ref)
    assert rmax == pytest.approx(0.02 / 4.0)
    assert rmean == pytest.approx((0.03 / 4) / (7.5 / 4))


# ------------------------------------------------- quantiser (upstream of the packing)

def test_quantiser_worked_example():
    g = _golden("int4_quantiser_worked_example.json")
    w, s = oracle.quantize_int4(_f16_bits(g["W"]), g["G"])
    assert w.tolist() == g["packed"]
    assert s.view(np.float16).astype(np.float64).tolist() == g["scales"]
    assert oracle.unpack_int4(w, g["K"]).tolist() == g["q"]
    assert oracle.dequant_int4(w, s, g["K"], g["G"]).astype(np.float64).tolist() == g["dequant"]


@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_quantiser_error_within_half_a_step(G):
    # Rounding to the nearest step: |W - (q - 8) S| <= S / 2 for every weight, and the
    # largest magnitude of a group lands on q - 8 = +-7 (groups with a normal fp16 scale;
    # a subnormal scale is coarser than amax / 7 and may clamp).  An all-zero group gets
    # S = 0 and q = 8.
    rng = np.random.default_rng(300 + G)
    N, K = 64, 1024
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    W[3, :G] = 0
    W[5, G:2 * G] *= np.float16(1e-3)
    w, s = oracle.quantize_int4(W.view(np.uint16), G)
    q = oracle.unpack_int4(w, K).astype(np.int64)
    S = s.view(np.float16).astype(np.float64)               # [K/G][N]
    Sk = np.repeat(S.T, G, axis=1)                          # [N][K]
    Wd = W.astype(np.float64)
    normal = np.repeat((S.T >= 2.0 ** -14), G, axis=1)
    err = np.abs(Wd - (q - 8) * Sk)
    assert np.all(err[normal] <= Sk[normal] / 2)
    assert np.all(q[3, :G] == 8) and S[0, 3] == 0
    absw = np.abs(Wd).reshape(N, K // G, G)
    top = np.take_along_axis(q.reshape(N, K // G, G), absw.argmax(axis=2)[..., None], axis=2)[..., 0]
    assert np.all(np.abs(top[S.T >= 2.0 ** -14] - 8) == 7)


def test_quantiser_reproduces_exactly_representable_weights():
    # W = (q - 8) S with a code of +-7 in every group and scales of at most 8 significant
    # bits, so every weight is an fp16 value: quantising W gives q and S back exactly
    rng = np.random.default_rng(310)
    N, K, G = 16, 512, 64
    q = rng.integers(1, 16, size=(N, K))
    q.reshape(N, K // G, G)[:, :, 0] = rng.choice([1, 15], size=(N, K // G))
    S = rng.integers(128, 256, size=(K // G, N)) * 2.0 ** (rng.integers(-12, -4, size=(K // G, N)) - 7)
    W = (q - 8) * np.repeat(S.T, G, axis=1)
    assert np.array_equal(W.astype(np.float16).astype(np.float64), W)
    w, s = oracle.quantize_int4(W.astype(np.float16).view(np.uint16), G)
    assert np.array_equal(oracle.unpack_int4(w, K), q)
    assert np.array_equal(s.view(np.float16).astype(np.float64), S)


# ------------------------------------------------------------- zero-point INT4

def test_zero_point_worked_example():
    g = _golden("int4_zero_point_worked_example.json")
    w = np.array(g["packed"], dtype=np.uint8)
    s = _f16_bits(g["scales"])
    z = np.array(g["zeros"], dtype=np.uint8)
    assert oracle.dequant_int4_zp(w, s, z, g["K"], g["G"]).astype(np.float64).tolist() == g["w"]
    A = _f16_bits(g["A"])
    out = oracle.gemm_w4a16_zp(A, False, w, s, z, g["M"], g["N"], g["K"], g["G"])
    assert out.tolist() == g["out"]


def test_zero_point_eight_is_the_symmetric_format():
    # Z = 8 everywhere is exactly the symmetric (q - 8) * S format
    rng = np.random.default_rng(320)
    M, N, K, G = 3, 40, 256, 64
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    w = oracle.pack_int4(q)
    s = _f16_bits(rng.uniform(0.005, 0.02, size=(K // G, N)))
    A = _f16_bits(rng.standard_normal((M, K)))
    z = np.full((K // G, N), 8, dtype=np.uint8)
    assert np.array_equal(oracle.dequant_int4_zp(w, s, z, K, G), oracle.dequant_int4(w, s, K, G))
    assert np.array_equal(oracle.gemm_w4a16_zp(A, False, w, s, z, M, N, K, G), oracle.gemm_w4a16(A, False, w, s, M, N, K, G))


def test_zero_point_brute_force():
    # a pure-Python triple loop on a tiny case, zero points and scales varying per group and row
    rng = np.random.default_rng(321)
    M, N, K, G = 2, 5, 64, 32
    q = rng.integers(0, 16, size=(N, K))
    z = rng.integers(0, 16, size=(K // G, N)).astype(np.uint8)
    sv = rng.uniform(0.01, 0.1, size=(K // G, N))
    s = _f16_bits(sv)
    sd = s.view(np.float16).astype(np.float64)
    Av = rng.standard_normal((M, K))
    A = _f16_bits(Av)
    Ad = A.view(np.float16).astype(np.float64)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += Ad[m, k] * (int(q[n, k]) - int(z[k // G, n])) * sd[k // G, n]
            want[m, n] = acc
    got = oracle.gemm_w4a16_zp(A, False, oracle.pack_int4(q.astype(np.uint8)), s, z, M, N, K, G)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- INT4 codebook (NF4-style)

def test_codebook_worked_example():
    g = _golden("int4_codebook_worked_example.json")
    q = np.array(g["q"], dtype=np.uint8)
    w = np.array(g["packed"], dtype=np.uint8)
    assert np.array_equal(oracle.pack_int4(q), w)
    s = _f16_bits(g["scales"])
    lut = _f16_bits(g["lut"])
    assert oracle.dequant_int4_lut(w, s, lut, g["K"], g["G"]).astype(np.float64).tolist() == g["w"]
    A = _f16_bits(g["A"])
    assert oracle.gemm_w4a16_lut(A, False, w, s, lut, g["M"], g["N"], g["K"], g["G"]).tolist() == g["out"]


def test_codebook_of_the_uniform_grid_is_the_symmetric_format():
    # LUT[q] = q - 8 turns the codebook format into the symmetric INT4 format
    rng = np.random.default_rng(330)
    M, N, K, G = 3, 24, 256, 32
    w = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = _f16_bits(rng.uniform(0.005, 0.02, size=(K // G, N)))
    A = _f16_bits(rng.standard_normal((M, K)))
    lut = _f16_bits(np.arange(16) - 8.0)
    assert np.array_equal(oracle.dequant_int4_lut(w, s, lut, K, G), oracle.dequant_int4(w, s, K, G))
    for bf in (False, True):
        Ab = synth.activations(M, K, "bf16", 331) if bf else A
        assert np.array_equal(oracle.gemm_w4a16_lut(Ab, bf, w, s, lut, M, N, K, G),
                              oracle.gemm_w4a16(Ab, bf, w, s, M, N, K, G))


def test_codebook_brute_force():
    # a pure-Python triple loop, a random table and scales varying per group and row
    rng = np.random.default_rng(332)
    M, N, K, G = 2, 5, 64, 32
    q = rng.integers(0, 16, size=(N, K))
    lut = synth.random_codebook(333)
    lutd = lut.view(np.float16).astype(np.float64)
    s = _f16_bits(rng.uniform(0.01, 0.1, size=(K // G, N)))
    sd = s.view(np.float16).astype(np.float64)
    A = _f16_bits(rng.standard_normal((M, K)))
    Ad = A.view(np.float16).astype(np.float64)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += Ad[m, k] * lutd[q[n, k]] * sd[k // G, n]
            want[m, n] = acc
    got = oracle.gemm_w4a16_lut(A, False, oracle.pack_int4(q.astype(np.uint8)), s, lut, M, N, K, G)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_codebook_identity_activations_return_the_weight():
    # A = I: out = w^T exactly (one non-zero product per output)
    rng = np.random.default_rng(334)
    N, K, G = 8, 64, 32
    w = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = _f16_bits(rng.uniform(0.005, 0.02, size=(K // G, N)))
    lut = synth.normal_quantile_codebook()
    A = _f16_bits(np.eye(K))
    out = oracle.gemm_w4a16_lut(A, False, w, s, lut, K, N, K, G)
    assert np.array_equal(out, oracle.dequant_int4_lut(w, s, lut, K, G).astype(np.float64).T)


def test_normal_quantile_codebook_shape():
    # the generator's table: 16 ascending fp16 values in [-1, 1] with an exact zero
    v = synth.normal_quantile_codebook().view(np.float16).astype(np.float64)
    assert v.shape == (16,) and np.all(np.diff(v) > 0)
    assert v[0] == -1.0 and v[15] == 1.0 and v[7] == 0.0


# ------------------------------------------------------------- INT2 (W2A16)

def test_int2_worked_example():
    g = _golden("int2_worked_example.json")
    q = np.array(g["q"], dtype=np.uint8)
    w = oracle.pack_int2(q)
    assert w.tolist() == g["packed"]
    assert np.array_equal(oracle.unpack_int2(w, g["K"]), q)
    s = _f16_bits(g["scales"])
    assert oracle.dequant_int2(w, s, g["K"], g["G"]).astype(np.float64).tolist() == g["w"]
    A = _f16_bits(g["A"])
    assert oracle.gemm_w2a16(A, False, w, s, g["M"], g["N"], g["K"], g["G"]).tolist() == g["out"]


def test_int2_pack_round_trip():
    rng = np.random.default_rng(340)
    q = rng.integers(0, 4, size=(7, 96), dtype=np.uint8)
    w = oracle.pack_int2(q)
    assert w.shape == (7, 24)
    assert np.array_equal(oracle.unpack_int2(w, 96), q)
    # every byte value decodes to four codes that re-pack to it
    allb = np.arange(256, dtype=np.uint8).reshape(1, 256)
    assert np.array_equal(oracle.pack_int2(oracle.unpack_int2(allb, 1024)), allb)


def test_int2_is_int4_shifted_by_six():
    # an INT2 code q has the value of the INT4 code q + 6: (q + 6) - 8 = q - 2
    rng = np.random.default_rng(341)
    M, N, K, G = 3, 16, 128, 32
    q = rng.integers(0, 4, size=(N, K), dtype=np.uint8)
    s = _f16_bits(rng.uniform(0.005, 0.02, size=(K // G, N)))
    A = _f16_bits(rng.standard_normal((M, K)))
    w2 = oracle.pack_int2(q)
    w4 = oracle.pack_int4((q + 6).astype(np.uint8))
    assert np.array_equal(oracle.dequant_int2(w2, s, K, G), oracle.dequant_int4(w4, s, K, G))
    assert np.array_equal(oracle.gemm_w2a16(A, False, w2, s, M, N, K, G), oracle.gemm_w4a16(A, False, w4, s, M, N, K, G))


def test_int2_brute_force():
    rng = np.random.default_rng(342)
    M, N, K, G = 2, 5, 64, 32
    q = rng.integers(0, 4, size=(N, K))
    s = _f16_bits(rng.uniform(0.01, 0.1, size=(K // G, N)))
    sd = s.view(np.float16).astype(np.float64)
    A = _f16_bits(rng.standard_normal((M, K)))
    Ad = A.view(np.float16).astype(np.float64)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += Ad[m, k] * (int(q[n, k]) - 2) * sd[k // G, n]
            want[m, n] = acc
    got = oracle.gemm_w2a16(A, False, oracle.pack_int2(q.astype(np.uint8)), s, M, N, K, G)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- row / column subsets
#
# The large-M GPU tests compare sampled output rows (and the CPU baseline sampled
# columns) against the oracle called with `rows` / `cols`.  Each format's subset path
# must give exactly the entries of the full product, for unsorted and repeated
# indices, first and last rows and columns included.

_SUB_ROWS = [8, 0, 4, 4, 10]
_SUB_COLS = [19, 3, 0, 7, 7, 12]


def _check_subsets(call, M, N):
    full = call(None, None)
    assert full.shape == (M, N)
    rows_only = call(_SUB_ROWS, None)
    cols_only = call(None, _SUB_COLS)
    both = call(_SUB_ROWS, _SUB_COLS)
    assert np.array_equal(rows_only, full[_SUB_ROWS, :])
    assert np.array_equal(cols_only, full[:, _SUB_COLS])
    assert np.array_equal(both, full[np.ix_(_SUB_ROWS, _SUB_COLS)])
    # a single entry equals the full product's entry (no dependence on the other indices)
    assert call([10], [19])[0, 0] == full[10, 19]


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_fp8_row_and_column_subsets(a_dtype):
    M, N, K = 11, 20, 128
    A = synth.activations(M, K, a_dtype, seed=40)
    wts = synth.fp8_weights(N, K, seed=41)
    bias = synth.bias(N, a_dtype, seed=42)
    _check_subsets(lambda r, c: oracle.gemm_w8a16_fp8(A, a_dtype == "bf16", wts.w, float(wts.scale), M, N, K,
                                                      bias_bits=bias, rows=r, cols=c), M, N)


def test_fp4_row_and_column_subsets():
    M, N, K = 11, 20, 96
    A = synth.activations(M, K, "bf16", seed=43)
    wts = synth.fp4_weights(N, K, seed=44)
    _check_subsets(lambda r, c: oracle.gemm_bf16_fp4(A, wts.w, wts.sf, float(wts.alpha), M, N, K, rows=r, cols=c),
                   M, N)
    # and the subset entries against the independent brute-force loop
    want = _brute_force_fp4(A, wts.w, wts.sf, float(wts.alpha), M, N, K)
    got = oracle.gemm_bf16_fp4(A, wts.w, wts.sf, float(wts.alpha), M, N, K, rows=_SUB_ROWS, cols=_SUB_COLS)
    assert np.allclose(got, want[np.ix_(_SUB_ROWS, _SUB_COLS)], rtol=1e-14, atol=1e-15)


def test_zero_point_row_and_column_subsets():
    M, N, K, G = 11, 20, 128, 32
    A = synth.activations(M, K, "f16", seed=45)
    wts = synth.int4_weights(N, K, G, seed=46)
    z = synth.int4_zeros(N, K, G, seed=47)
    _check_subsets(lambda r, c: oracle.gemm_w4a16_zp(A, False, wts.w, wts.s, z, M, N, K, G, rows=r, cols=c), M, N)


def test_codebook_row_and_column_subsets():
    M, N, K, G = 11, 20, 128, 64
    A = synth.activations(M, K, "bf16", seed=48)
    wts = synth.int4_weights(N, K, G, seed=49)
    lut = synth.random_codebook(50)
    _check_subsets(lambda r, c: oracle.gemm_w4a16_lut(A, True, wts.w, wts.s, lut, M, N, K, G, rows=r, cols=c),
                   M, N)


def test_int2_row_and_column_subsets():
    M, N, K, G = 11, 20, 128, 32
    A = synth.activations(M, K, "f16", seed=51)
    wts = synth.int2_weights(N, K, G, seed=52)
    _check_subsets(lambda r, c: oracle.gemm_w2a16(A, False, wts.w, wts.s, M, N, K, G, rows=r, cols=c), M, N)


def test_int4_subsets_against_brute_force():
    M, N, K, G = 11, 20, 64, 32
    A = synth.activations(M, K, "f16", seed=53)
    wts = synth.int4_weights(N, K, G, seed=54)
    _check_subsets(lambda r, c: oracle.gemm_w4a16(A, False, wts.w, wts.s, M, N, K, G, rows=r, cols=c), M, N)
    want = _brute_force_int4(A, wts.w, wts.s, M, N, K, G)
    got = oracle.gemm_w4a16(A, False, wts.w, wts.s, M, N, K, G, rows=_SUB_ROWS, cols=_SUB_COLS)
    assert np.allclose(got, want[np.ix_(_SUB_ROWS, _SUB_COLS)], rtol=0, atol=1e-12)
