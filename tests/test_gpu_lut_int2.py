"""GPU parity of the codebook INT4 format (w = LUT[q] * S, an NF4-style 16-entry
table) and of INT2 W2A16 (w = (q - 2) * S, four codes per byte along K)."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, Int2Problem, check_close, out_bits, out_to_f64, to_dev_f16bits

pytestmark = pytest.mark.gpu


def _eye_bits(K, a_dtype):
    eye = np.eye(K, dtype=np.float32)
    if a_dtype == "f16":
        return eye.astype(np.float16).view(np.uint16)
    return torch.from_numpy(eye).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _adt(a_dtype):
    return wq.WQ_BF16 if a_dtype == "bf16" else wq.WQ_F16


def _check(p, out, rows, what):
    """fp16: the accuracy bar against the float64 oracle.  bf16: the operand
    RN_bf(w) loses ~2^-9 per weight, so the bar is the same rounding done by
    materialising the bf16 weight and calling a dense GEMM (as for the symmetric format)."""
    ref = p.ref(rows=rows)
    got = out_to_f64(out)
    got = got if rows is None else got[rows]
    if p.a_dtype == "f16":
        check_close(got, ref, what=what)
        return
    cast = torch.nn.functional.linear(p.A_d, torch.from_numpy(p.dequant_ref()).to(DEV).to(torch.bfloat16))
    c = out_to_f64(cast)
    c = c if rows is None else c[rows]
    k_max, k_mean = oracle.rel_errors(got, ref)
    _, c_mean = oracle.rel_errors(c, ref)
    assert k_max <= 5e-3, f"{what} rel_max={k_max:.3e}"
    assert k_mean <= 1.02 * c_mean, f"{what} kernel {k_mean:.3e} vs cast-copy {c_mean:.3e}"


def _rn(w, a_dtype):
    w = w.astype(np.float64)
    return oracle.round_f16_array(w) if a_dtype == "f16" else oracle.round_bf16_array(w)


# ------------------------------------------------------------------ codebook INT4

class LutProblem:
    def __init__(self, M, N, K, G, a_dtype="f16", seed=0, A_bits=None, lut=None):
        self.M, self.N, self.K, self.G, self.a_dtype = M, N, K, G, a_dtype
        self.A = A_bits if A_bits is not None else synth.activations(M, K, a_dtype, seed)
        self.wts = synth.int4_weights(N, K, G, seed + 1)
        self.lut = lut if lut is not None else synth.normal_quantile_codebook()
        self.A_d = to_dev_f16bits(self.A, a_dtype)
        w_d = torch.from_numpy(self.wts.w).to(DEV)
        s_d = to_dev_f16bits(self.wts.s, "f16")
        self.wk, self.sk = wq.wq_pack_int4(w_d, s_d, N, K, G)
        self.lut_d = to_dev_f16bits(self.lut, "f16")

    def run(self):
        return wq.wq_gemm_w4a16_lut(self.A_d, self.wk, self.sk, self.lut_d, self.N, self.K, self.G)

    def ref(self, rows=None):
        return oracle.gemm_w4a16_lut(self.A, self.a_dtype == "bf16", self.wts.w, self.wts.s, self.lut, self.M,
                                     self.N, self.K, self.G, rows=rows)

    def dequant_ref(self):
        return oracle.dequant_int4_lut(self.wts.w, self.wts.s, self.lut, self.K, self.G)


@pytest.mark.parametrize("table", ["nf4", "random"])
def test_lut_debug_dequant_bit_exact(table):
    N, K, G = 200, 512, 64
    lut = synth.normal_quantile_codebook() if table == "nf4" else synth.random_codebook(700)
    p = LutProblem(1, N, K, G, seed=701, lut=lut)
    got = wq.wq_debug_dequant_int4_lut(p.wk, p.sk, p.lut_d, N, K, G).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), p.dequant_ref().view(np.uint32))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
@pytest.mark.parametrize("table", ["nf4", "random"])
def test_lut_identity_A_bit_exact(G, a_dtype, table):
    # one non-zero product per output: out[m, n] = RN(LUT[q] * s) exactly, so every
    # code of every row half goes through the kernel's byte-permute lookup
    K, N = 256, 384
    lut = synth.normal_quantile_codebook() if table == "nf4" else synth.random_codebook(702 + G)
    p = LutProblem(K, N, K, G, a_dtype=a_dtype, seed=703, A_bits=_eye_bits(K, a_dtype), lut=lut)
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), _rn(p.dequant_ref().T, a_dtype))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_lut_identity_A_pair_kernel_bit_exact(a_dtype):
    K, G, N, M = 256, 128, 8192, 4096
    A = np.tile(_eye_bits(K, a_dtype), (M // K, 1))
    p = LutProblem(M, N, K, G, a_dtype=a_dtype, seed=704, A_bits=A, lut=synth.random_codebook(705))
    assert wq.get_plan(wq.WQ_OP_W4A16_LUT, _adt(a_dtype), M, N, K, G)["kernel"] == wq.WQ_KERNEL_TILE_PAIR
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), np.tile(_rn(p.dequant_ref().T, a_dtype), (M // K, 1)))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K,G", [(4, 1056, 32), (200, 1024, 128), (4096, 1024, 128)])
def test_lut_uniform_grid_matches_int4_bitwise(M, K, G, a_dtype):
    # LUT[q] = q - 8 gives the symmetric operand RN((q - 8) * s): the same bits as the
    # zero-point tile kernel with Z = 8 (K % 64 != 0 keeps M = 4 off the register
    # decode kernel, which the zero-point entry takes for M <= 16)
    N = 512
    p = LutProblem(M, N, K, G, a_dtype=a_dtype, seed=706, lut=(np.arange(16) - 8.0).astype(np.float16).view(np.uint16))
    got = p.run()
    z = wq.wq_pack_int4_zeros(torch.full((K // G, N), 8, dtype=torch.uint8, device=DEV), N, K, G)
    ref = wq.wq_gemm_w4a16_zp(p.A_d, p.wk, p.sk, z, N, K, G)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,G", [(1, 4096, 1024, 128), (16, 4096, 4096, 128), (13, 200, 96, 32),
                                     (96, 512, 2048, 64), (300, 1024, 1024, 256), (1000, 768, 512, 32)])
def test_lut_random_vs_oracle(M, N, K, G, a_dtype):
    p = LutProblem(M, N, K, G, a_dtype=a_dtype, seed=707 + M + K)
    decode = a_dtype == "f16" and M <= 16 and K % 64 == 0
    assert (wq.get_plan(wq.WQ_OP_W4A16_LUT, _adt(a_dtype), M, N, K, G)["kernel"] == wq.WQ_KERNEL_DECODE) == decode
    out = p.run()
    torch.cuda.synchronize()
    _check(p, out, None, f"lut M{M} N{N} K{K} G{G}")


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_lut_large_pair_sampled_rows(a_dtype):
    M, N, K, G = 4100, 4096, 4096, 128
    p = LutProblem(M, N, K, G, a_dtype=a_dtype, seed=708)
    out = p.run()
    torch.cuda.synchronize()
    rows = synth.sample_rows(M, 24, seed=709)
    _check(p, out, rows, "lut pair sampled")


# ------------------------------------------------------------------ codebook decode kernel
# fp16 activations, M <= 16, K % 64 == 0: the register decode kernel looks up LUT[q]
# with byte permutes into the MMA fragment registers and applies the group scale to
# the fp32 sums, so an output is RN16(s * sum_k A LUT[q]) (one rounding of an fp32 value)

def _lut_plan(M, N, K, G, a_dtype="f16"):
    return wq.get_plan(wq.WQ_OP_W4A16_LUT, _adt(a_dtype), M, N, K, G)


def test_lut_decode_plan():
    assert _lut_plan(1, 4096, 4096, 128)["kernel"] == wq.WQ_KERNEL_DECODE
    assert _lut_plan(16, 4096, 4096, 128)["kernel"] == wq.WQ_KERNEL_DECODE
    assert _lut_plan(16, 4096, 4096, 128)["bk"] == 128
    assert _lut_plan(17, 4096, 4096, 128)["kernel"] == wq.WQ_KERNEL_TILE
    assert _lut_plan(16, 4096, 4096, 128, "bf16")["kernel"] == wq.WQ_KERNEL_TILE
    assert _lut_plan(4, 1024, 1056, 32)["kernel"] == wq.WQ_KERNEL_TILE   # K % 64 == 32


@pytest.mark.parametrize("G", [32, 64, 128, 256])
@pytest.mark.parametrize("table", ["nf4", "random"])
def test_lut_decode_identity_rows_bit_exact(G, table):
    # A = the first 16 rows of the identity: out[m, n] = RN16(LUT[q[n, m]] * s) exactly
    # (one non-zero product; s * LUT[q] has at most 22 significant bits, exact in fp32),
    # so every code position of every row half goes through the lookup and the fragment
    # order, with K split over several slices
    M, N, K = 16, 384, 1024
    lut = synth.normal_quantile_codebook() if table == "nf4" else synth.random_codebook(720 + G)
    p = LutProblem(M, N, K, G, seed=721, A_bits=_eye_bits(K, "f16")[:M].copy(), lut=lut)
    plan = _lut_plan(M, N, K, G)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] > 1
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), _rn(p.dequant_ref().T[:M], "f16"))


@pytest.mark.parametrize("shift", [0, 1])
def test_lut_decode_one_hot_every_k_step(shift):
    # token m selects k_m over all 16 positions of a k step and over stages and slices
    M, N, K, G = 16, 256, 2048, 128
    ks = [16 * ((7 * m + 5 * shift) % (K // 16)) + (m + 3 * shift) % 16 for m in range(M)]
    assert sorted(k % 16 for k in ks) == list(range(16))
    A = np.zeros((M, K), dtype=np.float32)
    A[np.arange(M), ks] = 1.0
    p = LutProblem(M, N, K, G, seed=722 + shift, A_bits=A.astype(np.float16).view(np.uint16),
                   lut=synth.random_codebook(723 + shift))
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), _rn(p.dequant_ref()[:, ks].T, "f16"))


@pytest.mark.parametrize("M", [1, 9, 16])
def test_lut_decode_uniform_grid_matches_symmetric(M):
    # LUT[q] = q - 8 is the symmetric format: the operands equal the symmetric decode
    # kernel's q - 8, and with the same 128-value stages (K % 256 == 64) and K slices
    # the sums and the outputs are the same bits
    N, K, G = 512, 4160, 64
    p = LutProblem(M, N, K, G, seed=724 + M, lut=(np.arange(16) - 8.0).astype(np.float16).view(np.uint16))
    lp = _lut_plan(M, N, K, G)
    sp = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, G)
    assert lp["kernel"] == sp["kernel"] == wq.WQ_KERNEL_DECODE and lp["bk"] == sp["bk"] == 128
    got = p.run()
    sym = wq.wq_gemm_w4a16(p.A_d, p.wk, p.sk, N, K, G)
    torch.cuda.synchronize()
    check_close(out_to_f64(got), p.ref(), what=f"lut decode q-8 M={M}")
    if lp["splits"] == sp["splits"]:
        assert torch.equal(got.view(torch.int16), sym.view(torch.int16))


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_lut_decode_every_token_count(M):
    p = LutProblem(M, 256, 1024, 128, seed=730 + M, lut=synth.random_codebook(731))
    out = p.run()
    torch.cuda.synchronize()
    check_close(out_to_f64(out), p.ref(), what=f"lut decode M={M}")


@pytest.mark.parametrize("M,N,K,G", [(1, 1000, 4160, 64), (7, 136, 1088, 32), (16, 11008, 4096, 128),
                                     (3, 264, 192, 64), (16, 256, 16384, 128)])
def test_lut_decode_ragged_and_deterministic(M, N, K, G):
    # tail rows, K % 128 == 64 (a half stage of zero fill), one stage, the largest cluster
    p = LutProblem(M, N, K, G, seed=740 + M + K)
    assert _lut_plan(M, N, K, G)["kernel"] == wq.WQ_KERNEL_DECODE
    wq.wq_clear_device_status()
    first = p.run()
    torch.cuda.synchronize()
    assert wq.wq_device_status() == 0
    check_close(out_to_f64(first), p.ref(), what=f"lut decode M={M} N={N} K={K} G={G}")
    for _ in range(3):
        assert torch.equal(p.run(), first)


@pytest.mark.parametrize("M", [1, 16, 64])
def test_lut_table_written_by_the_preceding_kernel(M):
    # the table may be produced by the kernel right before the GEMM on the stream (the
    # GEMM may start early, programmatic dependent launch, but reads lut only after
    # waiting for it): a copy kernel writes the table, then the GEMM runs, back to back,
    # on the decode kernel (M <= 16) and the tile kernel
    N, K, G = 1024, 2048, 128
    lut_new = synth.random_codebook(750 + M)
    p = LutProblem(M, N, K, G, seed=751 + M, lut=lut_new)
    src = to_dev_f16bits(lut_new, "f16")
    for _ in range(3):
        p.lut_d.zero_()
        torch.cuda.synchronize()
        torch.mul(src, 1.0, out=p.lut_d)   # an elementwise kernel, not a copy-engine transfer
        out = p.run()
        torch.cuda.synchronize()
        check_close(out_to_f64(out), p.ref(), what=f"lut written before the GEMM M={M}")


def test_lut_bad_arguments():
    N, K, G = 256, 256, 128
    p = LutProblem(4, N, K, G, seed=710)
    lib = wq.lib()
    out = torch.empty(4, N, dtype=torch.float16, device=DEV)
    st = lib.wq_gemm_w4a16_lut(p.A_d.data_ptr(), 0, p.wk.data_ptr(), p.sk.data_ptr(), None, 4, N, K, G,
                               out.data_ptr(), None, 0, None)
    assert st == 1   # WQ_ERR_NULL: the table is required
    lut2 = torch.zeros(24, dtype=torch.float16, device=DEV)
    st = lib.wq_gemm_w4a16_lut(p.A_d.data_ptr(), 0, p.wk.data_ptr(), p.sk.data_ptr(), lut2.data_ptr() + 2, 4, N,
                               K, G, out.data_ptr(), None, 0, None)
    assert st == 4   # WQ_ERR_MISALIGNED: the table is read as two 16-byte vectors
    st = lib.wq_gemm_w4a16_lut(p.A_d.data_ptr(), 0, p.wk.data_ptr(), p.sk.data_ptr(), p.lut_d.data_ptr(), 4, N,
                               K, 48, out.data_ptr(), None, 0, None)
    assert st == 3   # WQ_ERR_GROUP


# ------------------------------------------------------------------ INT2 (W2A16)

def test_int2_packed_scales_bytes():
    assert wq.wq_int2_packed_scales_bytes(200, 192, 64) == 256 * (256 // 64) * 2
    _, sb = wq.wq_int4_packed_bytes(4096, 4096, 128)
    assert wq.wq_int2_packed_scales_bytes(4096, 4096, 128) == sb


@pytest.mark.parametrize("N,K,G", [(200, 192, 64), (512, 1024, 32), (384, 2048, 256)])
def test_int2_debug_dequant_bit_exact(N, K, G):
    p = Int2Problem(1, N, K, G, seed=720 + K)
    got = wq.wq_debug_dequant_int2(p.w_d, p.sk, N, K, G).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), p.dequant_ref().view(np.uint32))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_int2_identity_A_bit_exact(G, a_dtype):
    # out[m, n] = RN((q - 2) * s) exactly: every code position of the magic-number unpack
    K, N = 256, 384
    p = Int2Problem(K, N, K, G, a_dtype=a_dtype, seed=721, A_bits=_eye_bits(K, a_dtype))
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), _rn(p.dequant_ref().T, a_dtype))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_int2_identity_A_pair_kernel_bit_exact(a_dtype):
    K, G, N, M = 256, 128, 8192, 4096
    A = np.tile(_eye_bits(K, a_dtype), (M // K, 1))
    p = Int2Problem(M, N, K, G, a_dtype=a_dtype, seed=722, A_bits=A)
    assert wq.get_plan(wq.WQ_OP_W2A16, _adt(a_dtype), M, N, K, G)["kernel"] == wq.WQ_KERNEL_TILE_PAIR
    out = p.run()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), np.tile(_rn(p.dequant_ref().T, a_dtype), (M // K, 1)))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [4, 200, 4096])
def test_int2_matches_int4_shifted_codes_bitwise(M, a_dtype, monkeypatch):
    # an INT2 code q has the operand of the INT4 code q + 6; the tile kernels tile both
    # formats alike, so the outputs agree bit for bit (INT4 through the codebook entry
    # with the uniform-grid table LUT[q] = q - 8, kept on the tile kernels: with fp16
    # activations and M <= 16 the codebook entry would take the register decode kernel)
    monkeypatch.setenv("WQ_DISABLE_DECODE", "1")
    N, K, G = 512, 1024, 64
    rng = np.random.default_rng(723)
    q = rng.integers(0, 4, size=(N, K), dtype=np.uint8)
    p = Int2Problem(M, N, K, G, a_dtype=a_dtype, seed=724, codes=q)
    got = p.run()
    w4 = torch.from_numpy(oracle.pack_int4((q + 6).astype(np.uint8))).to(DEV)
    wk, sk = wq.wq_pack_int4(w4, p.s_d, N, K, G)
    grid = to_dev_f16bits((np.arange(16) - 8.0).astype(np.float16).view(np.uint16), "f16")
    ref = wq.wq_gemm_w4a16_lut(p.A_d, wk, sk, grid, N, K, G)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,G", [(1, 4096, 1024, 128), (16, 4096, 4096, 128), (13, 200, 192, 64),
                                     (96, 512, 2048, 64), (300, 1024, 1024, 256), (1000, 768, 320, 32)])
def test_int2_random_vs_oracle(M, N, K, G, a_dtype):
    p = Int2Problem(M, N, K, G, a_dtype=a_dtype, seed=725 + M + K)
    out = p.run()
    torch.cuda.synchronize()
    _check(p, out, None, f"int2 M{M} N{N} K{K} G{G}")


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_int2_large_pair_sampled_rows(a_dtype):
    M, N, K, G = 4100, 4096, 4096, 128
    p = Int2Problem(M, N, K, G, a_dtype=a_dtype, seed=726)
    out = p.run()
    torch.cuda.synchronize()
    rows = synth.sample_rows(M, 24, seed=727)
    _check(p, out, rows, "int2 pair sampled")


def test_int2_bad_arguments():
    lib = wq.lib()
    N, K, G = 256, 256, 128
    p = Int2Problem(4, N, K, G, seed=728)
    out = torch.empty(4, N, dtype=torch.float16, device=DEV)
    st = lib.wq_gemm_w2a16(p.A_d.data_ptr(), 0, p.w_d.data_ptr(), p.sk.data_ptr(), 4, N, 224, 32, out.data_ptr(),
                           None, 0, None)
    assert st == 2   # WQ_ERR_SHAPE: K % 64
    st = lib.wq_gemm_w2a16(p.A_d.data_ptr(), 0, p.w_d.data_ptr(), p.sk.data_ptr(), 4, N, K, 96, out.data_ptr(),
                           None, 0, None)
    assert st == 3   # WQ_ERR_GROUP
    st = lib.wq_gemm_w2a16(p.A_d.data_ptr(), 0, p.w_d.data_ptr() + 4, p.sk.data_ptr(), 4, N, K, G, out.data_ptr(),
                           None, 0, None)
    assert st == 4   # WQ_ERR_MISALIGNED
    st = lib.wq_pack_int2_scales(None, N, K, G, p.sk.data_ptr(), None)
    assert st == 1
