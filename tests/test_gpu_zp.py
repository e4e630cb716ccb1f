"""GPU parity of zero-point (asymmetric) INT4: w = (q - Z) * S, Z per group and row."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, check_close, out_bits, out_to_f64, to_dev_f16bits

pytestmark = pytest.mark.gpu


class ZpProblem:
    def __init__(self, M, N, K, G, a_dtype="f16", seed=0, A_bits=None, z=None):
        self.M, self.N, self.K, self.G, self.a_dtype = M, N, K, G, a_dtype
        self.A = A_bits if A_bits is not None else synth.activations(M, K, a_dtype, seed)
        self.wts = synth.int4_weights(N, K, G, seed + 1)
        self.z = z if z is not None else synth.int4_zeros(N, K, G, seed + 2)
        self.A_d = to_dev_f16bits(self.A, a_dtype)
        w_d = torch.from_numpy(self.wts.w).to(DEV)
        s_d = to_dev_f16bits(self.wts.s, "f16")
        self.wk, self.sk = wq.wq_pack_int4(w_d, s_d, N, K, G)
        self.zk = wq.wq_pack_int4_zeros(torch.from_numpy(self.z).to(DEV), N, K, G)

    def run(self):
        return wq.wq_gemm_w4a16_zp(self.A_d, self.wk, self.sk, self.zk, self.N, self.K, self.G)

    def ref(self, rows=None):
        return oracle.gemm_w4a16_zp(self.A, self.a_dtype == "bf16", self.wts.w, self.wts.s, self.z, self.M, self.N,
                                    self.K, self.G, rows=rows)


def _check(p, out, rows, what):
    """fp16: the accuracy bar against the float64 oracle.  bf16: the operand
    RN_bf((q - z) * s) loses ~2^-9 per weight, so the bar is the same rounding done by
    materialising the bf16 weight and calling a dense GEMM (the symmetric format's bar)."""
    ref = p.ref(rows=rows)
    got = out_to_f64(out)
    got = got if rows is None else got[rows]
    if p.a_dtype == "f16":
        check_close(got, ref, what=what)
        return
    w = oracle.dequant_int4_zp(p.wts.w, p.wts.s, p.z, p.K, p.G)
    cast = torch.nn.functional.linear(p.A_d, torch.from_numpy(w).to(DEV).to(torch.bfloat16))
    c = out_to_f64(cast)
    c = c if rows is None else c[rows]
    k_max, k_mean = oracle.rel_errors(got, ref)
    _, c_mean = oracle.rel_errors(c, ref)
    assert k_max <= 5e-3, f"{what} rel_max={k_max:.3e}"
    assert k_mean <= 1.02 * c_mean, f"{what} kernel {k_mean:.3e} vs cast-copy {c_mean:.3e}"


def _eye_bits(K, a_dtype):
    eye = np.eye(K, dtype=np.float32)
    if a_dtype == "f16":
        return eye.astype(np.float16).view(np.uint16)
    return torch.from_numpy(eye).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_packed_zeros_bytes():
    assert wq.wq_int4_packed_zeros_bytes(200, 96, 32) == 256 * (256 // 32)
    _, sb = wq.wq_int4_packed_bytes(4096, 4096, 128)
    assert wq.wq_int4_packed_zeros_bytes(4096, 4096, 128) == sb // 2


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
@pytest.mark.parametrize("N", [384, 512])
def test_identity_A_returns_rounded_weight_bit_exact(G, a_dtype, N):
    # one non-zero product per output: out[m, n] = RN((q - z) * s) exactly, every
    # (group, row) zero point exercised; M = K = 256 runs the one-CTA tile kernel
    K = 256
    p = ZpProblem(K, N, K, G, a_dtype=a_dtype, seed=601, A_bits=_eye_bits(K, a_dtype))
    out = p.run()
    torch.cuda.synchronize()
    w = oracle.dequant_int4_zp(p.wts.w, p.wts.s, p.z, K, G).astype(np.float64)
    rn = oracle.round_f16_array(w.T) if a_dtype == "f16" else oracle.round_bf16_array(w.T)
    assert np.array_equal(out_bits(out), rn)


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_identity_A_pair_kernel_bit_exact(a_dtype):
    # enough 256 x 256 tiles to take the two-CTA kernel; identity blocks down the rows
    K, G, N, M = 256, 128, 8192, 4096
    A = np.tile(_eye_bits(K, a_dtype), (M // K, 1))
    p = ZpProblem(M, N, K, G, a_dtype=a_dtype, seed=602, A_bits=A)
    plan = wq.get_plan(wq.WQ_OP_W4A16_ZP, wq.WQ_BF16 if a_dtype == "bf16" else wq.WQ_F16, M, N, K, G)
    assert plan["kernel"] == wq.WQ_KERNEL_TILE_PAIR
    out = p.run()
    torch.cuda.synchronize()
    w = oracle.dequant_int4_zp(p.wts.w, p.wts.s, p.z, K, G).astype(np.float64)
    rn = oracle.round_f16_array(w.T) if a_dtype == "f16" else oracle.round_bf16_array(w.T)
    assert np.array_equal(out_bits(out), np.tile(rn, (M // K, 1)))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_zero_point_eight_matches_symmetric_bitwise(a_dtype):
    # Z = 8 everywhere is the symmetric format: same kernel arithmetic, same bits
    M, N, K, G = 200, 512, 1024, 128
    z = np.full((K // G, N), 8, dtype=np.uint8)
    p = ZpProblem(M, N, K, G, a_dtype=a_dtype, seed=603, z=z)
    got = p.run()
    sym = wq.wq_gemm_w4a16(p.A_d, p.wk, p.sk, N, K, G)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), sym.view(torch.int16))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,G", [(1, 4096, 1024, 128), (16, 4096, 4096, 128), (13, 200, 96, 32),
                                     (96, 512, 2048, 64), (300, 1024, 1024, 256), (1000, 768, 512, 32)])
def test_random_vs_oracle(M, N, K, G, a_dtype):
    p = ZpProblem(M, N, K, G, a_dtype=a_dtype, seed=604 + M + K)
    plan = wq.get_plan(wq.WQ_OP_W4A16_ZP, wq.WQ_BF16 if a_dtype == "bf16" else wq.WQ_F16, M, N, K, G)
    # M <= 16 with K % 64 == 0 takes the register decode kernel, the rest the tile kernels
    assert (plan["kernel"] == wq.WQ_KERNEL_DECODE) == (M <= 16 and K % 64 == 0)
    out = p.run()
    torch.cuda.synchronize()
    _check(p, out, None, f"zp M{M} N{N} K{K} G{G}")


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_large_pair_sampled_rows(a_dtype):
    # two-CTA kernel with a ragged last token tile; the oracle computes sampled rows
    M, N, K, G = 4100, 4096, 4096, 128
    p = ZpProblem(M, N, K, G, a_dtype=a_dtype, seed=605)
    out = p.run()
    torch.cuda.synchronize()
    rows = synth.sample_rows(M, 24, seed=606)   # includes the first and the last row
    _check(p, out, rows, "zp pair sampled")


def test_bad_arguments():
    N, K, G = 256, 256, 128
    p = ZpProblem(4, N, K, G, seed=607)
    lib = wq.lib()
    st = lib.wq_gemm_w4a16_zp(p.A_d.data_ptr(), 0, p.wk.data_ptr(), p.sk.data_ptr(), None, 4, N, K, G,
                              torch.empty(4, N, dtype=torch.float16, device=DEV).data_ptr(), None, 0, None)
    assert st == 1   # WQ_ERR_NULL: zero points required
    st = lib.wq_pack_int4_zeros(None, N, K, G, p.zk.data_ptr(), None)
    assert st == 1
    st = lib.wq_pack_int4_zeros(p.zk.data_ptr(), N, K, 48, p.zk.data_ptr(), None)
    assert st == 3   # WQ_ERR_GROUP
    st = lib.wq_pack_int4_zeros(p.zk.data_ptr(), N, K, G, p.zk.data_ptr() + 1, None)
    assert st == 4   # WQ_ERR_MISALIGNED


# ------------------------------------------------------------------ decode kernel (M <= 16)

@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,G", [(1, 128), (5, 32), (16, 64), (9, 256)])
def test_decode_zero_point_eight_matches_symmetric_bitwise(M, G, a_dtype):
    # Z = 8: the fold adds (8 - z) S_g = 0 exactly, so the bits equal the symmetric
    # decode kernel's
    N, K = 1024, 2048
    z = np.full((K // G, N), 8, dtype=np.uint8)
    p = ZpProblem(M, N, K, G, a_dtype=a_dtype, seed=610 + M, z=z)
    assert wq.get_plan(wq.WQ_OP_W4A16_ZP, wq.WQ_BF16 if a_dtype == "bf16" else wq.WQ_F16, M, N, K, G)["kernel"] \
        == wq.WQ_KERNEL_DECODE
    got = p.run()
    sym = wq.wq_gemm_w4a16(p.A_d, p.wk, p.sk, N, K, G)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), sym.view(torch.int16))


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_decode_identity_rows_bit_exact(G, a_dtype):
    # A = the first 16 rows of the identity: out[m, n] = RN((q[n, m] - z) * s) exactly
    # (one non-zero product, and the fold's (b + z) S_g terms are exact integers times 1)
    M, N, K = 16, 384, 512
    A = _eye_bits(K, a_dtype)[:M].copy()
    p = ZpProblem(M, N, K, G, a_dtype=a_dtype, seed=611, A_bits=A)
    out = p.run()
    torch.cuda.synchronize()
    w = oracle.dequant_int4_zp(p.wts.w, p.wts.s, p.z, K, G).astype(np.float64)
    rn = oracle.round_f16_array(w.T[:M]) if a_dtype == "f16" else oracle.round_bf16_array(w.T[:M])
    assert np.array_equal(out_bits(out), rn)


@pytest.mark.parametrize("case", synth.DECODE, ids=lambda c: f"M{c.M}_N{c.N}_K{c.K}")
def test_decode_configs_with_zero_points(case):
    p = ZpProblem(case.M, case.N, case.K, case.G, seed=612 + case.M + case.N)
    out = p.run()
    torch.cuda.synchronize()
    _check(p, out, None, f"zp decode {case}")
