"""Shared helpers for the GPU parity tests (not collected as tests)."""
import numpy as np
import torch

import oracle
from weight_only_quantized_tma_gb300 import synth

# Accuracy bar for fp16 / bf16 outputs against the float64 oracle: max|out-ref|/max|ref|
# and mean|out-ref|/mean|ref| ("Low Bit Triton Kernels", exercise 4: mean / max
# relative error near 1e-3 / 5e-3).
REL_MAX = 5e-3
REL_MEAN = 1e-3

DEV = torch.device("cuda:0")


def to_dev_f16bits(bits: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.to(DEV)


def out_to_f64(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def out_bits(out: torch.Tensor) -> np.ndarray:
    return out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class Int4Problem:
    """Seeded INT4 problem on host and device, with the packed device buffers."""

    def __init__(self, M, N, K, G, a_dtype="f16", seed=0, A_bits=None, wts=None):
        self.M, self.N, self.K, self.G, self.a_dtype = M, N, K, G, a_dtype
        self.A = A_bits if A_bits is not None else synth.activations(M, K, a_dtype, seed)
        self.wts = wts if wts is not None else synth.int4_weights(N, K, G, seed + 1)
        self.A_d = to_dev_f16bits(self.A, a_dtype)
        self.w_d = torch.from_numpy(self.wts.w).to(DEV)
        self.s_d = to_dev_f16bits(self.wts.s, "f16")

    def pack(self):
        import weight_only_quantized_tma_gb300 as wq
        self.wk, self.sk = wq.wq_pack_int4(self.w_d, self.s_d, self.N, self.K, self.G)
        return self

    def run(self, out=None, ws=None):
        import weight_only_quantized_tma_gb300 as wq
        return wq.wq_gemm_w4a16(self.A_d, self.wk, self.sk, self.N, self.K, self.G, out=out, ws=ws)

    @property
    def out_dtype(self):
        return self.a_dtype

    def ref(self, rows=None):
        return oracle.gemm_w4a16(self.A, self.a_dtype == "bf16", self.wts.w, self.wts.s, self.M, self.N, self.K,
                                 self.G, rows=rows)


class Fp8Problem:
    """Seeded FP8 (W8A16) problem: e4m3 codes, per-tensor scale, optional bias."""

    def __init__(self, M, N, K, a_dtype="bf16", seed=0, with_bias=False):
        self.M, self.N, self.K, self.a_dtype = M, N, K, a_dtype
        self.A = synth.activations(M, K, a_dtype, seed)
        self.wts = synth.fp8_weights(N, K, seed + 1)
        self.bias = synth.bias(N, a_dtype, seed + 2) if with_bias else None
        self.A_d = to_dev_f16bits(self.A, a_dtype)
        self.w_d = torch.from_numpy(self.wts.w).to(DEV)
        self.alpha = torch.tensor([self.wts.scale], dtype=torch.float32, device=DEV)
        self.bias_d = to_dev_f16bits(self.bias, a_dtype) if with_bias else None

    def run(self, alpha=None):
        import weight_only_quantized_tma_gb300 as wq
        return wq.wq_gemm_w8a16_fp8(self.A_d, self.w_d, self.alpha if alpha is None else alpha, bias=self.bias_d)

    def ref(self, rows=None):
        return oracle.gemm_w8a16_fp8(self.A, self.a_dtype == "bf16", self.wts.w, float(self.wts.scale), self.M,
                                     self.N, self.K, bias_bits=self.bias, rows=rows)


class Fp4Problem:
    """Seeded BF16 x FP4 problem: e2m1 codes, e4m3 block scales (prepacked), global alpha."""

    def __init__(self, M, N, K, seed=0):
        self.M, self.N, self.K = M, N, K
        self.A = synth.activations(M, K, "bf16", seed)
        self.wts = synth.fp4_weights(N, K, seed + 1)
        self.A_d = to_dev_f16bits(self.A, "bf16")
        self.w_d = torch.from_numpy(self.wts.w).to(DEV)
        self.sf_d = torch.from_numpy(self.wts.sf).to(DEV)
        import weight_only_quantized_tma_gb300 as wq
        self.sfk = wq.wq_pack_fp4_sf(self.sf_d, N, K)
        self.alpha = torch.tensor([self.wts.alpha], dtype=torch.float32, device=DEV)

    def run(self):
        import weight_only_quantized_tma_gb300 as wq
        return wq.wq_gemm_bf16_fp4(self.A_d, self.w_d, self.sfk, self.alpha)

    def ref(self, rows=None):
        return oracle.gemm_bf16_fp4(self.A, self.wts.w, self.wts.sf, float(self.wts.alpha), self.M, self.N, self.K,
                                    rows=rows)


def rounded_ref(ref, out_dtype):
    """The float64 reference correctly rounded (RNE) to the output type."""
    if out_dtype == "bf16":
        return oracle.bf16_bits_to_double_array(oracle.round_bf16_array(ref))
    return oracle.f16_bits_to_double_array(oracle.round_f16_array(ref))


def check_close(got, ref, out_dtype="f16", rel_max=REL_MAX, rel_mean=REL_MEAN, what=""):
    """rel_max against the float64 reference; rel_mean against it for fp16 outputs and
    against the correctly rounded reference for bf16 outputs, whose own rounding
    (8 significant bits) already costs ~1.4e-3 in mean relative error."""
    rmax, rmean = oracle.rel_errors(got, ref)
    mean_ref = ref if out_dtype == "f16" else rounded_ref(ref, out_dtype)
    _, rmean_vs = oracle.rel_errors(got, mean_ref)
    assert rmax <= rel_max and rmean_vs <= rel_mean, \
        f"{what} rel_max={rmax:.3e} rel_mean={rmean:.3e} rel_mean_vs_rounded={rmean_vs:.3e}"
    return rmax, rmean


class Int2Problem:
    """Seeded INT2 (W2A16) problem: canonical 2-bit codes on the device and packed scales."""

    def __init__(self, M, N, K, G, a_dtype="f16", seed=0, A_bits=None, codes=None):
        self.M, self.N, self.K, self.G, self.a_dtype = M, N, K, G, a_dtype
        self.A = A_bits if A_bits is not None else synth.activations(M, K, a_dtype, seed)
        self.wts = synth.int2_weights(N, K, G, seed + 1)
        if codes is not None:
            self.wts.w = oracle.pack_int2(codes)
        self.A_d = to_dev_f16bits(self.A, a_dtype)
        self.w_d = torch.from_numpy(self.wts.w).to(DEV)
        self.s_d = to_dev_f16bits(self.wts.s, "f16")
        import weight_only_quantized_tma_gb300 as wq
        self.sk = wq.wq_pack_int2_scales(self.s_d, N, K, G)

    def run(self):
        import weight_only_quantized_tma_gb300 as wq
        return wq.wq_gemm_w2a16(self.A_d, self.w_d, self.sk, self.N, self.K, self.G)

    def ref(self, rows=None):
        return oracle.gemm_w2a16(self.A, self.a_dtype == "bf16", self.wts.w, self.wts.s, self.M, self.N, self.K,
                                 self.G, rows=rows)

    def dequant_ref(self):
        return oracle.dequant_int2(self.wts.w, self.wts.s, self.K, self.G)
