"""GPU parity of the synthetic INT4 quantiser (wq_quantize_int4) against the oracle.

The quantiser is the step upstream of the packing ("Low Bit Triton Kernels", hands-on
exercise 1: fp16 weight -> group-wise quantize -> two nibbles per byte, checked by a
round trip).  Codes and scales are integers / fp16 values decided the same way on both
sides, so they must match bit for bit.  The pipeline test quantises on the GPU, packs,
runs the W4A16 GEMM and reports the quantisation error against the fp16 weight.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, check_close, out_to_f64, to_dev_f16bits

pytestmark = pytest.mark.gpu


def _weights(N, K, G, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    W[1, :G] = 0                                   # all-zero group: S = 0, q = 8
    W[2, G:2 * G] *= np.float16(1e-3)              # subnormal scale
    W[3, :G] = np.float16(60000.0) * np.sign(W[3, :G])   # near the top of the fp16 range
    # exact half-way quotients: S = 2^-6 (amax = 7 S), elements (j + 1/2) S
    S = 2.0 ** -6
    ties = (np.arange(G) % 14 - 7 + 0.5) * S
    ties[0] = 7 * S
    W[4, :G] = ties.astype(np.float16)
    return W


@pytest.mark.parametrize("G", [32, 64, 128, 256])
@pytest.mark.parametrize("N,K", [(64, 1024), (200, 2048 + 256)])
def test_quantiser_bit_exact(N, K, G):
    W = _weights(N, K, G, seed=400 + G + N)
    w_ref, s_ref = oracle.quantize_int4(W.view(np.uint16), G)
    w_d, s_d = wq.wq_quantize_int4(to_dev_f16bits(W.view(np.uint16), "f16"), G)
    torch.cuda.synchronize()
    assert np.array_equal(w_d.cpu().numpy(), w_ref)
    assert np.array_equal(s_d.view(torch.int16).cpu().numpy().view(np.uint16), s_ref)


def test_quantiser_rejects_bad_arguments():
    W = torch.zeros((8, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(wq.WQError):
        wq.wq_quantize_int4(W, 48)                 # G not in {32, 64, 128, 256}
    with pytest.raises(wq.WQError):
        wq.wq_quantize_int4(torch.zeros((8, 48), dtype=torch.float16, device=DEV), 32)   # K % 32
    with pytest.raises(ValueError):
        wq.wq_quantize_int4(W.float(), 32)


@pytest.mark.parametrize("G", [32, 128])
def test_quantise_pack_gemm_pipeline(G):
    # fp16 W -> wq_quantize_int4 -> wq_pack_int4 -> wq_gemm_w4a16: the GEMM matches the
    # oracle on the quantised weight, and the error against the unquantised fp16 weight
    # is the quantisation error the page asks to look at as a distribution
    M, N, K = 16, 1024, 4096
    W = (np.random.default_rng(410 + G).standard_normal((N, K)) * 0.02).astype(np.float16)
    A_bits = synth.activations(M, K, "f16", 411)
    w_c, s_c = wq.wq_quantize_int4(to_dev_f16bits(W.view(np.uint16), "f16"), G)
    wk, sk = wq.wq_pack_int4(w_c, s_c, N, K, G)
    out = wq.wq_gemm_w4a16(to_dev_f16bits(A_bits, "f16"), wk, sk, N, K, G)
    torch.cuda.synchronize()
    w_ref, s_ref = oracle.quantize_int4(W.view(np.uint16), G)
    ref_q = oracle.gemm_w4a16(A_bits, False, w_ref, s_ref, M, N, K, G)
    check_close(out_to_f64(out), ref_q, what=f"quantised GEMM G={G}")
    ref_fp16 = A_bits.view(np.float16).astype(np.float64) @ W.astype(np.float64).T
    rel_max, rel_mean = oracle.rel_errors(out_to_f64(out), ref_fp16)
    print(f"quantisation error (G={G}) vs fp16 weight: rel_max {rel_max:.3f} rel_mean {rel_mean:.3f}")
    # symmetric 4-bit with amax / 7 steps: the step is ~2.5/7 of the group's rms range;
    # the rounding noise of a K-long dot product stays near 0.1 of the output's scale
    assert rel_mean < 0.15 and (G == 32 or rel_mean > 0.05)
