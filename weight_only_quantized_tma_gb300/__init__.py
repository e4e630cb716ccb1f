"""Weight-only quantized GEMM for GB300 (sm_103a).

out[M, N] = A[M, K] . dequant(W)[N, K]^T with fp16/bf16 activations, fp32
accumulation, and INT4 (group-scaled, symmetric, zero-point or codebook), INT2
(group-scaled), FP8-e4m3 (per-tensor scale) or FP4-e2m1 (block-scaled) weights.  The computation runs in hand-written CUDA kernels in
libwq.so (C ABI: include/wq.h); this package only binds it.
"""
from ._lib import (  # noqa: F401
    WQError,
    get_plan,
    lib,
    wq_clear_device_status,
    wq_debug_dequant_fp4,
    wq_debug_dequant_fp8,
    wq_debug_dequant_int2,
    wq_debug_dequant_int4,
    wq_debug_dequant_int4_lut,
    wq_debug_wait_probe,
    wq_device_status,
    wq_fp4_packed_sf_bytes,
    wq_gemm_bf16_fp4,
    wq_gemm_w2a16,
    wq_gemm_w4a16,
    wq_gemm_w4a16_lut,
    wq_gemm_w4a16_noalloc,
    wq_gemm_w4a16_zp,
    wq_gemm_w8a16_fp8,
    wq_int2_packed_scales_bytes,
    wq_int4_packed_bytes,
    wq_int4_packed_zeros_bytes,
    wq_pack_fp4_sf,
    wq_pack_int2_scales,
    wq_pack_int4,
    wq_pack_int4_zeros,
    wq_quantize_int4,
    wq_unpack_int4,
    WQ_BF16,
    WQ_F16,
    WQ_KERNEL_DECODE,
    WQ_KERNEL_TILE,
    WQ_KERNEL_TILE_PAIR,
    WQ_OP_FP4,
    WQ_OP_FP8,
    WQ_OP_W4A16,
    WQ_OP_W2A16,
    WQ_OP_W4A16_LUT,
    WQ_OP_W4A16_ZP,
)
