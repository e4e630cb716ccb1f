"""ctypes binding of libwq.so (include/wq.h).

Argument marshalling only: torch tensors are checked for device, dtype, shape
and contiguity, then their data pointers, the sizes and the current CUDA stream
are passed to the C entry point of the same name.  Every step of the GEMM runs
in the library's CUDA kernels; there is no fallback: if libwq.so is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")

WQ_F16, WQ_BF16 = 0, 1
WQ_OP_W4A16, WQ_OP_FP8, WQ_OP_FP4, WQ_OP_W4A16_ZP, WQ_OP_W4A16_LUT, WQ_OP_W2A16 = 0, 1, 2, 3, 4, 5
WQ_KERNEL_TILE, WQ_KERNEL_DECODE, WQ_KERNEL_TILE_PAIR = 0, 1, 2
STATUS_NAMES = {
    0: "WQ_OK", 1: "WQ_ERR_NULL", 2: "WQ_ERR_SHAPE", 3: "WQ_ERR_GROUP", 4: "WQ_ERR_MISALIGNED",
    5: "WQ_ERR_DTYPE", 6: "WQ_ERR_WORKSPACE", 7: "WQ_ERR_UNSUPPORTED_DEVICE", 8: "WQ_ERR_CUDA",
    9: "WQ_ERR_TIMEOUT",
}

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t


class WQError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


class WqPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "bn", "bk", "stages", "splits", "grid", "threads", "smem_bytes", "n_items", "walk_n_fast",
        "tiles_n", "tiles_m", "ctas_per_sm", "kernel", "cluster_split", "cluster_capacity")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_SIGNATURES = {
    "wq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "wq_int4_packed_bytes": (ctypes.c_int, [_i64, _i64, _i32, ctypes.POINTER(_sz), ctypes.POINTER(_sz)]),
    "wq_pack_int4": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "wq_quantize_int4": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "wq_unpack_int4": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "wq_debug_dequant_int4": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "wq_gemm_w4a16": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _sz, _vp]),
    "wq_int4_packed_zeros_bytes": (ctypes.c_int, [_i64, _i64, _i32, ctypes.POINTER(_sz)]),
    "wq_pack_int4_zeros": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp]),
    "wq_gemm_w4a16_zp": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _sz,
                                        _vp]),
    "wq_gemm_w4a16_lut": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _sz,
                                         _vp]),
    "wq_debug_dequant_int4_lut": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "wq_int2_packed_scales_bytes": (ctypes.c_int, [_i64, _i64, _i32, ctypes.POINTER(_sz)]),
    "wq_pack_int2_scales": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp]),
    "wq_debug_dequant_int2": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "wq_gemm_w2a16": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _sz, _vp]),
    "wq_debug_dequant_fp8": (ctypes.c_int, [_vp, _i64, _i64, ctypes.c_int, _vp, _vp]),
    "wq_gemm_w8a16_fp8": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "wq_fp4_packed_sf_bytes": (ctypes.c_int, [_i64, _i64, ctypes.POINTER(_sz)]),
    "wq_pack_fp4_sf": (ctypes.c_int, [_vp, _i64, _i64, _vp, _vp]),
    "wq_debug_dequant_fp4": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp]),
    "wq_gemm_bf16_fp4": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "wq_get_plan": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _i32, ctypes.POINTER(WqPlan),
                                   ctypes.POINTER(_sz)]),
    "wq_workspace_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _i32,
                                          ctypes.POINTER(_sz)]),
    "wq_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "wq_clear_device_status": (ctypes.c_int, []),
    "wq_debug_wait_probe": (ctypes.c_int, [_i64, _vp]),
    "wq_gemm_w4a16_noalloc": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp]),
    "wq_debug_fastdiv": (ctypes.c_int, [ctypes.c_uint32, ctypes.c_uint32, _vp, _i64, _vp, ctypes.POINTER(_i32)]),
}

WQ_NOALLOC_SCRATCH_BYTES = 8 << 20


def lib():
    """The loaded libwq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(the library has no CPU fallback)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def exported_symbols():
    return sorted(_SIGNATURES)


def _check(status: int, fn: str):
    if status != 0:
        raise WQError(status, fn)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _adtype(A: torch.Tensor) -> int:
    if A.dtype == torch.float16:
        return WQ_F16
    if A.dtype == torch.bfloat16:
        return WQ_BF16
    raise ValueError(f"activations must be float16 or bfloat16, got {A.dtype}")


# ------------------------------------------------------------------ workspaces

_ws_cache: dict = {}


def workspace(op: int, a_dtype: int, M: int, N: int, K: int, G: int, device) -> tuple:
    """(tensor or None, bytes): a zero-filled workspace shared by calls on one stream."""
    need = _sz(0)
    _check(lib().wq_workspace_bytes(op, a_dtype, M, N, K, G, ctypes.byref(need)), "wq_workspace_bytes")
    if need.value == 0:
        return None, 0
    dev = torch.device(device)
    key = (dev.index if dev.index is not None else torch.cuda.current_device(),
           torch.cuda.current_stream(dev).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < need.value:
        buf = torch.zeros(max(need.value, 1 << 20), dtype=torch.uint8, device=dev)
        _ws_cache[key] = buf
    return buf, buf.numel()


def get_plan(op: int, a_dtype: int, M: int, N: int, K: int, G: int = 128) -> dict:
    plan = WqPlan()
    ws = _sz(0)
    _check(lib().wq_get_plan(op, a_dtype, M, N, K, G, ctypes.byref(plan), ctypes.byref(ws)), "wq_get_plan")
    d = plan.as_dict()
    d["ws_bytes"] = ws.value
    return d


# ------------------------------------------------------------------ INT4

def wq_int4_packed_bytes(N: int, K: int, G: int):
    wb, sb = _sz(0), _sz(0)
    _check(lib().wq_int4_packed_bytes(N, K, G, ctypes.byref(wb), ctypes.byref(sb)), "wq_int4_packed_bytes")
    return wb.value, sb.value


def wq_pack_int4(w_canon: torch.Tensor, s_canon: torch.Tensor, N: int, K: int, G: int):
    """Canonical uint8 [N, K/2] codes + fp16 [K/G, N] scales -> kernel-order buffers."""
    _need(w_canon, "w_canon", torch.uint8, (N, K // 2))
    _need(s_canon, "s_canon", torch.float16, (K // G, N))
    wb, sb = wq_int4_packed_bytes(N, K, G)
    wk = torch.empty(wb, dtype=torch.uint8, device=w_canon.device)
    sk = torch.empty(sb // 2, dtype=torch.float16, device=w_canon.device)
    _check(lib().wq_pack_int4(_ptr(w_canon), _ptr(s_canon), N, K, G, _ptr(wk), _ptr(sk), _stream(w_canon)),
           "wq_pack_int4")
    return wk, sk


def wq_quantize_int4(w: torch.Tensor, G: int):
    """fp16 weight [N, K] -> canonical uint8 codes [N, K/2] + fp16 scales [K/G, N]
    (group-wise symmetric: S = RN16(amax / 7), q = clamp(rint(w / S) + 8, 0, 15))."""
    if w.dtype != torch.float16 or w.dim() != 2:
        raise ValueError("wq_quantize_int4: w must be a 2-D float16 tensor")
    w = w.contiguous()
    N, K = w.shape
    w_canon = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    s_canon = torch.empty((K // G, N), dtype=torch.float16, device=w.device)
    _check(lib().wq_quantize_int4(_ptr(w), N, K, G, _ptr(w_canon), _ptr(s_canon), _stream(w)), "wq_quantize_int4")
    return w_canon, s_canon


def wq_unpack_int4(w_kernel: torch.Tensor, s_kernel: torch.Tensor, N: int, K: int, G: int):
    w = torch.empty((N, K // 2), dtype=torch.uint8, device=w_kernel.device)
    s = torch.empty((K // G, N), dtype=torch.float16, device=w_kernel.device)
    _check(lib().wq_unpack_int4(_ptr(w_kernel), _ptr(s_kernel), N, K, G, _ptr(w), _ptr(s), _stream(w_kernel)),
           "wq_unpack_int4")
    return w, s


def wq_debug_dequant_int4(w_kernel: torch.Tensor, s_kernel: torch.Tensor, N: int, K: int, G: int):
    out = torch.empty((N, K), dtype=torch.float32, device=w_kernel.device)
    _check(lib().wq_debug_dequant_int4(_ptr(w_kernel), _ptr(s_kernel), N, K, G, _ptr(out), _stream(w_kernel)),
           "wq_debug_dequant_int4")
    return out


def wq_gemm_w4a16(A: torch.Tensor, w_kernel: torch.Tensor, s_kernel: torch.Tensor, N: int, K: int, G: int,
                  out: torch.Tensor = None, ws: torch.Tensor = None) -> torch.Tensor:
    """out[M, N] = A[M, K] . ((q - 8) * S)^T, out in the dtype of A."""
    a_dtype = _adtype(A)
    _need(A, "A", A.dtype)
    if A.dim() != 2 or A.shape[1] != K:
        raise ValueError(f"A must be [M, {K}]")
    M = A.shape[0]
    _need(w_kernel, "w_kernel", torch.uint8)
    _need(s_kernel, "s_kernel", torch.float16)
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _need(out, "out", A.dtype, (M, N))
    if ws is None:
        ws, ws_bytes = workspace(WQ_OP_W4A16, a_dtype, M, N, K, G, A.device)
    else:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().wq_gemm_w4a16(_ptr(A), a_dtype, _ptr(w_kernel), _ptr(s_kernel), M, N, K, G, _ptr(out), _ptr(ws),
                               ws_bytes, _stream(A)), "wq_gemm_w4a16")
    return out


def wq_int4_packed_zeros_bytes(N: int, K: int, G: int) -> int:
    zb = _sz(0)
    _check(lib().wq_int4_packed_zeros_bytes(N, K, G, ctypes.byref(zb)), "wq_int4_packed_zeros_bytes")
    return zb.value


def wq_pack_int4_zeros(z_canon: torch.Tensor, N: int, K: int, G: int) -> torch.Tensor:
    """Canonical uint8 zero points [K/G, N] (0..15) -> kernel-order buffer."""
    _need(z_canon, "z_canon", torch.uint8, (K // G, N))
    zk = torch.empty(wq_int4_packed_zeros_bytes(N, K, G), dtype=torch.uint8, device=z_canon.device)
    _check(lib().wq_pack_int4_zeros(_ptr(z_canon), N, K, G, _ptr(zk), _stream(z_canon)), "wq_pack_int4_zeros")
    return zk


def wq_gemm_w4a16_zp(A: torch.Tensor, w_kernel: torch.Tensor, s_kernel: torch.Tensor, z_kernel: torch.Tensor,
                     N: int, K: int, G: int, out: torch.Tensor = None, ws: torch.Tensor = None) -> torch.Tensor:
    """out[M, N] = A[M, K] . ((q - Z) * S)^T, out in the dtype of A."""
    a_dtype = _adtype(A)
    _need(A, "A", A.dtype)
    if A.dim() != 2 or A.shape[1] != K:
        raise ValueError(f"A must be [M, {K}]")
    M = A.shape[0]
    _need(w_kernel, "w_kernel", torch.uint8)
    _need(s_kernel, "s_kernel", torch.float16)
    _need(z_kernel, "z_kernel", torch.uint8)
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _need(out, "out", A.dtype, (M, N))
    if ws is None:
        ws, ws_bytes = workspace(WQ_OP_W4A16_ZP, a_dtype, M, N, K, G, A.device)
    else:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().wq_gemm_w4a16_zp(_ptr(A), a_dtype, _ptr(w_kernel), _ptr(s_kernel), _ptr(z_kernel), M, N, K, G,
                                  _ptr(out), _ptr(ws), ws_bytes, _stream(A)), "wq_gemm_w4a16_zp")
    return out


def wq_gemm_w4a16_lut(A: torch.Tensor, w_kernel: torch.Tensor, s_kernel: torch.Tensor, lut: torch.Tensor,
                      N: int, K: int, G: int, out: torch.Tensor = None, ws: torch.Tensor = None) -> torch.Tensor:
    """out[M, N] = A[M, K] . (LUT[q] * S)^T with a 16-entry fp16 codebook, out in the dtype of A."""
    a_dtype = _adtype(A)
    _need(A, "A", A.dtype)
    if A.dim() != 2 or A.shape[1] != K:
        raise ValueError(f"A must be [M, {K}]")
    M = A.shape[0]
    _need(w_kernel, "w_kernel", torch.uint8)
    _need(s_kernel, "s_kernel", torch.float16)
    _need(lut, "lut", torch.float16, (16,))
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _need(out, "out", A.dtype, (M, N))
    if ws is None:
        ws, ws_bytes = workspace(WQ_OP_W4A16_LUT, a_dtype, M, N, K, G, A.device)
    else:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().wq_gemm_w4a16_lut(_ptr(A), a_dtype, _ptr(w_kernel), _ptr(s_kernel), _ptr(lut), M, N, K, G,
                                   _ptr(out), _ptr(ws), ws_bytes, _stream(A)), "wq_gemm_w4a16_lut")
    return out


def wq_debug_dequant_int4_lut(w_kernel: torch.Tensor, s_kernel: torch.Tensor, lut: torch.Tensor, N: int, K: int,
                              G: int) -> torch.Tensor:
    _need(lut, "lut", torch.float16, (16,))
    out = torch.empty((N, K), dtype=torch.float32, device=w_kernel.device)
    _check(lib().wq_debug_dequant_int4_lut(_ptr(w_kernel), _ptr(s_kernel), _ptr(lut), N, K, G, _ptr(out),
                                           _stream(w_kernel)), "wq_debug_dequant_int4_lut")
    return out


def wq_int2_packed_scales_bytes(N: int, K: int, G: int) -> int:
    sb = _sz(0)
    _check(lib().wq_int2_packed_scales_bytes(N, K, G, ctypes.byref(sb)), "wq_int2_packed_scales_bytes")
    return sb.value


def wq_pack_int2_scales(s_canon: torch.Tensor, N: int, K: int, G: int) -> torch.Tensor:
    """fp16 scales [K/G, N] -> the kernel-order scale buffer of the INT2 GEMM."""
    _need(s_canon, "s_canon", torch.float16, (K // G, N))
    sk = torch.empty(wq_int2_packed_scales_bytes(N, K, G) // 2, dtype=torch.float16, device=s_canon.device)
    _check(lib().wq_pack_int2_scales(_ptr(s_canon), N, K, G, _ptr(sk), _stream(s_canon)), "wq_pack_int2_scales")
    return sk


def wq_debug_dequant_int2(w_canon: torch.Tensor, s_kernel: torch.Tensor, N: int, K: int, G: int) -> torch.Tensor:
    _need(w_canon, "w_canon", torch.uint8, (N, K // 4))
    out = torch.empty((N, K), dtype=torch.float32, device=w_canon.device)
    _check(lib().wq_debug_dequant_int2(_ptr(w_canon), _ptr(s_kernel), N, K, G, _ptr(out), _stream(w_canon)),
           "wq_debug_dequant_int2")
    return out


def wq_gemm_w2a16(A: torch.Tensor, w_canon: torch.Tensor, s_kernel: torch.Tensor, N: int, K: int, G: int,
                  out: torch.Tensor = None, ws: torch.Tensor = None) -> torch.Tensor:
    """out[M, N] = A[M, K] . ((q - 2) * S)^T, 2-bit codes [N, K/4], out in the dtype of A."""
    a_dtype = _adtype(A)
    _need(A, "A", A.dtype)
    if A.dim() != 2 or A.shape[1] != K:
        raise ValueError(f"A must be [M, {K}]")
    M = A.shape[0]
    _need(w_canon, "w_canon", torch.uint8, (N, K // 4))
    _need(s_kernel, "s_kernel", torch.float16)
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _need(out, "out", A.dtype, (M, N))
    if ws is None:
        ws, ws_bytes = workspace(WQ_OP_W2A16, a_dtype, M, N, K, G, A.device)
    else:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().wq_gemm_w2a16(_ptr(A), a_dtype, _ptr(w_canon), _ptr(s_kernel), M, N, K, G, _ptr(out), _ptr(ws),
                               ws_bytes, _stream(A)), "wq_gemm_w2a16")
    return out


def wq_gemm_w4a16_noalloc(A: torch.Tensor, w_kernel: torch.Tensor, s_kernel: torch.Tensor, N: int, K: int, G: int,
                          out: torch.Tensor = None) -> torch.Tensor:
    """wq_gemm_w4a16 without a workspace argument, for callers that cannot allocate
    device memory (the split-K scratch is a fixed array inside the library).  The C
    entry point allocates nothing; pass `out` as well for the whole call to allocate
    nothing (when `out` is None this wrapper creates it with torch.empty)."""
    a_dtype = _adtype(A)
    _need(A, "A", A.dtype)
    if A.dim() != 2 or A.shape[1] != K:
        raise ValueError(f"A must be [M, {K}]")
    M = A.shape[0]
    _need(w_kernel, "w_kernel", torch.uint8)
    _need(s_kernel, "s_kernel", torch.float16)
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _need(out, "out", A.dtype, (M, N))
    _check(lib().wq_gemm_w4a16_noalloc(_ptr(A), a_dtype, _ptr(w_kernel), _ptr(s_kernel), M, N, K, G, _ptr(out),
                                       _stream(A)), "wq_gemm_w4a16_noalloc")
    return out


# ------------------------------------------------------------------ FP8

def wq_debug_dequant_fp8(w: torch.Tensor, operand_bf16: bool = True) -> torch.Tensor:
    _need(w, "w", torch.uint8)
    N, K = w.shape
    out = torch.empty((N, K), dtype=torch.float32, device=w.device)
    _check(lib().wq_debug_dequant_fp8(_ptr(w), N, K, WQ_BF16 if operand_bf16 else WQ_F16, _ptr(out), _stream(w)),
           "wq_debug_dequant_fp8")
    return out


def wq_gemm_w8a16_fp8(A: torch.Tensor, w: torch.Tensor, alpha: torch.Tensor, bias: torch.Tensor = None,
                      out: torch.Tensor = None, ws: torch.Tensor = None) -> torch.Tensor:
    """out = alpha * (A . e4m3(W)^T) + bias; w is uint8 (e4m3 codes) [N, K], alpha a 1-element fp32 tensor."""
    a_dtype = _adtype(A)
    _need(A, "A", A.dtype)
    if w.dtype == getattr(torch, "float8_e4m3fn", None):
        w = w.view(torch.uint8)
    _need(w, "w", torch.uint8)
    N, K = w.shape
    if A.dim() != 2 or A.shape[1] != K:
        raise ValueError(f"A must be [M, {K}]")
    M = A.shape[0]
    _need(alpha, "alpha", torch.float32)
    if alpha.numel() != 1:
        raise ValueError("alpha must hold one element")
    if bias is not None:
        _need(bias, "bias", A.dtype, (N,))
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _need(out, "out", A.dtype, (M, N))
    if ws is None:
        ws, ws_bytes = workspace(WQ_OP_FP8, a_dtype, M, N, K, 0, A.device)
    else:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().wq_gemm_w8a16_fp8(_ptr(A), a_dtype, _ptr(w), _ptr(alpha), _ptr(bias), M, N, K, _ptr(out),
                                   _ptr(ws), ws_bytes, _stream(A)), "wq_gemm_w8a16_fp8")
    return out


# ------------------------------------------------------------------ FP4

def wq_fp4_packed_sf_bytes(N: int, K: int) -> int:
    b = _sz(0)
    _check(lib().wq_fp4_packed_sf_bytes(N, K, ctypes.byref(b)), "wq_fp4_packed_sf_bytes")
    return b.value


def wq_pack_fp4_sf(sf: torch.Tensor, N: int, K: int) -> torch.Tensor:
    """e4m3 block scales uint8 [N, K/16] -> kernel order."""
    if sf.dtype == getattr(torch, "float8_e4m3fn", None):
        sf = sf.view(torch.uint8)
    _need(sf, "sf", torch.uint8, (N, K // 16))
    out = torch.empty(wq_fp4_packed_sf_bytes(N, K), dtype=torch.uint8, device=sf.device)
    _check(lib().wq_pack_fp4_sf(_ptr(sf), N, K, _ptr(out), _stream(sf)), "wq_pack_fp4_sf")
    return out


def wq_debug_dequant_fp4(w: torch.Tensor, sf_kernel: torch.Tensor, N: int, K: int) -> torch.Tensor:
    _need(w, "w", torch.uint8, (N, K // 2))
    out = torch.empty((N, K), dtype=torch.float32, device=w.device)
    _check(lib().wq_debug_dequant_fp4(_ptr(w), _ptr(sf_kernel), N, K, _ptr(out), _stream(w)),
           "wq_debug_dequant_fp4")
    return out


def wq_gemm_bf16_fp4(A: torch.Tensor, w: torch.Tensor, sf_kernel: torch.Tensor, alpha: torch.Tensor,
                     out: torch.Tensor = None, ws: torch.Tensor = None) -> torch.Tensor:
    """out bf16 = alpha * (A . (e2m1(W) * e4m3(SF))^T); w uint8 [N, K/2], sf_kernel from wq_pack_fp4_sf."""
    _need(A, "A", torch.bfloat16)
    _need(w, "w", torch.uint8)
    N, K = w.shape[0], w.shape[1] * 2
    if A.dim() != 2 or A.shape[1] != K:
        raise ValueError(f"A must be [M, {K}]")
    M = A.shape[0]
    _need(sf_kernel, "sf_kernel", torch.uint8)
    _need(alpha, "alpha", torch.float32)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(out, "out", torch.bfloat16, (M, N))
    if ws is None:
        ws, ws_bytes = workspace(WQ_OP_FP4, WQ_BF16, M, N, K, 0, A.device)
    else:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().wq_gemm_bf16_fp4(_ptr(A), _ptr(w), _ptr(sf_kernel), _ptr(alpha), M, N, K, _ptr(out), _ptr(ws),
                                  ws_bytes, _stream(A)), "wq_gemm_bf16_fp4")
    return out


# ------------------------------------------------------------------ device status

def wq_device_status() -> int:
    bits = ctypes.c_uint32(0)
    st = lib().wq_device_status(ctypes.byref(bits))
    if st not in (0, 9):
        raise WQError(st, "wq_device_status")
    return bits.value


def wq_clear_device_status():
    _check(lib().wq_clear_device_status(), "wq_clear_device_status")


def wq_debug_wait_probe(timeout_ns: int):
    _check(lib().wq_debug_wait_probe(int(timeout_ns), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)),
           "wq_debug_wait_probe")
