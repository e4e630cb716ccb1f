"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
entry point include/wq.h declares, and rejects bad arguments before touching the
device (validation runs first; nothing is launched)."""
import ctypes
import os
import re

import pytest

import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wq.h")

OK, NULL, SHAPE, GROUP, MISALIGNED, DTYPE, WORKSPACE, UNSUPPORTED, CUDA, TIMEOUT = range(10)


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    return wq.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/wq.h but not exported"
    assert set(names) == set(_lib.exported_symbols())


def test_status_strings(L):
    for s in range(10):
        assert L.wq_status_string(s).decode().startswith(_lib.STATUS_NAMES[s])


def test_int4_packed_sizes(L):
    wb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.wq_int4_packed_bytes(4096, 4096, 128, ctypes.byref(wb), ctypes.byref(sb)) == OK
    assert wb.value == 4096 * 4096 // 2 and sb.value == 4096 * 32 * 2
    # N padded to 128, K to 256
    assert L.wq_int4_packed_bytes(200, 96, 32, ctypes.byref(wb), ctypes.byref(sb)) == OK
    assert wb.value == 256 * 256 // 2 and sb.value == 256 * (256 // 32) * 2
    assert L.wq_int4_packed_bytes(128, 100, 32, ctypes.byref(wb), ctypes.byref(sb)) == SHAPE
    assert L.wq_int4_packed_bytes(128, 256, 48, ctypes.byref(wb), ctypes.byref(sb)) == GROUP
    assert L.wq_int4_packed_bytes(128, 96, 64, ctypes.byref(wb), ctypes.byref(sb)) == GROUP


def test_fp4_sf_sizes(L):
    b = ctypes.c_size_t()
    assert L.wq_fp4_packed_sf_bytes(12800, 5120, ctypes.byref(b)) == OK
    assert b.value == 12800 * 5120 // 16
    assert L.wq_fp4_packed_sf_bytes(100, 96, ctypes.byref(b)) == OK
    assert b.value == 128 * 2 * 4          # N -> 128 rows, K -> 128 = two 64-wide quads, 4 bytes each
    assert L.wq_fp4_packed_sf_bytes(128, 160, ctypes.byref(b)) == OK
    assert b.value == 128 * 4 * 4          # K = 160 pads to 256: four quads


P = 0x10000  # a 16-byte-aligned fake device address: validation never dereferences it


def test_gemm_w4a16_validation(L):
    f = L.wq_gemm_w4a16
    assert f(None, 0, P, P, 4, 512, 1024, 128, P, None, 0, None) == NULL
    assert f(P, 0, P, P, -1, 512, 1024, 128, P, None, 0, None) == SHAPE
    assert f(P, 0, P, P, 4, 512, 1000, 128, P, None, 0, None) == SHAPE      # K % 32
    assert f(P, 0, P, P, 4, 500, 1024, 128, P, None, 0, None) == SHAPE      # N % 8
    assert f(P, 0, P, P, 4, 512, 1024, 96, P, None, 0, None) == GROUP
    assert f(P, 0, P, P, 4, 512, 1056, 64, P, None, 0, None) == GROUP       # K % G
    assert f(P, 7, P, P, 4, 512, 1024, 128, P, None, 0, None) == DTYPE
    assert f(P + 8, 0, P, P, 4, 512, 1024, 128, P, None, 0, None) == MISALIGNED
    assert f(P, 0, P, P + 4, 4, 512, 1024, 128, P, None, 0, None) == MISALIGNED
    assert f(P, 0, P, P, 4, 512, 1024, 128, P + 2, None, 0, None) == MISALIGNED


def test_gemm_fp8_validation(L):
    f = L.wq_gemm_w8a16_fp8
    assert f(P, 1, P, None, None, 4, 512, 1024, P, None, 0, None) == NULL    # alpha
    assert f(P, 1, P, P, None, 4, 512, 1000, P, None, 0, None) == SHAPE      # K % 16
    # a scalar alpha only needs 4-byte alignment (address % 16 == 4 is accepted by
    # validation; it only fails later for want of a device here)
    assert f(P, 1, P, P + 4, None, 4, 512, 1024, P, None, 0, None) != MISALIGNED
    assert f(P, 1, P, P + 2, None, 4, 512, 1024, P, None, 0, None) == MISALIGNED
    assert f(P, 1, P, P, P + 1, 4, 512, 1024, P, None, 0, None) == MISALIGNED   # bias


def test_gemm_fp4_validation(L):
    f = L.wq_gemm_bf16_fp4
    assert f(P, P, None, P, 4, 512, 1024, P, None, 0, None) == NULL
    assert f(P, P, P, P, 4, 512, 1040, P, None, 0, None) == SHAPE            # K % 32
    assert f(P, P + 8, P, P, 4, 512, 1024, P, None, 0, None) == MISALIGNED


def test_pack_validation(L):
    assert L.wq_pack_int4(None, P, 128, 256, 128, P, P, None) == NULL
    assert L.wq_pack_int4(P, P, 128, 250, 128, P, P, None) == SHAPE
    assert L.wq_pack_int4(P, P, 128, 256, 100, P, P, None) == GROUP
    assert L.wq_pack_int4(P, P, 128, 256, 128, P + 8, P, None) == MISALIGNED
    assert L.wq_pack_fp4_sf(P, 128, 100, P, None) == SHAPE


def test_no_device_is_an_error_not_a_crash(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = L.wq_gemm_w4a16(P, 0, P, P, 4, 512, 1024, 128, P, None, 0, None)
    assert st in (CUDA, UNSUPPORTED)


def test_python_binding_rejects_bad_tensors():
    import torch
    with pytest.raises(ValueError):
        wq.wq_gemm_w4a16(torch.zeros(4, 64, dtype=torch.float32), torch.zeros(1, dtype=torch.uint8),
                         torch.zeros(1, dtype=torch.float16), 128, 64, 32)


def test_gemm_lut_validation(L):
    f = L.wq_gemm_w4a16_lut
    assert f(P, 0, P, P, None, 4, 512, 1024, 128, P, None, 0, None) == NULL        # the table
    assert f(P, 0, P, P, P, 4, 512, 1000, 128, P, None, 0, None) == SHAPE          # K % 32
    assert f(P, 0, P, P, P, 4, 512, 1024, 96, P, None, 0, None) == GROUP
    assert f(P, 0, P, P, P + 2, 4, 512, 1024, 128, P, None, 0, None) == MISALIGNED  # two 16-byte vectors
    # an empty problem is valid and touches nothing
    assert f(None, 0, None, None, None, 0, 512, 1024, 128, None, None, 0, None) == OK
    d = L.wq_debug_dequant_int4_lut
    assert d(P, P, None, 512, 1024, 128, P, None) == NULL
    assert d(P, P, P + 1, 512, 1024, 128, P, None) == MISALIGNED


def test_int2_sizes_and_validation(L):
    b = ctypes.c_size_t()
    assert L.wq_int2_packed_scales_bytes(4096, 4096, 128, ctypes.byref(b)) == OK
    assert b.value == 4096 * 32 * 2
    assert L.wq_int2_packed_scales_bytes(200, 192, 64, ctypes.byref(b)) == OK
    assert b.value == 256 * (256 // 64) * 2          # N -> 256, K -> 256
    assert L.wq_int2_packed_scales_bytes(128, 96, 32, ctypes.byref(b)) == SHAPE    # K % 64
    assert L.wq_int2_packed_scales_bytes(128, 256, 48, ctypes.byref(b)) == GROUP
    f = L.wq_gemm_w2a16
    assert f(P, 0, None, P, 4, 512, 1024, 128, P, None, 0, None) == NULL
    assert f(P, 0, P, P, 4, 512, 1056, 32, P, None, 0, None) == SHAPE              # K % 64
    assert f(P, 0, P, P, 4, 500, 1024, 128, P, None, 0, None) == SHAPE             # N % 8
    assert f(P, 0, P, P, 4, 512, 1024, 96, P, None, 0, None) == GROUP
    assert f(P, 5, P, P, 4, 512, 1024, 128, P, None, 0, None) == DTYPE
    assert f(P, 0, P + 4, P, 4, 512, 1024, 128, P, None, 0, None) == MISALIGNED
    assert f(None, 0, None, None, 0, 512, 1024, 128, None, None, 0, None) == OK
    assert L.wq_pack_int2_scales(None, 128, 256, 128, P, None) == NULL
    assert L.wq_pack_int2_scales(P, 128, 256, 128, P + 8, None) == MISALIGNED
    assert L.wq_debug_dequant_int2(P, P, 128, 200, 40, P, None) == SHAPE


def test_gemm_zp_validation(L):
    f = L.wq_gemm_w4a16_zp
    assert f(P, 0, P, P, None, 4, 512, 1024, 128, P, None, 0, None) == NULL
    assert f(P, 0, P, P, P + 8, 4, 512, 1024, 128, P, None, 0, None) == MISALIGNED
    assert f(None, 0, None, None, None, 0, 512, 1024, 128, None, None, 0, None) == OK


def test_plan_ops_are_validated(L):
    plan = _lib.WqPlan()
    n = ctypes.c_size_t()
    assert L.wq_get_plan(9, 0, 4, 512, 1024, 128, ctypes.byref(plan), ctypes.byref(n)) == SHAPE
    assert L.wq_get_plan(_lib.WQ_OP_W2A16, 0, 4, 512, 1024, 100, ctypes.byref(plan), ctypes.byref(n)) == GROUP
    assert L.wq_get_plan(_lib.WQ_OP_W4A16_LUT, 3, 4, 512, 1024, 128, ctypes.byref(plan), ctypes.byref(n)) == DTYPE


# ------------------------------------------------------------- division by a runtime constant
#
# The tile walk and the split-K item decode divide work-item indices with a
# multiply-shift ("FlashInfer W8A16 GEMM (mm_bf16_fp8) analysis", §3(b): the
# divisor-1 magic number 2^40 overflowed int64 there).  The host copy of that
# division is checked here against plain integer division at its edges.

def _fastdiv(L, d, x_max, xs):
    import numpy as np
    x = np.ascontiguousarray(np.asarray(xs, dtype=np.uint32))
    q = np.zeros_like(x)
    used = ctypes.c_int32(-1)
    st = L.wq_debug_fastdiv(d, x_max, x.ctypes.data, x.size, q.ctypes.data, ctypes.byref(used))
    return st, q, used.value


def _edge_dividends(x_max, d):
    xs = {0, 1, 2, x_max, max(0, x_max - 1), max(0, x_max - d), max(0, x_max - d + 1)}
    for k in (1, 2, 3, 7):
        for base in (k * d, (x_max // d) * d):
            for off in (-1, 0, 1):
                v = base + off
                if 0 <= v <= x_max:
                    xs.add(v)
    return sorted(v for v in xs if v <= x_max)


@pytest.mark.parametrize("d", [1, 2, 3, 7, 128, 152, 304, 1000, 65535, 65536, (1 << 20) + 1, (1 << 31) - 1])
@pytest.mark.parametrize("x_max", [1, 1000, 123456, (1 << 20), (1 << 31) - 1])
def test_fastdiv_matches_integer_division(L, d, x_max):
    import random
    rnd = random.Random(d * 7919 + x_max)
    xs = _edge_dividends(x_max, d) + [rnd.randint(0, x_max) for _ in range(2000)]
    st, q, used = _fastdiv(L, d, x_max, xs)
    assert st == OK
    assert [int(v) for v in q] == [x // d for x in xs]
    assert used in (0, 1)


def test_fastdiv_overflow_guard_falls_back(L):
    # the guard: the multiply-shift is used only while x_max * magic fits in 63 bits.
    # For the largest divisors the magic number is just under 2^32:
    for d in [(1 << 30) + 1, (1 << 30) + 12345, (1 << 31) - 3, (1 << 31) - 1]:
        for x_max in [(1 << 31) - 1, 1 << 30, 3]:
            xs = _edge_dividends(x_max, d)
            st, q, used = _fastdiv(L, d, x_max, xs)
            assert st == OK
            assert [int(v) for v in q] == [x // d for x in xs]
            # magic = ceil(2^(31+l) / d) <= 2^32, so x_max * magic < 2^63 for every
            # x_max < 2^31: the multiply path is safe and must be the one taken
            assert used == 1
    # divisor 1 has magic 2^31 exactly: 2^31 * x_max < 2^62, multiply path, exact
    st, q, used = _fastdiv(L, 1, (1 << 31) - 1, [0, 1, (1 << 31) - 1])
    assert st == OK and [int(v) for v in q] == [0, 1, (1 << 31) - 1] and used == 1
    # dividends or divisors at or beyond 2^31 are outside the multiply-shift's range:
    # plain division, still exact
    st, q, used = _fastdiv(L, 3, (1 << 32) - 1, [(1 << 32) - 1, 1 << 31])
    assert st == OK and [int(v) for v in q] == [((1 << 32) - 1) // 3, (1 << 31) // 3] and used == 0
    st, q, used = _fastdiv(L, (1 << 31) + 5, (1 << 32) - 1, [(1 << 32) - 1])
    assert st == OK and int(q[0]) == ((1 << 32) - 1) // ((1 << 31) + 5) and used == 0


def test_fastdiv_argument_checks(L):
    used = ctypes.c_int32()
    assert L.wq_debug_fastdiv(0, 10, None, 0, None, ctypes.byref(used)) == SHAPE
    assert L.wq_debug_fastdiv(3, 10, None, 1, None, ctypes.byref(used)) == NULL
    st, _, _ = _fastdiv(L, 3, 10, [11])
    assert st == SHAPE
