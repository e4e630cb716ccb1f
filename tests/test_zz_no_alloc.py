"""wq_gemm_w4a16_noalloc: the W4A16 GEMM for callers that cannot allocate device memory.

A framework that owns all device memory through its own pool, or a decode loop in
which cudaMalloc (and the device synchronisation it may cause) is not allowed, cannot
hand the GEMM a split-K workspace.  This entry point uses a fixed scratch array built
into the library instead.  The test calls it through the C ABI twice in a row and
checks each result against the workspace entry point, with the tolerance the other
tests use, and checks that the two calls leave the device's free memory unchanged.
The file is named to be collected last, and it works in a fresh process as well as
after the other tests.
"""
import ctypes

import pytest
import torch

import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import _lib

from gpu_helpers import Int4Problem, check_close, out_to_f64

pytestmark = pytest.mark.gpu

WQ_ERR_WORKSPACE = 6


def _call(L, p, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    a_dtype = wq.WQ_BF16 if p.a_dtype == "bf16" else wq.WQ_F16
    return L.wq_gemm_w4a16_noalloc(ctypes.c_void_p(p.A_d.data_ptr()), a_dtype, ctypes.c_void_p(p.wk.data_ptr()),
                                   ctypes.c_void_p(p.sk.data_ptr()), p.M, p.N, p.K, p.G,
                                   ctypes.c_void_p(out.data_ptr()), stream)


def _torch_dtype(a_dtype):
    return torch.bfloat16 if a_dtype == "bf16" else torch.float16


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,scratch", [(32, 1024, 1024, True), (20, 512, 2048, True), (32, 4096, 1024, False),
                                           (1, 11008, 4096, False), (16, 4096, 4096, False)])
def test_noalloc_matches_workspace_entry_on_two_calls(M, N, K, scratch, a_dtype, monkeypatch):
    G = 128
    if scratch:
        # tile-kernel split-K with the workspace reduction (the tile kernel otherwise
        # reduces its slices inside a cluster): the built-in scratch is really exercised
        monkeypatch.setenv("WQ_SPLITK_WORKSPACE", "1")
    op_dtype = wq.WQ_BF16 if a_dtype == "bf16" else wq.WQ_F16
    plan = wq.get_plan(wq.WQ_OP_W4A16, op_dtype, M, N, K, G)
    if scratch:
        assert plan["splits"] > 1 and 0 < plan["ws_bytes"] <= _lib.WQ_NOALLOC_SCRATCH_BYTES
        assert plan["cluster_split"] == 0
    else:
        # the decode kernel and the tile kernel's cluster split-K need no scratch
        assert plan["ws_bytes"] == 0
    p = Int4Problem(M, N, K, G, a_dtype=a_dtype, seed=901 + M).pack()
    expected = p.run()                       # the entry point with a caller workspace
    torch.cuda.synchronize()
    L = wq.lib()
    outs = [torch.full((M, N), float("nan"), dtype=_torch_dtype(a_dtype), device=p.A_d.device) for _ in range(3)]
    # a first call looks the scratch array up and loads the kernels
    assert _call(L, p, outs[0]) == 0
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for out in outs[1:]:
        assert _call(L, p, out) == 0
        torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "the no-allocation entry point changed free device memory"
    ref = p.ref() if a_dtype == "f16" else None
    for out in outs:
        check_close(out_to_f64(out), out_to_f64(expected), out_dtype=a_dtype, what="noalloc vs workspace entry")
        if ref is not None:
            # (bf16 activations: the workspace entry point's own accuracy is gated by the
            # INT4 parity tests; here the two entry points must agree)
            check_close(out_to_f64(out), ref, what="noalloc vs oracle")


@pytest.mark.parametrize("a_dtype", ["f16", "bf16"])
def test_noalloc_python_binding(a_dtype, monkeypatch):
    # the Python wrapper, with the output passed in, on the scratch-using path
    monkeypatch.setenv("WQ_SPLITK_WORKSPACE", "1")
    M, N, K, G = 32, 1024, 1024, 128
    p = Int4Problem(M, N, K, G, a_dtype=a_dtype, seed=960).pack()
    expected = p.run()
    out = torch.empty((M, N), dtype=_torch_dtype(a_dtype), device=p.A_d.device)
    for _ in range(2):
        got = wq.wq_gemm_w4a16_noalloc(p.A_d, p.wk, p.sk, N, K, G, out=out)
        torch.cuda.synchronize()
        assert got is out
        check_close(out_to_f64(got), out_to_f64(expected), out_dtype=a_dtype, what="noalloc binding")
    with pytest.raises(ValueError):
        wq.wq_gemm_w4a16_noalloc(p.A_d[:, : K // 2].contiguous(), p.wk, p.sk, N, K, G, out=out)


def test_noalloc_rejects_problems_beyond_its_scratch(monkeypatch):
    monkeypatch.setenv("WQ_SPLITK_WORKSPACE", "1")
    M, N, K, G = 256, 2048, 4096, 128
    plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, G)
    assert plan["ws_bytes"] > _lib.WQ_NOALLOC_SCRATCH_BYTES
    p = Int4Problem(M, N, K, G, seed=950).pack()
    out = torch.empty((M, N), dtype=torch.float16, device=p.A_d.device)
    assert _call(wq.lib(), p, out) == WQ_ERR_WORKSPACE
