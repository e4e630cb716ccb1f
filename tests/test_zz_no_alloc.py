"""wq_gemm_w4a16_noalloc: the W4A16 GEMM for callers that cannot allocate device memory.

A framework that owns all device memory through its own pool, or a decode loop in
which cudaMalloc (and the device synchronisation it may cause) is not allowed, cannot
hand the GEMM a split-K workspace.  This entry point uses a fixed scratch array built
into the library instead.  The test calls it through the C ABI twice in a row and
checks each result against the workspace entry point, with the tolerance the other
tests use.  The file is named to be collected last, and it works in a fresh process
as well as after the other tests.
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
    return L.wq_gemm_w4a16_noalloc(ctypes.c_void_p(p.A_d.data_ptr()), 0, ctypes.c_void_p(p.wk.data_ptr()),
                                   ctypes.c_void_p(p.sk.data_ptr()), p.M, p.N, p.K, p.G,
                                   ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("M,N,K,scratch", [(32, 4096, 1024, True), (20, 1024, 2048, True), (32, 4096, 1024, False),
                                           (1, 11008, 4096, False), (16, 4096, 4096, False)])
def test_noalloc_matches_workspace_entry_on_two_calls(M, N, K, scratch, monkeypatch):
    G = 128
    if scratch:
        # tile-kernel split-K with the workspace reduction (the tile kernel otherwise
        # reduces its slices inside a cluster): the built-in scratch is really exercised
        monkeypatch.setenv("WQ_SPLITK_WORKSPACE", "1")
    plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, G)
    if scratch:
        assert plan["splits"] > 1 and 0 < plan["ws_bytes"] <= _lib.WQ_NOALLOC_SCRATCH_BYTES
        assert plan["cluster_split"] == 0
    else:
        # the decode kernel and the tile kernel's cluster split-K need no scratch
        assert plan["ws_bytes"] == 0
    p = Int4Problem(M, N, K, G, seed=901 + M).pack()
    expected = p.run()                       # the entry point with a caller workspace
    torch.cuda.synchronize()
    L = wq.lib()
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=p.A_d.device)
        assert _call(L, p, out) == 0
        torch.cuda.synchronize()
        check_close(out_to_f64(out), out_to_f64(expected), what="noalloc vs workspace entry")
        check_close(out_to_f64(out), p.ref(), what="noalloc vs oracle")


def test_noalloc_rejects_problems_beyond_its_scratch(monkeypatch):
    monkeypatch.setenv("WQ_SPLITK_WORKSPACE", "1")
    M, N, K, G = 256, 2048, 4096, 128
    plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, G)
    assert plan["ws_bytes"] > _lib.WQ_NOALLOC_SCRATCH_BYTES
    p = Int4Problem(M, N, K, G, seed=950).pack()
    out = torch.empty((M, N), dtype=torch.float16, device=p.A_d.device)
    assert _call(wq.lib(), p, out) == WQ_ERR_WORKSPACE
