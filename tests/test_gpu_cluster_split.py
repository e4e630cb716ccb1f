"""Split-K reduced inside thread-block clusters (the tile kernel's default for S <= 16
slices) against the workspace reduction (WQ_SPLITK_WORKSPACE=1): both add the fp32
partial sums of the slices in slice order 0..S-1 starting from zero, so the outputs
must agree bit for bit; and against the oracle for a few shapes."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_tma_gb300 as wq
from weight_only_quantized_tma_gb300 import synth

from gpu_helpers import DEV, Int4Problem, check_close, out_to_f64, to_dev_f16bits

pytestmark = pytest.mark.gpu


def _int4(M, N, K, G, seed):
    p = Int4Problem(M, N, K, G, seed=seed).pack()
    return (wq.WQ_OP_W4A16, wq.WQ_F16, G), (lambda: p.run()), p.ref


def _fp8(M, N, K, seed, bias=False):
    A = synth.activations(M, K, "bf16", seed)
    w8 = synth.fp8_weights(N, K, seed + 1)
    A_d = to_dev_f16bits(A, "bf16")
    wd = torch.from_numpy(w8.w).to(DEV)
    alpha = torch.tensor([w8.scale], dtype=torch.float32, device=DEV)
    bb = synth.bias(N, "bf16", seed + 2) if bias else None
    b_d = to_dev_f16bits(bb, "bf16") if bias else None
    ref = lambda: oracle.gemm_w8a16_fp8(A, True, w8.w, float(w8.scale), M, N, K, bias_bits=bb)
    return (wq.WQ_OP_FP8, wq.WQ_BF16, 0), (lambda: wq.wq_gemm_w8a16_fp8(A_d, wd, alpha, bias=b_d)), ref


def _fp4(M, N, K, seed):
    A = synth.activations(M, K, "bf16", seed)
    w4 = synth.fp4_weights(N, K, seed + 1)
    A_d = to_dev_f16bits(A, "bf16")
    wd = torch.from_numpy(w4.w).to(DEV)
    sfk = wq.wq_pack_fp4_sf(torch.from_numpy(w4.sf).to(DEV), N, K)
    alpha = torch.tensor([w4.alpha], dtype=torch.float32, device=DEV)
    ref = lambda: oracle.gemm_bf16_fp4(A, w4.w, w4.sf, float(w4.alpha), M, N, K)
    return (wq.WQ_OP_FP4, wq.WQ_BF16, 0), (lambda: wq.wq_gemm_bf16_fp4(A_d, wd, sfk, alpha)), ref


def _lut(M, N, K, G, seed):
    A = synth.activations(M, K, "f16", seed)
    wts = synth.int4_weights(N, K, G, seed + 1)
    lut = synth.normal_quantile_codebook()
    A_d = to_dev_f16bits(A, "f16")
    wk, sk = wq.wq_pack_int4(torch.from_numpy(wts.w).to(DEV), to_dev_f16bits(wts.s, "f16"), N, K, G)
    lut_d = to_dev_f16bits(lut, "f16")
    ref = lambda: oracle.gemm_w4a16_lut(A, False, wts.w, wts.s, lut, M, N, K, G)
    return (wq.WQ_OP_W4A16_LUT, wq.WQ_F16, G), (lambda: wq.wq_gemm_w4a16_lut(A_d, wk, sk, lut_d, N, K, G)), ref


def _int2(M, N, K, G, seed):
    A = synth.activations(M, K, "f16", seed)
    w2 = synth.int2_weights(N, K, G, seed + 1)
    A_d = to_dev_f16bits(A, "f16")
    wd = torch.from_numpy(w2.w).to(DEV)
    sk = wq.wq_pack_int2_scales(to_dev_f16bits(w2.s, "f16"), N, K, G)
    ref = lambda: oracle.gemm_w2a16(A, False, w2.w, w2.s, M, N, K, G)
    return (wq.WQ_OP_W2A16, wq.WQ_F16, G), (lambda: wq.wq_gemm_w2a16(A_d, wd, sk, N, K, G)), ref


CASES = {
    "int4_M20": lambda: _int4(20, 1024, 2048, 128, 801),
    "int4_M32": lambda: _int4(32, 4096, 1024, 128, 802),
    "int4_M128": lambda: _int4(128, 4096, 4096, 128, 803),
    "int4_M300_N520": lambda: _int4(300, 520, 4096, 64, 804),
    "fp8_M1": lambda: _fp8(1, 10240, 5120, 805),
    "fp8_M16_bias": lambda: _fp8(16, 10240, 5120, 806, bias=True),
    "fp8_M64": lambda: _fp8(64, 10240, 5120, 807),
    "fp4_M1": lambda: _fp4(1, 12800, 5120, 808),
    "fp4_M128": lambda: _fp4(128, 6656, 19968, 809),
    "lut_M16": lambda: _lut(16, 4096, 4096, 128, 810),
    "int2_M7": lambda: _int2(7, 4096, 4096, 32, 811),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_cluster_and_workspace_split_vs_oracle(name, monkeypatch):
    # the default plan (cluster split-K for token tiles >= 64 when the clusters fit in
    # one wave) and the workspace reduction both match the oracle; with the same slice
    # count they add the same partial sums in the same order, so the bits agree.  FP8
    # at M <= 16 runs on the tile kernel here (WQ_DISABLE_DECODE=1), not the decode one
    monkeypatch.setenv("WQ_DISABLE_DECODE", "1")
    (op, adt, G), run, ref = CASES[name]()
    shape = run_shape(name)
    want = ref()
    kind = "bf16" if adt == wq.WQ_BF16 else "f16"
    outs, plans = [], []
    for mode in ("default", "workspace"):
        if mode == "workspace":
            monkeypatch.setenv("WQ_SPLITK_WORKSPACE", "1")
        plan = wq.get_plan(op, adt, *shape, G)
        assert plan["splits"] > 1 and plan["kernel"] == wq.WQ_KERNEL_TILE
        if mode == "workspace":
            assert plan["cluster_split"] == 0 and plan["ws_bytes"] > 0
        if plan["cluster_split"]:
            assert plan["ws_bytes"] == 0 and plan["bn"] >= 64
            assert plan["grid"] == plan["tiles_n"] * plan["tiles_m"] * plan["splits"]
            assert plan["tiles_n"] * plan["tiles_m"] <= plan["cluster_capacity"]
        got = run()
        torch.cuda.synchronize()
        check_close(out_to_f64(got), want, out_dtype=kind, what=f"{name} {mode}")
        outs.append(got)
        plans.append(plan)
    if name in ("int4_M32", "int4_M128"):
        assert plans[0]["cluster_split"] == 1
    if plans[0]["splits"] == plans[1]["splits"]:
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), name


@pytest.mark.parametrize("name", ["int4_M300_N520", "fp8_M1", "fp4_M128", "int2_M7", "lut_M16"])
def test_forced_cluster_split_vs_oracle(name, monkeypatch):
    # WQ_SPLITK_CLUSTER=1: the cluster reduction at any token tile (16 and 256 too)
    # whenever the clusters fit in one wave; checked against the oracle (tile kernel
    # for FP8 at M <= 16 too)
    monkeypatch.setenv("WQ_SPLITK_CLUSTER", "1")
    monkeypatch.setenv("WQ_DISABLE_DECODE", "1")
    (op, adt, G), run, ref = CASES[name]()
    plan = wq.get_plan(op, adt, *run_shape(name), G)
    if plan["cluster_split"]:
        assert plan["ws_bytes"] == 0
        assert plan["tiles_n"] * plan["tiles_m"] <= plan["cluster_capacity"]
    got = run()
    torch.cuda.synchronize()
    check_close(out_to_f64(got), ref(), out_dtype="bf16" if adt == wq.WQ_BF16 else "f16", what=f"{name} forced")


def run_shape(name):
    return {"int4_M20": (20, 1024, 2048), "int4_M32": (32, 4096, 1024), "int4_M128": (128, 4096, 4096),
            "int4_M300_N520": (300, 520, 4096), "fp8_M1": (1, 10240, 5120), "fp8_M16_bias": (16, 10240, 5120),
            "fp8_M64": (64, 10240, 5120), "fp4_M1": (1, 12800, 5120), "fp4_M128": (128, 6656, 19968),
            "lut_M16": (16, 4096, 4096), "int2_M7": (7, 4096, 4096)}[name]


def test_cluster_split_repeatable():
    # the same call twice: identical bits (no state carried between calls)
    (_, _, _), run, _ = _int4(64, 2048, 4096, 128, 812)
    a = run()
    b = run()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
