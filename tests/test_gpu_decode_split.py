"""GPU parity of the decode kernels' split-K exchange against the float64 oracle.

The S K slices of a 128-row weight tile are the CTAs of one cluster; CTA q owns rows
[128 q / S, 128 (q + 1) / S) of the tile and adds the S slices' partial sums of them in
rank order.  With a split into blocks of ceil(128 / S) rows, 14 slices would leave the
last CTA no rows (13 x 10 > 128) and a negative byte count on its inbox barrier; these
tests take every cluster size from 2 to 16, the 14-way split at the decode shapes'
token counts, and check every output element, the device status word and run-to-run bits.
"""
import pytest
import torch

import weight_only_quantized_tma_gb300 as wq

from gpu_helpers import Fp8Problem, Int4Problem, check_close, out_to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 16])
def test_w4a16_decode_fourteen_way_split(M):
    # two weight tiles, 28 k-blocks of 256: 14 slices of a tile, 9 or 10 rows per owner
    N, K = 256, 7168
    plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, M, N, K, 128)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["splits"] == 14
    wq.wq_clear_device_status()
    p = Int4Problem(M, N, K, 128, seed=540 + M).pack()
    out = p.run()
    torch.cuda.synchronize()
    assert wq.wq_device_status() == 0
    check_close(out_to_f64(out), p.ref(), what=f"14-way split M={M}")
    for _ in range(3):
        assert torch.equal(p.run(), out)


@pytest.mark.parametrize("M", [1, 16, 25, 32])
def test_fp8_decode_fourteen_way_split(M):
    # FP8 stages hold 128 values: two weight tiles and 28 k-blocks; 25 and 32 tokens
    # send 4 token tiles of partial sums per owned row
    N, K = 256, 3584
    plan = wq.get_plan(wq.WQ_OP_FP8, wq.WQ_BF16, M, N, K, 0)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE
    if plan["splits"] != 14:
        assert M > 16
        pytest.skip(f"the plan takes {plan['splits']} slices for M = {M}")
    wq.wq_clear_device_status()
    p = Fp8Problem(M, N, K, seed=550 + M, with_bias=True)
    out = p.run()
    torch.cuda.synchronize()
    assert wq.wq_device_status() == 0
    check_close(out_to_f64(out), p.ref(), out_dtype="bf16", what=f"fp8 14-way split M={M}")


@pytest.mark.parametrize("S", list(range(2, 17)))
def test_decode_every_cluster_size(S):
    # one weight tile and 2 S + 1 k-blocks of 128 (K % 256 == 64): the plan takes S
    # slices, and every slice count from 2 to 16 shares the tile's 128 rows
    N, K = 128, (2 * S + 1) * 128 - 64
    plan = wq.get_plan(wq.WQ_OP_W4A16, wq.WQ_F16, 3, N, K, 32)
    assert plan["kernel"] == wq.WQ_KERNEL_DECODE and plan["bk"] == 128
    if plan["splits"] != S:
        pytest.skip(f"the plan takes {plan['splits']} slices for K = {K}")
    wq.wq_clear_device_status()
    p = Int4Problem(3, N, K, 32, seed=560 + S).pack()
    out = p.run()
    torch.cuda.synchronize()
    assert wq.wq_device_status() == 0
    check_close(out_to_f64(out), p.ref(), what=f"S={S}")
