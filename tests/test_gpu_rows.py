"""A few rows (T = 1 .. 16) through the decode-style path, moe_forward_rows
(section "Limits of further optimization": verification of drafted tokens
processes groups of two to five rows): against the fp64 oracle, which selects
experts from the kernel's own fp32 router logits, and against one decode
launch per row, whose arithmetic it repeats operation for operation."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_layer_close, host_layer, logits_bound, make_ctx
from oracle import moe_oracle as orc
from sparse_moe_gb300 import MoEError

pytestmark = pytest.mark.gpu


def _check_rows(ctx, w, x, int4=False):
    T = x.shape[0]
    y = ctx.forward_rows(0, x)
    r = ctx.rows_routing(T)
    torch.cuda.synchronize()
    lg = r["logits"].cpu().numpy()
    x_np = x.float().cpu().numpy()
    wr = w["router_w"].float().cpu().numpy()
    b = None if w.get("router_b") is None else w["router_b"].cpu().numpy()
    ref_l = orc.router_logits(x_np, wr, b)
    assert np.all(np.abs(lg - ref_l) <= logits_bound(x_np, wr, ref_l, b))
    o = orc.route(lg, ctx.top_k)
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), o["topk_idx"])
    assert np.abs(r["topk_w"].cpu().numpy() - o["topk_w"]).max() <= 4e-6
    ref = orc.moe_layer(x_np, host_layer(w), ctx.top_k, logits=lg)
    assert_layer_close(y.float().cpu().numpy(), ref, int4=int4, what=f"rows T={T}")
    return y


def _decode_each(ctx, x):
    return torch.stack([ctx.forward_decode(0, x[t:t + 1].contiguous()).reshape(-1)
                        for t in range(x.shape[0])])


@pytest.mark.parametrize("T", [1, 2, 5, 16])
def test_rows_tiny(T):
    wl = moe_synth.Workload("r", moe_synth.TINY, T=T, bias_std=1.5, seed=50 + T)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    _check_rows(ctx, w, moe_synth.make_x(wl, device="cuda"))


@pytest.fixture(scope="module")
def rows_qwen():
    wl = moe_synth.Workload("rq", moe_synth.QWEN, T=16, bias_std=1.5, seed=60)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    return wl, ctx, w


@pytest.mark.parametrize("T", [2, 5, 16])
def test_rows_qwen_bf16(rows_qwen, T):
    wl, ctx, w = rows_qwen
    x = moe_synth.make_x(wl, device="cuda")[:T].contiguous()
    _check_rows(ctx, w, x)


def test_rows_equal_one_decode_per_row(rows_qwen):
    # same dot products in the same order as moe_forward_decode, row by row
    wl, ctx, w = rows_qwen
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_rows(0, x)
    yd = _decode_each(ctx, x)
    torch.cuda.synchronize()
    assert torch.equal(y, yd)
    assert ctx.check_device() == 0


def test_rows_shared_expert_rows_repeat():
    # identical rows select identical experts: every union expert has all
    # T rows as users, and each output row equals the one-row result
    wl = moe_synth.Workload("rr", moe_synth.QWEN, T=1, seed=61)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    x1 = moe_synth.make_x(wl, device="cuda")
    x = x1.expand(7, -1).contiguous()
    y = ctx.forward_rows(0, x)
    y1 = ctx.forward_decode(0, x1)
    torch.cuda.synchronize()
    assert torch.equal(y, y1.expand(7, -1))


@pytest.mark.parametrize("wfmt", [moe_synth.WFMT_INT4, moe_synth.WFMT_INT4_AFFINE])
def test_rows_int4(wfmt):
    wl = moe_synth.Workload("r4", moe_synth.QWEN, T=4, bias_std=1.5, wfmt=wfmt, seed=62)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    x = moe_synth.make_x(wl, device="cuda")
    _check_rows(ctx, w, x, int4=True)
    y = ctx.forward_rows(0, x)
    yd = _decode_each(ctx, x)
    torch.cuda.synchronize()
    assert torch.equal(y, yd)


def test_rows_rejects_bad_arguments(rows_qwen):
    wl, ctx, w = rows_qwen
    x = moe_synth.make_x(wl, device="cuda")
    with pytest.raises(MoEError):
        ctx.forward_rows(0, x[:0].contiguous())
    big = torch.cat([x, x[:1]]).contiguous()   # 17 rows
    with pytest.raises(MoEError):
        ctx.forward_rows(0, big)
