"""A few rows (T = 1 .. 16) through the decode-style path, moe_forward_rows
(section "Limits of further optimization": verification of drafted tokens
processes groups of two to five rows): against the fp64 oracle, which selects
experts from the kernel's own fp32 router logits, and against one decode
launch per row.  int4 rows, and bf16 calls of fewer than 5 rows, repeat the
decode's arithmetic operation for operation; bf16 calls of 5 or more rows run
their gate/up dot products on the tensor cores, so they match the decode
within its tolerances.  Each row's result is independent of the values of
the other rows."""
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


def test_rows_match_one_decode_per_row(rows_qwen):
    # bf16: the gate/up dot products on the tensor cores, the rest as in
    # moe_forward_decode: the same layer within the decode's tolerances
    wl, ctx, w = rows_qwen
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_rows(0, x)
    yd = _decode_each(ctx, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), yd.float().cpu().numpy(), what="rows vs decode")
    assert ctx.check_device() == 0


@pytest.mark.parametrize("lo,hi", [(0, 5), (3, 11), (9, 16), (0, 2), (12, 16)])
def test_rows_independent_of_other_rows(rows_qwen, lo, hi):
    # row t's result does not depend on the values of the other rows that
    # share the call, only on their number being below 5 (per-user passes) or
    # not (tensor cores: 8 or fewer rows take one column block, more two)
    wl, ctx, w = rows_qwen
    x = moe_synth.make_x(wl, device="cuda")
    ys = ctx.forward_rows(0, x[lo:hi].contiguous())
    if hi - lo >= 5:
        y = ctx.forward_rows(0, x)
        ref = y[lo:hi]
    else:
        # per-user passes: row for row the decode's arithmetic
        ref = _decode_each(ctx, x[lo:hi].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(ys, ref)


def test_rows_shared_expert_rows_repeat():
    # identical rows select identical experts: every union expert has all
    # T rows as users, and every output row equals the one-row result
    wl = moe_synth.Workload("rr", moe_synth.QWEN, T=1, seed=61)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    x1 = moe_synth.make_x(wl, device="cuda")
    x = x1.expand(7, -1).contiguous()
    y = ctx.forward_rows(0, x)
    y1 = ctx.forward_decode(0, x1)
    torch.cuda.synchronize()
    assert torch.equal(y, y[:1].expand(7, -1))
    assert_layer_close(y[:1].float().cpu().numpy(), y1.float().cpu().numpy(), what="rows vs decode")


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
