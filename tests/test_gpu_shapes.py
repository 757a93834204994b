"""A layer shape away from the Qwen one, through prefill, decode and the
few-rows path, against the fp64 oracle.  It reaches the paths the Qwen and
tiny shapes leave out: top-k above 8 (the combine's and decode's generic
slot loops), an expert count that is not a multiple of 32 (partial mask
words and router tiles), a hidden size whose 9 router k-steps do not split
(the top-k kernel's single-part path) and whose down projection ends in a
partial 256-row tile, and a shared expert wider than the routed ones
(I = 128, Is = 192: a half-used gate/up tile)."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_layer_close, check_routing, host_layer, logits_bound, make_ctx
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

ODD = moe_synth.Shape(hidden=576, n_experts=40, top_k=10, inter=128, shared_inter=192)


def _ctx(wfmt, T, chunk, seed):
    wl = moe_synth.Workload("odd", ODD, T=T, bias_std=1.0, wfmt=wfmt, seed=seed)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=chunk)
    return wl, ctx, w


@pytest.mark.parametrize("wfmt", [moe_synth.WFMT_BF16, moe_synth.WFMT_INT4])
def test_odd_shape_prefill(wfmt):
    wl, ctx, w = _ctx(wfmt, 300, 4096, 70)
    x = moe_synth.make_x(wl, device="cuda")
    lg = check_routing(ctx, w, x)
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    ref = orc.moe_layer(x.float().cpu().numpy(), host_layer(w), ctx.top_k, logits=lg)
    assert_layer_close(y.float().cpu().numpy(), ref, int4=wfmt != moe_synth.WFMT_BF16,
                       what=f"odd shape prefill {wfmt}")
    assert ctx.check_device() == 0


def test_odd_shape_prefill_chunks_equal_one_pass():
    # 300 rows in chunks of 64 (a ragged last chunk of 44): bit for bit the
    # one-pass result
    wl, ctx, w = _ctx(moe_synth.WFMT_BF16, 300, 64, 71)
    _, ctx1, _ = _ctx(moe_synth.WFMT_BF16, 300, 4096, 71)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    y1 = ctx1.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y, y1)


@pytest.mark.parametrize("wfmt", [moe_synth.WFMT_BF16, moe_synth.WFMT_INT4])
def test_odd_shape_decode_and_rows(wfmt):
    int4 = wfmt != moe_synth.WFMT_BF16
    wl, ctx, w = _ctx(wfmt, 3, 16, 72)
    x = moe_synth.make_x(wl, device="cuda")
    x_np = x.float().cpu().numpy()
    wr = w["router_w"].float().cpu().numpy()
    b = None if w.get("router_b") is None else w["router_b"].cpu().numpy()
    # decode, one row at a time
    yd = []
    for t in range(x.shape[0]):
        yd.append(ctx.forward_decode(0, x[t:t + 1].contiguous()).reshape(-1))
        r = ctx.decode_routing()
        torch.cuda.synchronize()
        lg = r["logits"].cpu().numpy()[None, :]
        ref_l = orc.router_logits(x_np[t:t + 1], wr, b)
        assert np.all(np.abs(lg - ref_l) <= logits_bound(x_np[t:t + 1], wr, ref_l, b))
        o = orc.route(lg, ctx.top_k)
        np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), o["topk_idx"][0])
        ref = orc.moe_layer(x_np[t:t + 1], host_layer(w), ctx.top_k, logits=lg)
        assert_layer_close(yd[-1][None].float().cpu().numpy(), ref, int4=int4,
                           what=f"odd shape decode row {t}")
    # the three rows in one launch repeat the decode arithmetic row by row
    y = ctx.forward_rows(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y, torch.stack(yd))
    assert ctx.check_device() == 0


def test_odd_shape_rows_on_tensor_cores():
    # 9 bf16 rows take the tensor-core phases (two column blocks, the second
    # with one row); routed and shared output projections of different widths
    # (I = 128, Is = 192) and 10 slots per row
    wl, ctx, w = _ctx(moe_synth.WFMT_BF16, 9, 16, 73)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_rows(0, x)
    r = ctx.rows_routing(9)
    torch.cuda.synchronize()
    lg = r["logits"].cpu().numpy()
    x_np = x.float().cpu().numpy()
    wr = w["router_w"].float().cpu().numpy()
    b = None if w.get("router_b") is None else w["router_b"].cpu().numpy()
    ref_l = orc.router_logits(x_np, wr, b)
    assert np.all(np.abs(lg - ref_l) <= logits_bound(x_np, wr, ref_l, b))
    o = orc.route(lg, ctx.top_k)
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), o["topk_idx"])
    ref = orc.moe_layer(x_np, host_layer(w), ctx.top_k, logits=lg)
    assert_layer_close(y.float().cpu().numpy(), ref, what="odd shape rows (tensor cores)")
    # the same rows among others: unchanged
    y5 = ctx.forward_rows(0, x[4:9].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(y5, y[4:9])
    assert ctx.check_device() == 0
