"""GPU routing (router GEMM on tcgen05, top-k, histogram, scan, scatter)
against the oracle: logits within the fp32 summation bound, everything else
bit-exact with the oracle selecting from the GPU's fp32 logits."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import check_routing, make_ctx

pytestmark = pytest.mark.gpu


def _wl(shape, T, bias=None, seed=0):
    return moe_synth.Workload("t", shape, T=T, bias_std=bias, seed=seed)


@pytest.mark.parametrize("T", [1, 16, 17, 33, 1000])
def test_route_tiny_shapes(T):
    wl = _wl(moe_synth.TINY, T, bias=1.0, seed=T)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=1024)
    x = moe_synth.make_x(wl, device="cuda")
    check_routing(ctx, w, x)


def test_route_qwen_8192_row_chunk():
    # one chunk of 8192 rows: 256 routing blocks, twice the default chunk's
    wl = _wl(moe_synth.QWEN, 8192, bias=1.5, seed=81)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=8192)
    x = moe_synth.make_x(wl, device="cuda")
    check_routing(ctx, w, x)


@pytest.mark.parametrize("T", [1, 300, 4096])
def test_route_qwen_shape(T):
    wl = moe_synth.PREFILL_BF16 if T == 4096 else _wl(moe_synth.QWEN, T, bias=1.5, seed=T)
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    lg = check_routing(ctx, w, x)
    if T == 4096:
        # the uneven load the skewing bias is there to produce
        counts = np.bincount(np.argsort(-lg, axis=1, kind="stable")[:, :8].ravel(), minlength=256)
        assert counts.max() > 4 * counts.mean() and (counts == 0).any()


def test_route_ties_prefer_lower_expert():
    wl = _wl(moe_synth.QWEN, 200, seed=3)
    ctx, (w,) = make_ctx(wl)
    w["router_w"][5].copy_(w["router_w"][3])        # experts 3 and 5 always tie
    w["router_w"][200].copy_(w["router_w"][3])
    x = moe_synth.make_x(wl, device="cuda")
    lg = check_routing(ctx, w, x)
    assert np.array_equal(lg[:, 3], lg[:, 5])


def test_route_all_tokens_one_expert():
    wl = _wl(moe_synth.QWEN, 600, seed=4)
    ctx, (w,) = make_ctx(wl)
    b = torch.zeros(256, device="cuda")
    b[7] = 100.0
    w["router_b"] = b
    ctx.load_weights(0, w)
    x = moe_synth.make_x(wl, device="cuda")
    check_routing(ctx, w, x)
    r = ctx.route(0, x)
    assert int(r["counts"][7]) == 600 and bool((r["topk_idx"][:, 0] == 7).all())


def test_route_zero_tokens_is_noop():
    wl = _wl(moe_synth.TINY, 16)
    ctx, _ = make_ctx(wl, max_chunk_rows=64)
    x = torch.empty((0, wl.shape.hidden), dtype=torch.bfloat16, device="cuda")
    r = ctx.route(0, x)
    assert r["topk_idx"].numel() == 0
    assert ctx.check_device() == 0


def test_route_too_many_rows_rejected():
    from sparse_moe_gb300 import MoEError
    wl = _wl(moe_synth.TINY, 16)
    ctx, _ = make_ctx(wl, max_chunk_rows=16)
    x = moe_synth.make_x(wl, device="cuda", T=17)
    with pytest.raises(MoEError):
        ctx.route(0, x)
