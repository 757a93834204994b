"""Edge cases of the layer on the GPU against the fp64 oracle:

* top-1 routing (k = 1: each token's single expert gets weight 1), through
  prefill, decode and the few-rows path;
* the fp16 intermediates of the prefill path (h and o are stored in fp16):
  activations sixteen times larger than unit variance, with part of the
  down-projection weights below 2^-17 (where fp16 keeps fewer than 8
  significant bits), still meet the tolerance; activations large enough to
  push h beyond 65504 are reported as MOE_ERR_RANGE by moe_check_device,
  while the decode path, which keeps h in fp32, still computes them.
"""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_layer_close, check_routing, host_layer, make_ctx
from oracle import moe_oracle as orc
from sparse_moe_gb300 import MoEError, _abi, with_f16_down

pytestmark = pytest.mark.gpu

TOP1 = moe_synth.Shape(hidden=256, n_experts=16, top_k=1, inter=64, shared_inter=64)


def test_top1_prefill_decode_rows():
    wl = moe_synth.Workload("top1", TOP1, T=200, bias_std=1.0, seed=91)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=256)
    x = moe_synth.make_x(wl, device="cuda")
    lg = check_routing(ctx, w, x)
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    hw = host_layer(w)
    ref = orc.moe_layer(x.float().cpu().numpy(), hw, 1, logits=lg)
    assert_layer_close(y.float().cpu().numpy(), ref, what="top-1 prefill")
    r = ctx.route(0, x)
    assert torch.all(r["topk_w"] == 1.0)
    # decode of one row and the few-rows path on three rows
    yd = ctx.forward_decode(0, x[:1].contiguous())
    lgd = ctx.decode_routing()["logits"].cpu().numpy()[None, :]
    refd = orc.moe_layer(x[:1].float().cpu().numpy(), hw, 1, logits=lgd)
    assert_layer_close(yd.float().cpu().numpy(), refd, what="top-1 decode")
    yr = ctx.forward_rows(0, x[:3].contiguous())
    lgr = ctx.rows_routing(3)["logits"].cpu().numpy()
    refr = orc.moe_layer(x[:3].float().cpu().numpy(), hw, 1, logits=lgr)
    assert_layer_close(yr.float().cpu().numpy(), refr, what="top-1 rows")
    assert ctx.check_device() == 0


def _scaled_case(scale, seed, tiny_down=False):
    wl = moe_synth.Workload("range", moe_synth.QWEN, T=256, bias_std=1.5, seed=seed)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=256)
    if tiny_down:
        # a quarter of the routed down-projection rows scaled to about 2^-20
        # (below 2^-17), and the shared expert's by 2^-9
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        rows = torch.rand(w["down"].shape[:2], generator=g, device="cuda") < 0.25
        w["down"][rows] = (w["down"][rows].float() * 2.0 ** -14).to(torch.bfloat16)
        w["sh_down"].mul_(2.0 ** -9)
        ctx.load_weights(0, with_f16_down(w))
    x = (moe_synth.make_x(wl, device="cuda").float() * scale).to(torch.bfloat16)
    return wl, ctx, w, x


def test_prefill_large_activations_and_tiny_weights_within_tolerance():
    wl, ctx, w, x = _scaled_case(16.0, 92, tiny_down=True)
    lg = ctx.route(0, x)["logits"]
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    ref = orc.moe_layer(x.float().cpu().numpy(), host_layer(w), wl.shape.top_k,
                        logits=lg.cpu().numpy())
    assert np.abs(ref).max() > 50.0   # well away from unit scale
    assert_layer_close(y.float().cpu().numpy(), ref, what="x * 16, tiny down weights")
    assert ctx.check_device() == 0


def test_prefill_reports_fp16_overflow_and_decode_does_not_overflow():
    wl, ctx, w, x = _scaled_case(400.0, 93)
    ctx.forward_prefill(0, x)
    with pytest.raises(MoEError) as ei:
        ctx.check_device()
    assert ei.value.status == _abi.MOE_ERR_RANGE
    assert ctx.check_device() == 0     # the status word was cleared
    # the same row through the decode path (h in fp32): finite and close to
    # the oracle
    yd = ctx.forward_decode(0, x[:1].contiguous())
    lgd = ctx.decode_routing()["logits"].cpu().numpy()[None, :]
    torch.cuda.synchronize()
    with np.errstate(over="ignore"):   # exp(-z) of large negative z: silu -> -0, as it should
        ref = orc.moe_layer(x[:1].float().cpu().numpy(), host_layer(w), wl.shape.top_k, logits=lgd)
    assert_layer_close(yd.float().cpu().numpy(), ref, what="decode at x * 400")
    assert ctx.check_device() == 0
