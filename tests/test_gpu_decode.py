"""Batch-1 decode GEMV path (bf16 and int4) against the fp64 oracle, which
selects experts from the decode router's own fp32 logits."""
import ctypes

import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_layer_close, host_layer, logits_bound, make_ctx
from oracle import moe_oracle as orc
from sparse_moe_gb300 import MoEError, _abi

pytestmark = pytest.mark.gpu


def _check_decode(ctx, w, x, layer=0, int4=False):
    y = ctx.forward_decode(layer, x)
    r = ctx.decode_routing()
    torch.cuda.synchronize()
    lg = r["logits"].cpu().numpy()[None, :]
    x_np = x.float().cpu().numpy()
    wr = w["router_w"].float().cpu().numpy()
    b = None if w.get("router_b") is None else w["router_b"].cpu().numpy()
    ref_l = orc.router_logits(x_np, wr, b)
    assert np.all(np.abs(lg - ref_l) <= logits_bound(x_np, wr, ref_l, b))
    o = orc.route(lg, ctx.top_k)
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), o["topk_idx"][0])
    assert np.abs(r["topk_w"].cpu().numpy() - o["topk_w"][0]).max() <= 4e-6
    ref = orc.moe_layer(x_np, host_layer(w), ctx.top_k, logits=lg)
    return y, assert_layer_close(y.float().cpu().numpy(), ref, int4=int4, what="decode")


def test_decode_tiny():
    wl = moe_synth.Workload("d", moe_synth.TINY, T=1, seed=11)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    _check_decode(ctx, w, moe_synth.make_x(wl, device="cuda"))


@pytest.fixture(scope="module")
def decode_bf16():
    wl = moe_synth.DECODE_BF16
    ctx, layers = make_ctx(wl, n_layers=2, max_chunk_rows=16, seed_layers=[0, 39])
    return wl, ctx, layers


@pytest.mark.parametrize("slot,src", [(0, 0), (1, 39)])
def test_decode_qwen_bf16(decode_bf16, slot, src):
    wl, ctx, layers = decode_bf16
    x = moe_synth.make_x(wl, layer=src, device="cuda")
    _check_decode(ctx, layers[slot], x, layer=slot)


def test_decode_deterministic_and_graph_replay(decode_bf16):
    wl, ctx, layers = decode_bf16
    xs = [moe_synth.make_x(wl, layer=l, device="cuda") for l in (0, 39)]
    ys = [torch.empty_like(x) for x in xs]
    for i in range(2):
        ctx.forward_decode(i, xs[i], ys[i])
    eager = [y.clone() for y in ys]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(2):
                ctx.forward_decode(i, xs[i], ys[i], stream=s)
    for y in ys:
        y.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, ys):
        assert torch.equal(a, b)


def test_decode_matches_prefill_one_token(decode_bf16):
    wl, ctx, layers = decode_bf16
    x = moe_synth.make_x(wl, layer=0, device="cuda")
    yd = ctx.forward_decode(0, x)
    yp = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    ref = yp.double().cpu().numpy()
    err = np.abs(yd.double().cpu().numpy() - ref).max()
    assert err <= 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("pinned_out", [True, False])
def test_decode_host_buffers_match_device_path(decode_bf16, pinned_out):
    # a page-locked output is written by the kernel directly, a pageable one
    # through the staging buffer and a copy
    wl, ctx, layers = decode_bf16
    x = moe_synth.make_x(wl, layer=0, device="cuda")
    yd = ctx.forward_decode(0, x)
    x_h = x.cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory() if pinned_out else torch.empty_like(x_h)
    ctx.forward_decode_host(0, x_h, y_h)
    torch.cuda.synchronize()
    assert torch.equal(y_h, yd.cpu())


def test_decode_int4_qwen():
    wl = moe_synth.DECODE_INT4
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    x = moe_synth.make_x(wl, device="cuda")
    _check_decode(ctx, w, x, int4=True)


def test_decode_int4_tiny():
    wl = moe_synth.Workload("d4", moe_synth.TINY, T=1, wfmt=moe_synth.WFMT_INT4, seed=12)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    _check_decode(ctx, w, moe_synth.make_x(wl, device="cuda"), int4=True)


def test_decode_int4_affine_qwen():
    wl = moe_synth.DECODE_INT4_AFFINE
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    x = moe_synth.make_x(wl, device="cuda")
    _check_decode(ctx, w, x, int4=True)


def test_decode_int4_affine_tiny():
    wl = moe_synth.Workload("d4a", moe_synth.TINY, T=1, wfmt=moe_synth.WFMT_INT4_AFFINE, seed=14)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    _check_decode(ctx, w, moe_synth.make_x(wl, device="cuda"), int4=True)


def test_decode_int4_affine_matches_prefill_one_token():
    wl = moe_synth.Workload("d4a1", moe_synth.QWEN, T=1, wfmt=moe_synth.WFMT_INT4_AFFINE, seed=15)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    x = moe_synth.make_x(wl, device="cuda")
    yd = ctx.forward_decode(0, x)
    yp = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    err = (yd.float() - yp.float()).abs().max().item()
    assert err <= 2e-2 * yp.float().abs().max().item()


# ---- several layers in one persistent launch: the same arithmetic as one
# launch per layer, so the outputs must match bit for bit, with independent
# inputs and with each layer's output feeding the next layer.

def _layers_ctx(wl, n):
    return make_ctx(wl, n_layers=n, max_chunk_rows=16, seed_layers=list(range(n)))


@pytest.mark.parametrize("wl", [moe_synth.DECODE_BF16, moe_synth.DECODE_INT4],
                         ids=["bf16", "int4"])
def test_decode_layers_independent_inputs_match_single_launches(wl):
    n = 3
    ctx, _ = _layers_ctx(wl, n)
    xs = torch.cat([moe_synth.make_x(wl, layer=l, device="cuda") for l in range(n)])
    ref = torch.stack([ctx.forward_decode(l, xs[l:l + 1])[0] for l in range(n)])
    y = torch.empty_like(xs)
    ctx.forward_decode_layers(0, xs, y)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert ctx.check_device() == 0


def test_decode_layers_chained_match_single_launches(decode_bf16):
    wl, ctx, layers = decode_bf16
    x0 = moe_synth.make_x(wl, layer=5, device="cuda")
    ref, x = [], x0
    for l in range(2):
        x = ctx.forward_decode(l, x)
        ref.append(x[0].clone())
    y = torch.empty((2, wl.shape.hidden), dtype=torch.bfloat16, device="cuda")
    ctx.forward_decode_layers(0, x0, y, chained=True)
    torch.cuda.synchronize()
    assert torch.equal(y, torch.stack(ref))
    # the last layer's routing is the one reported
    r = ctx.decode_routing()
    lg = r["logits"].cpu().numpy()[None, :]
    o = orc.route(lg, ctx.top_k)
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), o["topk_idx"][0])


def test_decode_layers_more_than_one_launch_and_oracle():
    """50 tiny layers (two launches of at most 48), chained; the first layer's
    output (equal to the multi-layer one) is also checked against the oracle.
    (Chained through 50 random layers the signal fades towards zero, so the
    relative error of a late layer is not a meaningful check.)"""
    wl = moe_synth.Workload("dl", moe_synth.TINY, T=1, seed=13)
    n = 50
    ctx, layers = _layers_ctx(wl, n)
    x0 = moe_synth.make_x(wl, device="cuda")
    ref, x = [], x0
    for l in range(n):
        x = ctx.forward_decode(l, x)
        ref.append(x[0].clone())
    y = torch.empty((n, wl.shape.hidden), dtype=torch.bfloat16, device="cuda")
    ctx.forward_decode_layers(0, x0, y, chained=True)
    torch.cuda.synchronize()
    assert torch.equal(y, torch.stack(ref))
    y0, _ = _check_decode(ctx, layers[0], x0, layer=0)
    assert torch.equal(y0[0], y[0])


def test_decode_layers_rejects_bad_arguments(decode_bf16):
    wl, ctx, _ = decode_bf16
    H = wl.shape.hidden
    x = torch.zeros((3, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(MoEError):
        ctx.forward_decode_layers(0, x, y)          # slots 0..2 of a 2-slot context
    lib = ctx.lib
    st = lib.moe_forward_decode_layers(ctx.handle, 0, 2, ctypes.c_void_p(x.data_ptr()), 3,
                                       ctypes.c_void_p(y.data_ptr()), H, None)
    assert st == _abi.MOE_ERR_INVALID_ARG             # stride not a multiple of 8
    assert lib.moe_forward_decode_layers(ctx.handle, 0, 0, None, 0, None, 0, None) == _abi.MOE_OK


def test_decode_phase_stamps(decode_bf16):
    # profiling on: every CTA stamps phase B; the output is unchanged by it
    wl, ctx, layers = decode_bf16
    x = moe_synth.make_x(wl, layer=0, device="cuda")
    y0 = ctx.forward_decode(0, x)
    ctx.profile(True)
    with pytest.raises(MoEError):   # nothing stamped since profiling was enabled
        ctx.decode_phase_read()
    y1 = ctx.forward_decode(0, x)
    ph = ctx.decode_phase_read()
    ctx.profile_read()
    ctx.profile(False)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert 0.0 < ph["median_us"] <= ph["window_us"] < 1e4
    assert ctx.check_device() == 0
