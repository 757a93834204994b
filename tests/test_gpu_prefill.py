"""GPU prefill path (router, routing, tcgen05 grouped gate/up+SwiGLU and down
GEMMs, combine) against the fp64 oracle, which selects experts from the
GPU's fp32 router logits."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_layer_close, check_routing, host_layer, make_ctx
from oracle import moe_oracle as orc
from sparse_moe_gb300 import MoEContext, MoEError, convert_bf16_to_f16, dequant_int4, with_f16_down

pytestmark = pytest.mark.gpu


def _wl(shape, T, bias=None, seed=0):
    return moe_synth.Workload("t", shape, T=T, bias_std=bias, seed=seed)


def _oracle_y(ctx, w, x, tokens=None):
    lg = ctx.route(0, x)["logits"].cpu().numpy()
    return orc.moe_layer(x.float().cpu().numpy(), host_layer(w), ctx.top_k, logits=lg,
                         tokens=tokens)


def test_prefill_tiny_full():
    wl = moe_synth.TINY_LAYER
    ctx, (w,) = make_ctx(wl, max_chunk_rows=64)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), _oracle_y(ctx, w, x), what="tiny T=16")


@pytest.mark.parametrize("T", [1, 17, 1000])
def test_prefill_tiny_shapes_many_tiles(T):
    # E=16, k=2: at T=1000 each expert gets ~125 rows on average and the
    # biased ones several 256-row blocks; T=17 leaves a ragged tail.
    wl = _wl(moe_synth.TINY, T, bias=1.5, seed=T + 1)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=1024)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), _oracle_y(ctx, w, x), what=f"tiny T={T}")


def test_prefill_qwen_ragged_full():
    wl = _wl(moe_synth.QWEN, 300, bias=1.5, seed=7)
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), _oracle_y(ctx, w, x), what="qwen T=300")


@pytest.fixture(scope="module")
def prefill_4096():
    wl = moe_synth.PREFILL_BF16
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    return ctx, w, x, y


def test_prefill_4096_sampled_tokens(prefill_4096):
    """The benchmarked workload at full size: routing checked in full, the layer
    output on sampled tokens (first, last and 62 random ones)."""
    ctx, w, x, y = prefill_4096
    check_routing(ctx, w, x)
    rng = np.random.default_rng(0)
    tokens = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 62, replace=False)]))
    ref = _oracle_y(ctx, w, x, tokens=tokens)
    assert_layer_close(y[tokens].float().cpu().numpy(), ref, what="qwen T=4096 sampled")


def test_prefill_4096_deterministic(prefill_4096):
    ctx, w, x, y = prefill_4096
    y2 = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    assert ctx.check_device() == 0


def test_prefill_chunking_does_not_change_output():
    """T=8192 run as two 4096-row chunks equals one 8192-row chunk, bit for
    bit (section 'Bound temporary memory with prompt chunking')."""
    wl = _wl(moe_synth.QWEN, 8192, bias=1.5, seed=8192)
    ctx4, (w,) = make_ctx(wl, max_chunk_rows=4096)
    ctx8 = make_ctx(wl, max_chunk_rows=8192)[0]
    ctx8.load_weights(0, w)
    x = moe_synth.make_x(wl, device="cuda")
    y4 = ctx4.forward_prefill(0, x)
    y8 = ctx8.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y4, y8)
    tokens = np.array([0, 4095, 4096, 8191])
    lg = torch.cat([ctx4.route(0, x[:4096])["logits"], ctx4.route(0, x[4096:])["logits"]])
    ref = orc.moe_layer(x.float().cpu().numpy(), host_layer(w), 8, logits=lg.cpu().numpy(),
                        tokens=tokens)
    assert_layer_close(y4[tokens].float().cpu().numpy(), ref, what="chunked")


def test_prefill_all_tokens_one_expert():
    wl = _wl(moe_synth.QWEN, 600, seed=5)
    ctx, (w,) = make_ctx(wl)
    b = torch.zeros(256, device="cuda")
    b[7] = 100.0
    w["router_b"] = b
    ctx.load_weights(0, w)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    tokens = np.arange(0, 600, 7)
    assert_layer_close(y[tokens].float().cpu().numpy(), _oracle_y(ctx, w, x, tokens=tokens),
                       what="one hot expert")


def test_prefill_zero_tokens_is_noop():
    wl = moe_synth.TINY_LAYER
    ctx, _ = make_ctx(wl, max_chunk_rows=64)
    x = torch.empty((0, wl.shape.hidden), dtype=torch.bfloat16, device="cuda")
    y = ctx.forward_prefill(0, x)
    assert y.numel() == 0 and ctx.launch_count == 0


def test_prefill_host_buffers_match_device_path():
    wl = _wl(moe_synth.QWEN, 640, bias=1.5, seed=9)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=256)      # three chunks through the staging path
    x = moe_synth.make_x(wl, device="cuda")
    y_dev = ctx.forward_prefill(0, x)
    x_h = x.cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    ctx.forward_prefill_host(0, x_h, y_h)
    torch.cuda.synchronize()
    assert torch.equal(y_h, y_dev.cpu())


@pytest.mark.parametrize("pinned_out", [True, False])
def test_prefill_host_back_to_back_calls_match_device_path(pinned_out):
    # consecutive calls without a synchronisation in between: their copies
    # run on the context's copy streams through alternating staging slots,
    # overlapping each other's compute; a decode from host buffers in between.
    # Page-locked outputs are written by the combine kernel directly, pageable
    # ones through the staging slots and an output copy.
    wl = _wl(moe_synth.QWEN, 300, bias=1.5, seed=10)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=256)      # two chunks per call
    base = moe_synth.make_x(wl, device="cuda")
    xs = [base, torch.flip(base, dims=[0]).contiguous(), (base.float() * 0.5).to(torch.bfloat16)]
    ys_dev = [ctx.forward_prefill(0, x) for x in xs]
    yd_dev = ctx.forward_decode(0, base[:1].contiguous())
    torch.cuda.synchronize()
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [torch.empty_like(x).pin_memory() if pinned_out else torch.empty_like(x) for x in xh]
    xdh = base[:1].cpu().pin_memory()
    ydh = torch.empty_like(xdh).pin_memory()
    for i in range(3):
        ctx.forward_prefill_host(0, xh[i], yh[i])
        if i == 1:
            ctx.forward_decode_host(0, xdh, ydh)
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(yh[i], ys_dev[i].cpu())
    assert torch.equal(ydh, yd_dev.cpu())


# ---- optional fp16 copies of the down weights: the down GEMM then feeds its
# weight tiles straight to the tensor cores instead of converting them in
# shared memory; the conversion is the same, so the output must not change.

@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 1000, (1 << 20) + 5])
def test_convert_bf16_to_f16_matches_torch(n):
    g = torch.Generator(device="cuda").manual_seed(n)
    src = (torch.randn(n, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    if n >= 9:
        # specials: +-inf, NaN, beyond the fp16 range, fp16 subnormals and below
        src[:9] = torch.tensor([float("inf"), -float("inf"), float("nan"), 7.0e4, -1.0e5,
                                6.0e-6, -3.0e-8, 1.0e-9, 65504.0], device="cuda").to(torch.bfloat16)
    got = convert_bf16_to_f16(src)
    ref = src.to(torch.float16)
    torch.cuda.synchronize()
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(got[~nan].view(torch.int16), ref[~nan].view(torch.int16))


@pytest.mark.parametrize("wl", [moe_synth.TINY_LAYER, _wl(moe_synth.QWEN, 300, bias=1.5, seed=7),
                                moe_synth.PREFILL_BF16], ids=["tiny", "qwen300", "qwen4096"])
def test_prefill_f16_down_copies_bit_identical(wl):
    ctx, (w,) = make_ctx(wl, max_chunk_rows=max(64, wl.T))
    x = moe_synth.make_x(wl, device="cuda")
    y_conv = ctx.forward_prefill(0, x)
    ctx.load_weights(0, with_f16_down(w))
    y_f16 = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y_conv, y_f16)
    assert ctx.check_device() == 0


def test_load_weights_rejects_lone_f16_down_copy():
    wl = moe_synth.TINY_LAYER
    ctx, (w,) = make_ctx(wl, max_chunk_rows=64)
    w2 = dict(w)
    w2["down_f16"] = convert_bf16_to_f16(w["down"])
    with pytest.raises(MoEError):
        ctx.load_weights(0, w2)


# ---- int4 weights (symmetric, group 64): dequantised inside the GEMMs; the
# oracle applies the same dequant definition in fp64.

def _wl4(shape, T, bias=None, seed=0):
    return moe_synth.Workload("t4", shape, T=T, bias_std=bias, seed=seed, wfmt=moe_synth.WFMT_INT4)


@pytest.mark.parametrize("T", [1, 16, 1000])
def test_prefill_int4_tiny(T):
    wl = _wl4(moe_synth.TINY, T, bias=1.5 if T > 16 else None, seed=40 + T)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=1024)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), _oracle_y(ctx, w, x), int4=True,
                       what=f"tiny int4 T={T}")


def test_prefill_int4_qwen_ragged_full():
    wl = _wl4(moe_synth.QWEN, 300, bias=1.5, seed=9)
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), _oracle_y(ctx, w, x), int4=True,
                       what="qwen int4 T=300")


def test_prefill_int4_4096_sampled_tokens():
    """The int4 prefill workload at full size: routing in full, the layer on
    sampled tokens."""
    wl = moe_synth.PREFILL_INT4
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    check_routing(ctx, w, x)
    rng = np.random.default_rng(1)
    tokens = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 30, replace=False)]))
    ref = _oracle_y(ctx, w, x, tokens=tokens)
    assert_layer_close(y[tokens].float().cpu().numpy(), ref, int4=True,
                       what="qwen int4 T=4096 sampled")
    y2 = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


# ---- affine int4 (the checkpoint format: a scale and a bias per 64 along K,
# unsigned codes): dequantised inside the GEMMs with one fused multiply-add
# per weight; the oracle applies w = scale * code + bias in fp64.

def _wl4a(shape, T, bias=None, seed=0):
    return moe_synth.Workload("t4a", shape, T=T, bias_std=bias, seed=seed,
                              wfmt=moe_synth.WFMT_INT4_AFFINE)


@pytest.mark.parametrize("T", [1, 16, 1000])
def test_prefill_int4_affine_tiny(T):
    wl = _wl4a(moe_synth.TINY, T, bias=1.5 if T > 16 else None, seed=60 + T)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=1024)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), _oracle_y(ctx, w, x), int4=True,
                       what=f"tiny int4 affine T={T}")


def test_prefill_int4_affine_qwen_ragged_full():
    wl = _wl4a(moe_synth.QWEN, 300, bias=1.5, seed=19)
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert_layer_close(y.float().cpu().numpy(), _oracle_y(ctx, w, x), int4=True,
                       what="qwen int4 affine T=300")


def test_prefill_int4_affine_4096_sampled_tokens():
    wl = moe_synth.PREFILL_INT4_AFFINE
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    check_routing(ctx, w, x)
    rng = np.random.default_rng(3)
    tokens = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 30, replace=False)]))
    ref = _oracle_y(ctx, w, x, tokens=tokens)
    assert_layer_close(y[tokens].float().cpu().numpy(), ref, int4=True,
                       what="qwen int4 affine T=4096 sampled")


def test_load_weights_affine_needs_biases():
    wl = _wl4a(moe_synth.TINY, 4, seed=5)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    w2 = dict(w)
    w2["down_bias"] = None
    with pytest.raises(MoEError):
        ctx.load_weights(0, w2)


# ---- stand-alone dequantisation (the page's "separate dequantization"
# ablation): rounded exactly as the fused expansion, so a bf16 layer on the
# expanded weights equals the int4 layer bit for bit.

@pytest.mark.parametrize("wfmt", [moe_synth.WFMT_INT4, moe_synth.WFMT_INT4_AFFINE])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float16])
def test_dequant_int4_rounds_once(wfmt, out):
    wl = moe_synth.Workload("dq", moe_synth.TINY, T=1, wfmt=wfmt, seed=31)
    w = moe_synth.make_layer(wl, device="cuda")
    got = dequant_int4(w["down"], w["down_scale"], w.get("down_bias"), out_dtype=out)
    torch.cuda.synchronize()
    L = moe_synth.to_numpy(w)
    if out == torch.float16:
        # fp16 operands: the bf16 scale and bias become fp16 values first
        # (exact unless below fp16's normal range, where they round)
        for name in ("down_scale", "down_bias"):
            if name in w and w[name] is not None:
                L[name] = w[name].cpu().half().double().numpy()
    exact = (orc.dequant_int4_affine_g64(L["down"], L["down_scale"], L["down_bias"])
             if wfmt == moe_synth.WFMT_INT4_AFFINE else
             orc.dequant_int4_sym_g64(L["down"], L["down_scale"]))
    g = got.double().cpu().numpy()
    # then correctly rounded: within half a unit in the last place of the format
    mant = 8 if out == torch.bfloat16 else 11
    e = np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -120)))
    half_ulp = 2.0 ** (e - mant)
    if out == torch.float16:
        half_ulp = np.maximum(half_ulp, 2.0 ** -25)   # fp16 subnormal spacing / 2
    assert np.all(np.abs(g - exact) <= half_ulp)
    if wfmt == moe_synth.WFMT_INT4:   # q * s is exact in fp32: one rounding in torch too
        ref = torch.from_numpy(exact.astype(np.float32)).to(out)
        assert torch.equal(got.cpu(), ref)


@pytest.mark.parametrize("wfmt", [moe_synth.WFMT_INT4, moe_synth.WFMT_INT4_AFFINE])
def test_prefill_on_dequantised_weights_equals_fused_int4(wfmt):
    wl = moe_synth.Workload("dqp", moe_synth.QWEN, T=300, bias_std=1.5, wfmt=wfmt, seed=33)
    ctx4, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y4 = ctx4.forward_prefill(0, x)
    s = wl.shape
    ctxb = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter)
    wb = {"router_w": w["router_w"], "router_b": w["router_b"], "sh_gate_w": w["sh_gate_w"]}
    for name in ("gate_up", "sh_gate_up", "down", "sh_down"):
        wb[name] = dequant_int4(w[name], w[name + "_scale"], w.get(name + "_bias"))
    wb["down_f16"] = dequant_int4(w["down"], w["down_scale"], w.get("down_bias"),
                                  out_dtype=torch.float16)
    wb["sh_down_f16"] = dequant_int4(w["sh_down"], w["sh_down_scale"], w.get("sh_down_bias"),
                                     out_dtype=torch.float16)
    ctxb.load_weights(0, wb)
    yb = ctxb.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y4, yb)


# ---- the ablation switches (measurement options read at context creation)
# change how the work is scheduled, never a result: each output row is the
# same dot products in the same order whatever block it lands in.

@pytest.mark.parametrize("env", [{"MOE_ABLATE_HOST_ROUTING": "1"}, {"MOE_ABLATE_TILE": "fixed256"},
                                 {"MOE_ABLATE_TILE": "rows16"}, {"MOE_ABLATE_TILE": "rows48"}])
def test_ablation_switches_change_no_result(env, monkeypatch):
    wl = _wl(moe_synth.QWEN, 700, bias=1.5, seed=41)
    ctx, (w,) = make_ctx(wl)
    x = moe_synth.make_x(wl, device="cuda")
    y0 = ctx.forward_prefill(0, x)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    s = wl.shape
    ctx2 = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter)
    ctx2.load_weights(0, w)
    y1 = ctx2.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert ctx2.check_device() == 0
