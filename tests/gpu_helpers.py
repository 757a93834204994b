"""Helpers for the GPU parity tests: build a context from a synthetic
workload, hand the oracle host copies of exactly the tensors it needs, and
apply the layer-output tolerances.

Tolerances (layer output y, bf16 on the GPU vs the fp64 oracle):
  bf16 weights: max|err| <= 1e-2 * max|ref|  and  mean|err| / mean|ref| <= 2e-3
  int4 weights: max|err| <= 2e-2 * max|ref|
Routing indices, counts, offsets and the permutation: bit-exact, with the
oracle selecting from the GPU's fp32 logits.  Routing weights: |err| <= 4e-6.
"""
import numpy as np
import torch

import moe_synth
from oracle import moe_oracle as orc
from sparse_moe_gb300 import MoEContext

WEIGHT_KEYS = ("router_w", "router_b", "gate_up", "gate_up_scale", "gate_up_bias", "down",
               "down_scale", "down_bias", "sh_gate_up", "sh_gate_up_scale", "sh_gate_up_bias",
               "sh_down", "sh_down_scale", "sh_down_bias", "sh_gate_w")


def make_ctx(wl, n_layers=1, max_chunk_rows=4096, seed_layers=None):
    s = wl.shape
    ctx = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, n_layers=n_layers,
                     max_chunk_rows=max_chunk_rows, wfmt=wl.wfmt)
    layers = []
    for i in range(n_layers):
        src = i if seed_layers is None else seed_layers[i]
        w = moe_synth.make_layer(wl, layer=src, device="cuda")
        ctx.load_weights(i, w)
        layers.append(w)
    return ctx, layers


class _LazyExperts:
    """Per-expert host copies on demand (the oracle indexes experts one by one)."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        v = self.t[e]
        return v.float().cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy()


def host_layer(w: dict) -> dict:
    """Oracle view of a device layer: small tensors copied, routed experts lazy."""
    out = {}
    for k in WEIGHT_KEYS:
        v = w.get(k)
        if v is None:
            out[k] = None
        elif k in ("gate_up", "gate_up_scale", "gate_up_bias", "down", "down_scale", "down_bias"):
            out[k] = _LazyExperts(v)
        else:
            out[k] = v.float().cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy()
    return out


def logits_bound(x_np, router_w_np, ref, bias_np=None):
    """Rigorous bound on |fp32 logits - exact| for a length-H dot product of
    exactly-multiplied bf16 values accumulated in fp32 (any order, any rounding
    mode with unit error <= 2^-23), plus the bias addition."""
    H = x_np.shape[1]
    absdot = np.abs(x_np.astype(np.float64)) @ np.abs(router_w_np.astype(np.float64)).T
    b = 0.0 if bias_np is None else np.abs(bias_np)[None, :]
    return H * 2.0 ** -23 * absdot + 2.0 ** -23 * (np.abs(ref) + b) + 1e-30


def check_routing(ctx, w, x, T=None):
    """Runs moe_route and checks it against the oracle.  Returns the GPU logits."""
    r = ctx.route(0, x)
    torch.cuda.synchronize()
    k, E = ctx.top_k, ctx.n_experts
    lg = r["logits"].cpu().numpy()
    x_np = x.float().cpu().numpy()
    wr = w["router_w"].float().cpu().numpy()
    b = None if w.get("router_b") is None else w["router_b"].cpu().numpy()
    ref = orc.router_logits(x_np, wr, b)
    bound = logits_bound(x_np, wr, ref, b)
    assert np.all(np.abs(lg.astype(np.float64) - ref) <= bound), \
        f"router logits outside the fp32 bound: max err {np.abs(lg - ref).max()}"
    o = orc.route(lg, k)
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), o["topk_idx"])
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), o["counts"])
    np.testing.assert_array_equal(r["offsets"].cpu().numpy(), o["offsets"])
    np.testing.assert_array_equal(r["sorted_rows"].cpu().numpy(), o["sorted_rows"])
    np.testing.assert_array_equal(r["pos_of_assign"].cpu().numpy(), o["pos_of_assign"])
    werr = np.abs(r["topk_w"].cpu().numpy().astype(np.float64) - o["topk_w"]).max()
    assert werr <= 4e-6, werr
    return lg


def assert_layer_close(y_gpu, y_ref, int4=False, what=""):
    y = np.asarray(y_gpu, dtype=np.float64)
    ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == ref.shape
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    max_ref = np.abs(ref).max()
    tol = (2e-2 if int4 else 1e-2) * max_ref
    assert err.max() <= tol, f"{what}: max|err| {err.max():.3e} > {tol:.3e}"
    if not int4:
        rel = err.mean() / np.abs(ref).mean()
        assert rel <= 2e-3, f"{what}: mean relative error {rel:.3e} > 2e-3"
    return float(err.max() / max_ref)
