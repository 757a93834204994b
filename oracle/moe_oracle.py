"""Plain, slow fp64 CPU oracle for the sparse mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke entry and the
benchmark's CPU-baseline leg may import this module.  It shares no code with
the CUDA library and never imports it; its only common dependency with the
CUDA side is the seeded input generator (`moe_synth`), which holds no layer
arithmetic.

What it computes follows "Optimizing On-Device Inference for Apple Silicon"
(Perplexity), sections
  * "Qwen creates three distinct workload shapes": a router scores 256 experts
    and selects eight per token; one shared expert processes every token;
  * "Keep expert routing on the GPU": assignments are counted per expert
    (histogram), turned into start offsets (prefix scan), and rows are placed
    into per-expert groups (scatter);
  * "Reduce intermediate and state traffic": each expert applies two input
    projections with a gated activation, then an output projection, and the
    result is combined with its routing score and the shared-expert result;
  * "Dequantize weights during matrix multiplication": weights may be stored
    as 4-bit codes with one bf16 scale per group of 64 along the reduction
    dimension; accumulation is in 32-bit float on the device.

Readings of what the page leaves open (each one is stated where it is used):
  * routing weights are softmax over all experts' logits, renormalised over
    the selected ones;
  * selection is on logits, descending, ties broken by the lower expert index;
  * a per-expert router bias, when present, is added to the logits before
    both selection and softmax;
  * the gated activation is SwiGLU: silu(gate) * up, silu(z) = z / (1 + e^-z);
  * the shared expert's output is scaled by sigmoid(x . w_sg), a scalar per
    token, and is not renormalised with the routed weights;
  * the int4 formats: symmetric, w = scale * q with q the two's-complement
    nibble in [-8, 7]; and affine (the page's checkpoint format: a bf16 scale
    and a bf16 bias per group of 64), w = scale * q + bias with q the unsigned
    nibble in [0, 15]; element 2m in the low nibble of byte m in both;
  * inside an expert's group, rows are ordered by ascending token index.

Everything is evaluated in float64 with no intermediate rounding.
"""
from __future__ import annotations

import numpy as np

GROUP = 64


# ----------------------------------------------------------------- weights --

def dequant_int4_sym_g64(packed, scale) -> np.ndarray:
    """Symmetric int4, group 64 along K: w[r, k] = scale[r, k // 64] * q[r, k].

    `packed` is uint8 [..., K/2]; byte m holds element 2m in its low nibble and
    element 2m+1 in its high nibble, each a two's-complement code in [-8, 7].
    The page's section "Dequantize weights during matrix multiplication"
    describes 4-bit codes with a bf16 parameter per group of 64 weights.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    K = packed.shape[-1] * 2
    q = np.empty(packed.shape[:-1] + (K,), dtype=np.int64)
    q[..., 0::2] = packed & 0x0F
    q[..., 1::2] = packed >> 4
    q = np.where(q >= 8, q - 16, q)
    s = np.asarray(scale, dtype=np.float64)
    assert s.shape[-1] * GROUP == K, "one scale per 64 elements along K"
    return np.repeat(s, GROUP, axis=-1) * q


def dequant_int4_affine_g64(packed, scale, bias) -> np.ndarray:
    """Affine int4, group 64 along K: w[r, k] = scale[r, k // 64] * q[r, k] +
    bias[r, k // 64], q the unsigned code in [0, 15] (same packing as the
    symmetric format).  Section "Dequantize weights during matrix
    multiplication": each weight is a 4-bit integer code, and every group of 64
    weights shares a bfloat16 scale and bias that reconstruct its values.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    K = packed.shape[-1] * 2
    q = np.empty(packed.shape[:-1] + (K,), dtype=np.int64)
    q[..., 0::2] = packed & 0x0F
    q[..., 1::2] = packed >> 4
    s = np.asarray(scale, dtype=np.float64)
    b = np.asarray(bias, dtype=np.float64)
    assert s.shape[-1] * GROUP == K and b.shape == s.shape, "one scale and bias per 64 along K"
    return np.repeat(s, GROUP, axis=-1) * q + np.repeat(b, GROUP, axis=-1)


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _matrix(layer: dict, name: str, index=None) -> np.ndarray:
    """A weight matrix (or one expert's slice of it) in float64."""
    w = layer[name]
    s = layer.get(name + "_scale")
    b = layer.get(name + "_bias")
    if index is not None:
        w = w[index]
        s = None if s is None else s[index]
        b = None if b is None else b[index]
    if s is None:
        return _f64(w)
    if b is not None:
        return dequant_int4_affine_g64(w, s, b)
    return dequant_int4_sym_g64(w, s)


def layer_dims(layer: dict) -> dict:
    E, H = layer["router_w"].shape
    I = layer["gate_up"].shape[-2] // 2
    Is = layer["sh_gate_up"].shape[0] // 2
    return dict(E=E, H=H, I=I, Is=Is)


# ------------------------------------------------------------------ router --

def router_logits(x, router_w, router_b=None) -> np.ndarray:
    """l[t, e] = sum_h x[t, h] * Wr[e, h] (+ b[e]).  The router "scores" each
    expert (section "Qwen creates three distinct workload shapes")."""
    l = _f64(x) @ _f64(router_w).T
    if router_b is not None:
        l = l + _f64(router_b)[None, :]
    return l


def select_topk(logits, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, in descending logit order;
    equal logits are ordered by the lower expert index (a stable sort of the
    negated logits).  Works on the logits' own precision: fp32 inputs are
    compared exactly as fp32 values (the widening to fp64 is exact)."""
    l = _f64(logits)
    order = np.argsort(-l, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def topk_weights(logits, idx) -> np.ndarray:
    """Softmax over all experts, renormalised over the selected ones, fp64."""
    l = _f64(logits)
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def group_by_expert(idx, n_experts: int) -> dict:
    """Histogram, exclusive prefix scan and scatter of the (token, slot)
    assignments into per-expert row segments (section "Keep expert routing on
    the GPU").  Assignment a = t * k + j.  Within an expert's segment rows are
    in ascending token order; each token selects an expert at most once, so
    ordering the assignments stably by expert gives exactly that order.

    Returns counts[E], offsets[E+1], sorted_rows[T*k] (token of each grouped
    row) and pos_of_assign[T*k] (grouped row of each assignment)."""
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=n_experts).astype(np.int64)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")          # assignments by (expert, t)
    sorted_rows = order // k
    pos_of_assign = np.empty(T * k, dtype=np.int64)
    pos_of_assign[order] = np.arange(T * k, dtype=np.int64)
    return dict(counts=counts, offsets=offsets, sorted_rows=sorted_rows,
                pos_of_assign=pos_of_assign)


def route(logits, k: int) -> dict:
    """Top-k selection, renormalised weights and the per-expert grouping."""
    l = _f64(logits)
    idx = select_topk(l, k)
    out = group_by_expert(idx, l.shape[1])
    out["topk_idx"] = idx
    out["topk_w"] = topk_weights(l, idx)
    return out


# ----------------------------------------------------------------- experts --

def silu(z):
    return z / (1.0 + np.exp(-z))


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def swiglu_ffn(x_rows, w_gate_up, w_down) -> np.ndarray:
    """down( silu(gate(x)) * up(x) ).  w_gate_up is [2I, H] with the gate rows
    first, w_down is [H, I]; both K-major, fp64."""
    I = w_gate_up.shape[0] // 2
    g = x_rows @ w_gate_up[:I].T
    u = x_rows @ w_gate_up[I:].T
    return (silu(g) * u) @ w_down.T


def shared_gate(x, sh_gate_w) -> np.ndarray:
    """sigmoid(x . w_sg), one scalar per token."""
    return sigmoid(_f64(x) @ _f64(sh_gate_w))


def moe_layer(x, layer: dict, k: int, logits=None, tokens=None) -> np.ndarray:
    """y[t] = sum_j w[t,j] * FFN_{idx[t,j]}(x[t]) + sigmoid(x[t].w_sg) * FFN_shared(x[t]).

    `logits` are the router logits used for selection and weights; when None
    the oracle's own fp64 logits are used.  `tokens` restricts the evaluation
    to a subset of rows (returns those rows only, in the given order).
    Each expert's rows are evaluated together with one matmul per projection:
    the rows are independent, so this changes no arithmetic of any row."""
    x = _f64(x)
    if logits is None:
        logits = router_logits(x, layer["router_w"], layer.get("router_b"))
    logits = _f64(logits)
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        x = x[tokens]
        logits = logits[tokens]
    T, H = x.shape
    r = route(logits, k)
    idx, w = r["topk_idx"], r["topk_w"]
    y = np.zeros((T, H), dtype=np.float64)
    E = logits.shape[1]
    for e in range(E):
        t_sel, j_sel = np.nonzero(idx == e)
        if t_sel.size == 0:
            continue
        o = swiglu_ffn(x[t_sel], _matrix(layer, "gate_up", e), _matrix(layer, "down", e))
        y[t_sel] += w[t_sel, j_sel][:, None] * o
    s = swiglu_ffn(x, _matrix(layer, "sh_gate_up"), _matrix(layer, "sh_down"))
    y += shared_gate(x, layer["sh_gate_w"])[:, None] * s
    return y
