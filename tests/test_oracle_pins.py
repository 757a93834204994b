"""Pins for the fp64 CPU oracle: brute force on tiny inputs, closed forms,
library routines for the special cases, invariants, and the numbers the page
prints.  None of these re-types the oracle's own formulas: each checks it
against something computed another way."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import moe_synth
from oracle import moe_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_inputs(seed=0, T=None):
    wl = moe_synth.TINY_LAYER
    if seed != wl.seed:
        wl = moe_synth.Workload("tiny", wl.shape, T=wl.T, seed=seed)
    x = moe_synth.make_x(wl, T=T).float().numpy()
    layer = moe_synth.to_numpy(moe_synth.make_layer(wl))
    return wl, x, layer


# ------------------------------------------------------------ selection --

def _valid_topk(l, S, k):
    """S is the top-k set iff every member beats every non-member under the
    order (larger logit first, then lower index)."""
    E = l.size
    for s in S:
        for u in range(E):
            if u in S:
                continue
            if not (l[s] > l[u] or (l[s] == l[u] and s < u)):
                return False
    return True


def test_topk_bruteforce_tiny():
    wl, x, layer = tiny_inputs()
    k, E = wl.shape.top_k, wl.shape.n_experts
    logits = orc.router_logits(x, layer["router_w"])
    idx = orc.select_topk(logits, k)
    for t in range(x.shape[0]):
        valid = [S for S in itertools.combinations(range(E), k) if _valid_topk(logits[t], S, k)]
        assert len(valid) == 1                              # all C(16,2) = 120 pairs tried
        assert set(idx[t].tolist()) == set(valid[0])
        # slot order: descending logit
        vals = logits[t, idx[t]]
        assert np.all(vals[:-1] >= vals[1:])


def test_topk_ties_prefer_lower_expert():
    l = np.array([[0.5, 1.0, 1.0, 0.2, 1.0, -3.0],
                  [0.0, -0.0, 0.0, 0.0, -1.0, -1.0]], dtype=np.float32)
    idx = orc.select_topk(l, 2)
    assert idx[0].tolist() == [1, 2]
    assert idx[1].tolist() == [0, 1]          # -0.0 equals 0.0: index decides
    assert orc.select_topk(l, 4)[0].tolist() == [1, 2, 4, 0]


def test_topk_bruteforce_with_ties_random():
    rng = np.random.default_rng(7)
    for _ in range(40):
        E, k = 7, 3
        l = rng.integers(-2, 3, size=E).astype(np.float64)   # many exact ties
        idx = orc.select_topk(l[None], k)[0]
        valid = [S for S in itertools.combinations(range(E), k) if _valid_topk(l, S, k)]
        assert len(valid) == 1 and set(idx.tolist()) == set(valid[0])
        order = sorted(valid[0], key=lambda e: (-l[e], e))
        assert idx.tolist() == order


# -------------------------------------------------------------- weights --

def test_weights_equal_softmax_of_selected_logits():
    """softmax-then-renormalise equals a softmax over the selected logits
    (scipy's softmax on the selected entries only)."""
    wl, x, layer = tiny_inputs()
    logits = orc.router_logits(x, layer["router_w"])
    idx = orc.select_topk(logits, wl.shape.top_k)
    w = orc.topk_weights(logits, idx)
    ref = scipy.special.softmax(np.take_along_axis(logits, idx, 1), axis=1)
    np.testing.assert_allclose(w, ref, rtol=1e-13, atol=0)


def test_weights_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(3)
    l = rng.normal(size=(5, 9)) * 3
    idx = orc.select_topk(l, 9)
    w = orc.topk_weights(l, idx)
    full = scipy.special.softmax(l, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx, 1), rtol=1e-13)


def test_weights_k1_is_one():
    rng = np.random.default_rng(4)
    l = rng.normal(size=(11, 16))
    w = orc.topk_weights(l, orc.select_topk(l, 1))
    assert np.all(w == 1.0)


def test_weight_invariants_qwen_shape():
    rng = np.random.default_rng(5)
    l = rng.normal(size=(300, 256)) + rng.normal(scale=1.5, size=256)[None]
    r = orc.route(l, 8)
    w = r["topk_w"]
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-12)
    assert np.all(w > 0)
    assert np.all(w[:, :-1] >= w[:, 1:])


# ------------------------------------------------------------- grouping --

def _grouping_bruteforce(idx, E):
    T, k = idx.shape
    lists = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            lists[idx[t, j]].append((t, j))
    counts = [len(lst) for lst in lists]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    sorted_rows = []
    pos = [None] * (T * k)
    for e in range(E):
        for (t, j) in lists[e]:
            pos[t * k + j] = len(sorted_rows)
            sorted_rows.append(t)
    return counts, offsets, sorted_rows, pos


@pytest.mark.parametrize("T,E,k,bias", [(16, 16, 2, 0.0), (37, 16, 4, 2.0), (200, 256, 8, 1.5)])
def test_grouping_bruteforce(T, E, k, bias):
    rng = np.random.default_rng(T)
    l = rng.normal(size=(T, E)) + rng.normal(scale=bias, size=E)[None]
    idx = orc.select_topk(l, k)
    g = orc.group_by_expert(idx, E)
    counts, offsets, sorted_rows, pos = _grouping_bruteforce(idx, E)
    assert g["counts"].tolist() == counts
    assert g["offsets"].tolist() == offsets
    assert g["sorted_rows"].tolist() == sorted_rows
    assert g["pos_of_assign"].tolist() == pos


def test_grouping_invariants():
    rng = np.random.default_rng(11)
    T, E, k = 513, 256, 8
    l = rng.normal(size=(T, E)) + rng.normal(scale=1.5, size=E)[None]
    idx = orc.select_topk(l, k)
    g = orc.group_by_expert(idx, E)
    pos = g["pos_of_assign"]
    assert sorted(pos.tolist()) == list(range(T * k))          # bijection
    t_of = np.repeat(np.arange(T), k)
    assert np.all(g["sorted_rows"][pos] == t_of)
    assert g["counts"].sum() == T * k
    off = g["offsets"]
    for t in range(0, T, 17):                                  # each token in k distinct segments
        segs = {int(np.searchsorted(off, p, side="right") - 1) for p in pos[t * k:(t + 1) * k]}
        assert segs == set(idx[t].tolist())
    for e in range(E):                                         # ascending tokens inside a segment
        seg = g["sorted_rows"][off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_pages_routing_load_2k_prompt():
    gold = json.load(open(os.path.join(GOLDEN, "pages_routing_load.json")))
    rng = np.random.default_rng(0)
    T, E, k = gold["T"], gold["n_experts"], gold["top_k"]
    l = rng.normal(size=(T, E)) + rng.normal(scale=1.5, size=E)[None]
    g = orc.group_by_expert(orc.select_topk(l, k), E)
    assert int(g["counts"].sum()) == gold["assignments"]
    assert g["counts"].sum() / E == gold["mean_rows_per_expert"]
    assert g["counts"].max() > 2 * gold["mean_rows_per_expert"]   # uneven under a skewing bias


# ---------------------------------------------------------- layer output --

def _torch_swiglu(x, w_gate_up, w_down):
    """Dense SwiGLU FFN with torch's library routines (fp64)."""
    I = w_gate_up.shape[0] // 2
    xt = torch.from_numpy(np.asarray(x, np.float64))
    wg = torch.from_numpy(np.asarray(w_gate_up[:I], np.float64))
    wu = torch.from_numpy(np.asarray(w_gate_up[I:], np.float64))
    wd = torch.from_numpy(np.asarray(w_down, np.float64))
    return F.linear(F.silu(F.linear(xt, wg)) * F.linear(xt, wu), wd).numpy()


def test_sparse_equals_dense_masked_tiny():
    """Every expert evaluated densely, masked by the routing weights (zero for
    unselected experts), equals the sparse grouped evaluation."""
    wl, x, layer = tiny_inputs()
    k, E = wl.shape.top_k, wl.shape.n_experts
    logits = orc.router_logits(x, layer["router_w"])
    idx = orc.select_topk(logits, k)
    G = np.zeros((x.shape[0], E))
    sel = np.take_along_axis(logits, idx, 1)
    np.put_along_axis(G, idx, scipy.special.softmax(sel, axis=1), 1)
    y_dense = np.zeros_like(x, dtype=np.float64)
    for e in range(E):
        y_dense += G[:, e:e + 1] * _torch_swiglu(x, layer["gate_up"][e], layer["down"][e])
    gate = scipy.special.expit(x.astype(np.float64) @ layer["sh_gate_w"].astype(np.float64))
    y_dense += gate[:, None] * _torch_swiglu(x, layer["sh_gate_up"], layer["sh_down"])
    y = orc.moe_layer(x, layer, k)
    np.testing.assert_allclose(y, y_dense, rtol=1e-10, atol=1e-13)


def test_token_subset_matches_full():
    wl, x, layer = tiny_inputs()
    y = orc.moe_layer(x, layer, wl.shape.top_k)
    sub = [3, 0, 15, 7]
    ys = orc.moe_layer(x, layer, wl.shape.top_k, tokens=sub)
    np.testing.assert_allclose(ys, y[sub], rtol=1e-12, atol=1e-15)


def _identity_like_layer(H, E, I, alpha, shared_same):
    gate_up = np.zeros((E, 2 * I, H))
    down = np.zeros((E, H, I))
    for i in range(I):
        gate_up[:, i, i] = alpha
        gate_up[:, I + i, i] = 1.0
        down[:, i, i] = 1.0
    rng = np.random.default_rng(1)
    layer = dict(router_w=rng.normal(scale=0.3, size=(E, H)), router_b=None,
                 gate_up=gate_up, down=down,
                 sh_gate_up=gate_up[0] if shared_same else np.zeros((2 * I, H)),
                 sh_down=down[0] if shared_same else np.zeros((H, I)),
                 sh_gate_w=rng.normal(scale=0.1, size=H))
    return layer


@pytest.mark.parametrize("shared_same", [False, True])
def test_identity_like_closed_form(shared_same):
    """Routed experts with Wg = alpha*[I|0], Wu = [I|0], Wd = [I;0]: every
    expert maps x to silu(alpha x_n) x_n on the first I features and 0 on the
    rest, so with weights summing to one y is that, whatever the routing.
    With the same shared expert, y is multiplied by (1 + sigmoid(x . w_sg))."""
    H, E, I, k, alpha = 24, 6, 10, 3, 0.7
    layer = _identity_like_layer(H, E, I, alpha, shared_same)
    x = np.random.default_rng(2).normal(size=(9, H))
    y = orc.moe_layer(x, layer, k)
    xt = torch.from_numpy(x)
    expect = torch.zeros_like(xt)
    expect[:, :I] = F.silu(alpha * xt[:, :I]) * xt[:, :I]
    if shared_same:
        expect = expect * (1.0 + torch.sigmoid(xt @ torch.from_numpy(layer["sh_gate_w"])))[:, None]
    np.testing.assert_allclose(y, expect.numpy(), rtol=1e-12, atol=1e-14)


def test_identical_experts_reduce_to_dense_ffn():
    """All routed experts equal: the output is one dense SwiGLU FFN for any
    routing (plus the gated shared expert)."""
    wl, x, layer = tiny_inputs()
    layer = dict(layer)
    layer["gate_up"] = np.repeat(layer["gate_up"][3:4], wl.shape.n_experts, 0)
    layer["down"] = np.repeat(layer["down"][3:4], wl.shape.n_experts, 0)
    y = orc.moe_layer(x, layer, wl.shape.top_k)
    ref = _torch_swiglu(x, layer["gate_up"][0], layer["down"][0])
    gate = scipy.special.expit(x.astype(np.float64) @ layer["sh_gate_w"].astype(np.float64))
    ref = ref + gate[:, None] * _torch_swiglu(x, layer["sh_gate_up"], layer["sh_down"])
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-13)


def test_shared_expert_sigmoid_gate():
    """Routed experts zero: y = sigmoid(x . w_sg) * SwiGLU_shared(x)."""
    wl, x, layer = tiny_inputs()
    layer = dict(layer)
    layer["down"] = np.zeros_like(layer["down"])
    y = orc.moe_layer(x, layer, wl.shape.top_k)
    gate = scipy.special.expit(x.astype(np.float64) @ layer["sh_gate_w"].astype(np.float64))
    ref = gate[:, None] * _torch_swiglu(x, layer["sh_gate_up"], layer["sh_down"])
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-14)


def test_router_bias_shapes_selection_and_weights():
    wl, x, layer = tiny_inputs()
    E = wl.shape.n_experts
    b = np.zeros(E)
    b[5] = 100.0
    l = orc.router_logits(x, layer["router_w"], b)
    assert np.all(orc.select_topk(l, 2)[:, 0] == 5)
    b = np.random.default_rng(9).normal(scale=1.5, size=E)
    l = orc.router_logits(x, layer["router_w"], b)
    raw = x.astype(np.float64) @ layer["router_w"].astype(np.float64).T
    idx = orc.select_topk(l, E)
    w = orc.topk_weights(l, idx)
    np.testing.assert_allclose(w, np.take_along_axis(scipy.special.softmax(raw + b, 1), idx, 1),
                               rtol=1e-12)


def test_silu_sigmoid_match_library():
    z = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(orc.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14,
                               atol=1e-300)
    np.testing.assert_allclose(orc.sigmoid(z), scipy.special.expit(z), rtol=1e-14)


# ----------------------------------------------------------------- int4 --

def test_int4_nibble_decoding_golden():
    gold = json.load(open(os.path.join(GOLDEN, "int4_nibbles.json")))
    byts = np.array([[int(c["byte"], 16) for c in gold["cases"]]], dtype=np.uint8)
    codes = np.array([c["codes"] for c in gold["cases"]]).reshape(1, -1)
    K = byts.shape[1] * 2
    pad = (-K) % 64
    byts = np.concatenate([byts, np.zeros((1, pad // 2), np.uint8)], 1)
    w = orc.dequant_int4_sym_g64(byts, np.ones((1, byts.shape[1] * 2 // 64)))
    assert w[0, :K].tolist() == codes[0].tolist()
    assert sorted(set(codes[0].tolist())) == list(range(-8, 8))   # all 16 codes covered
    packed = moe_synth.pack_int4(torch.tensor(codes, dtype=torch.int16))
    assert packed.numpy()[0].tolist() == byts[0, :K // 2].tolist()


def test_int4_onehot_gemv_returns_dequantised_column():
    """x = e_k through a GEMV picks column k: scale of group k // 64 times the
    code, exactly (pins group indexing)."""
    R, K = 3, 192
    codes = np.array([[((r * 5 + k * 3) % 15) - 7 for k in range(K)] for r in range(R)])
    scales = np.array([[2.0 ** -(r + g + 1) for g in range(K // 64)] for r in range(R)])
    packed = moe_synth.pack_int4(torch.tensor(codes, dtype=torch.int16)).numpy()
    W = orc.dequant_int4_sym_g64(packed, scales)
    for k in (0, 1, 63, 64, 65, 127, 128, 191):
        x = np.zeros(K)
        x[k] = 1.0
        col = W @ x
        for r in range(R):
            assert col[r] == codes[r, k] * 2.0 ** -(r + k // 64 + 1)


def test_int4_layer_equals_layer_on_dequantised_weights():
    wl = moe_synth.Workload("tiny_int4", moe_synth.TINY, T=8, wfmt=moe_synth.WFMT_INT4, seed=3)
    x = moe_synth.make_x(wl).float().numpy()
    layer = moe_synth.to_numpy(moe_synth.make_layer(wl))
    deq = dict(layer)
    for name in ("gate_up", "down", "sh_gate_up", "sh_down"):
        deq[name] = orc.dequant_int4_sym_g64(layer[name], layer[name + "_scale"])
        deq[name + "_scale"] = None
    np.testing.assert_allclose(orc.moe_layer(x, layer, 2), orc.moe_layer(x, deq, 2),
                               rtol=1e-13, atol=1e-16)


# ------------------------------------------------------------ generator --

def test_generator_distributions():
    wl = moe_synth.Workload("g", moe_synth.TINY, T=512, bias_std=1.5, seed=5)
    x = moe_synth.make_x(wl).float()
    L = moe_synth.make_layer(wl)
    assert abs(x.std().item() - 1.0) < 0.02
    assert abs(L["gate_up"].float().std().item() - 0.02) < 0.001
    assert abs(L["router_b"].std().item() - 1.5) < 0.6
    wl4 = moe_synth.Workload("g4", moe_synth.TINY, T=4, wfmt=moe_synth.WFMT_INT4, seed=5)
    L4 = moe_synth.to_numpy(moe_synth.make_layer(wl4))
    q = orc.dequant_int4_sym_g64(L4["gate_up"], np.ones_like(L4["gate_up_scale"]))
    assert q.min() == -7 and q.max() == 7
    assert np.all(L4["gate_up_scale"] > 0)
    # same seed, same bytes
    again = moe_synth.to_numpy(moe_synth.make_layer(wl4))
    assert np.array_equal(again["down"], L4["down"])


# --------------------------------------------------------- int4 affine --

def test_int4_affine_nibble_decoding_golden():
    """Unsigned codes, low nibble first, from hand-decoded bytes; all 16 codes
    appear; scale 1 and bias 0 return the codes themselves."""
    gold = json.load(open(os.path.join(GOLDEN, "int4_affine_nibbles.json")))
    byts = np.array([[int(c["byte"], 16) for c in gold["cases"]]], dtype=np.uint8)
    codes = np.array([c["codes"] for c in gold["cases"]]).reshape(1, -1)
    K = byts.shape[1] * 2
    pad = (-K) % 64
    byts = np.concatenate([byts, np.zeros((1, pad // 2), np.uint8)], 1)
    G = byts.shape[1] * 2 // 64
    w = orc.dequant_int4_affine_g64(byts, np.ones((1, G)), np.zeros((1, G)))
    assert w[0, :K].tolist() == codes[0].tolist()
    assert sorted(set(codes[0].tolist())) == list(range(16))


def test_int4_affine_with_bias_minus_8_scale_is_symmetric_format():
    """Closed form linking the two formats: for any bytes, flipping the top bit
    of every nibble (u -> u ^ 8) maps the unsigned code u to the two's-complement
    code q with u ^ 8 - 8 = q, so affine(bytes ^ 0x88, s, -8 s) == symmetric(bytes, s)."""
    rng = np.random.default_rng(7)
    byts = rng.integers(0, 256, size=(5, 96), dtype=np.uint8)
    # dyadic scales (small integer times a power of two): every product and
    # sum below is exact in fp64, so the two sides must agree bit for bit
    s = rng.choice([-1.0, 1.0], (5, 3)) * rng.integers(1, 64, (5, 3)) * 2.0 ** -rng.integers(
        4, 12, (5, 3)).astype(np.float64)
    sym = orc.dequant_int4_sym_g64(byts, s)
    aff = orc.dequant_int4_affine_g64(byts ^ np.uint8(0x88), s, -8.0 * s)
    np.testing.assert_array_equal(aff, sym)


def test_int4_affine_onehot_gemv_returns_dequantised_column():
    """x = e_k through a GEMV picks column k: scale * code + bias of group
    k // 64, exactly (dyadic scales and biases)."""
    R, K = 3, 192
    codes = np.array([[(r * 7 + k * 5) % 16 for k in range(K)] for r in range(R)])
    scales = np.array([[2.0 ** -(r + g + 2) for g in range(K // 64)] for r in range(R)])
    biases = np.array([[-(g + 1) * 2.0 ** -(r + 1) for g in range(K // 64)] for r in range(R)])
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    W = orc.dequant_int4_affine_g64(packed, scales, biases)
    for k in (0, 1, 63, 64, 65, 127, 128, 191):
        x = np.zeros(K)
        x[k] = 1.0
        col = W @ x
        for r in range(R):
            g = k // 64
            assert col[r] == codes[r, k] * 2.0 ** -(r + g + 2) - (g + 1) * 2.0 ** -(r + 1)


def test_int4_affine_layer_equals_layer_on_dequantised_weights():
    wl = moe_synth.Workload("tiny_int4a", moe_synth.TINY, T=8, wfmt=moe_synth.WFMT_INT4_AFFINE,
                            seed=4)
    x = moe_synth.make_x(wl).float().numpy()
    layer = moe_synth.to_numpy(moe_synth.make_layer(wl))
    deq = dict(layer)
    for name in ("gate_up", "down", "sh_gate_up", "sh_down"):
        deq[name] = orc.dequant_int4_affine_g64(layer[name], layer[name + "_scale"],
                                                layer[name + "_bias"])
        deq[name + "_scale"] = deq[name + "_bias"] = None
    np.testing.assert_allclose(orc.moe_layer(x, layer, 2), orc.moe_layer(x, deq, 2),
                               rtol=1e-13, atol=1e-16)


def test_generator_affine_distribution():
    wl = moe_synth.Workload("g4a", moe_synth.TINY, T=4, wfmt=moe_synth.WFMT_INT4_AFFINE, seed=5)
    L = moe_synth.to_numpy(moe_synth.make_layer(wl))
    G = L["gate_up_scale"].shape
    q = orc.dequant_int4_affine_g64(L["gate_up"], np.ones(G), np.zeros(G))
    assert q.min() == 0 and q.max() == 15
    s, b = L["gate_up_scale"], L["gate_up_bias"]
    assert np.all(s > 0) and np.all(b < 0)
    assert abs(np.median(-b / s) - 7.5) < 0.1
    w = orc.dequant_int4_affine_g64(L["gate_up"], s, b)
    assert abs(w.mean()) < 1e-3 and 0.01 < w.std() < 0.04
