"""Seeded synthetic inputs for the sparse mixture-of-experts layer.

This module only draws random numbers and lays them out in the storage format
both sides consume (the CUDA library and the CPU oracle).  It holds none of the
layer's arithmetic: no routing, no matmul, no activation, no dequantisation.

Workloads follow the shapes of the Qwen3.6-35B-A3B MoE layer described in
"Optimizing On-Device Inference for Apple Silicon" (section "Qwen creates three
distinct workload shapes": 256 routed experts, top-8, one shared expert), with
hidden size 2048 and expert intermediate size 512, plus a tiny variant that a
slow CPU reference finishes in seconds.

Storage layout (row-major, every weight K-major: each output row contiguous
along the reduction dimension):

    router_w      bf16  [E, H]
    router_b      fp32  [E]            (or None)
    gate_up       bf16  [E, 2I, H]     rows 0..I-1 = gate, rows I..2I-1 = up
    down          bf16  [E, H, I]
    sh_gate_up    bf16  [2Is, H]       rows 0..Is-1 = gate, Is..2Is-1 = up
    sh_down       bf16  [H, Is]
    sh_gate_w     bf16  [H]

int4 symmetric, group 64 along K (the compressed variant):
    <name>        uint8 [rows, K/2]    code of element 2m in the low nibble,
                                       element 2m+1 in the high nibble,
                                       two's complement in [-8, 7]
    <name>_scale  bf16  [rows, K/64]

Codes are drawn uniformly from [-7, 7]; scales are |N(0, 0.02)| / 7.

int4 affine, group 64 along K (the checkpoint format of section "Dequantize
weights during matrix multiplication": a bf16 scale and a bf16 bias per group):
    <name>        uint8 [rows, K/2]    unsigned codes in [0, 15], same packing
    <name>_scale  bf16  [rows, K/64]
    <name>_bias   bf16  [rows, K/64]   (weight = scale * code + bias)

Codes are drawn uniformly from [0, 15]; scales are |N(0, 0.02)| / 7 and biases
-scale * (7.5 + N(0, 0.5)), so each group spans about the range a min-max
quantiser of N(0, 0.02) weights would give it.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

WFMT_BF16 = "bf16"
WFMT_INT4 = "int4_sym_g64"
WFMT_INT4_AFFINE = "int4_affine_g64"

GROUP = 64


@dataclasses.dataclass(frozen=True)
class Shape:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int


QWEN = Shape(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512)
TINY = Shape(hidden=256, n_experts=16, top_k=2, inter=64, shared_inter=64)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    T: int
    wfmt: str = WFMT_BF16
    bias_std: Optional[float] = None   # per-expert router bias ~ N(0, bias_std)
    seed: int = 0
    n_layers: int = 1
    weight_std: float = 0.02
    x_std: float = 1.0


# The five workloads: tiny parity case, batch-1 decode over 40 independent
# layers, T=4096 prefill with a skewing router bias, the int4 variants of the
# decode and prefill cases, and the prompt-length sweep (seed = T).
TINY_LAYER = Workload("tiny_T16_H256_E16_k2_I64", TINY, T=16, seed=0)
DECODE_BF16 = Workload("decode_T1_H2048_E256_k8_I512_bf16_40layers", QWEN, T=1,
                       seed=1000, n_layers=40)
PREFILL_BF16 = Workload("prefill_T4096_H2048_E256_k8_I512_bf16_bias1.5", QWEN,
                        T=4096, bias_std=1.5, seed=0)
DECODE_INT4 = Workload("decode_T1_H2048_E256_k8_I512_int4g64_40layers", QWEN, T=1,
                       wfmt=WFMT_INT4, seed=2000, n_layers=40)
PREFILL_INT4 = Workload("prefill_T4096_H2048_E256_k8_I512_int4g64_bias1.5", QWEN,
                        T=4096, wfmt=WFMT_INT4, bias_std=1.5, seed=1)
# The affine int4 format of the page's checkpoint (a scale and a bias per 64).
DECODE_INT4_AFFINE = Workload("decode_T1_H2048_E256_k8_I512_int4affg64_40layers", QWEN, T=1,
                              wfmt=WFMT_INT4_AFFINE, seed=3000, n_layers=40)
PREFILL_INT4_AFFINE = Workload("prefill_T4096_H2048_E256_k8_I512_int4affg64_bias1.5", QWEN,
                               T=4096, wfmt=WFMT_INT4_AFFINE, bias_std=1.5, seed=3)
SWEEP_T = (256, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072)


def sweep_workload(T: int) -> Workload:
    return Workload(f"prefill_sweep_T{T}_bf16_bias1.5", QWEN, T=T, bias_std=1.5, seed=T)


_TENSOR_IDS = {
    "x": 1, "router_w": 2, "router_b": 3, "gate_up": 4, "down": 5,
    "sh_gate_up": 6, "sh_down": 7, "sh_gate_w": 8,
}


def _gen(seed: int, name: str, layer: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1009 + layer) * 64 + _TENSOR_IDS[name])
    return g


def _normal_bf16(shape, std, g, device, chunk_rows=None):
    """N(0, std) drawn in fp32 and rounded to bf16 (round-to-nearest-even)."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if chunk_rows is None or shape[0] <= chunk_rows:
        out.copy_(torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std))
        return out
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        sub = (r1 - r0,) + tuple(shape[1:])
        out[r0:r1].copy_(torch.randn(sub, generator=g, device=device,
                                     dtype=torch.float32).mul_(std))
    return out


def pack_int4(codes: torch.Tensor) -> torch.Tensor:
    """Pack signed codes in [-8, 7] (last dim even) two per byte, even index low."""
    c = codes.to(torch.int16) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).to(torch.uint8)


def _int4_affine_weight(shape, std, g, device):
    """Random affine int4 weight: packed codes U{0..15}, |N(0,std)|/7 scales and
    biases -scale * (7.5 + N(0, 0.5)), all per group of 64 along K."""
    *lead, K = shape
    assert K % GROUP == 0
    packed = torch.empty(tuple(lead) + (K // 2,), dtype=torch.uint8, device=device)
    rows = packed.view(-1, K // 2)
    step = 1 << 14
    for r0 in range(0, rows.shape[0], step):
        r1 = min(rows.shape[0], r0 + step)
        codes = torch.randint(0, 16, (r1 - r0, K), generator=g, device=device, dtype=torch.int16)
        rows[r0:r1] = pack_int4(codes)
    gshape = tuple(lead) + (K // GROUP,)
    scale32 = torch.randn(gshape, generator=g, device=device, dtype=torch.float32).abs_().mul_(
        std / 7.0)
    scale = scale32.to(torch.bfloat16)
    z = torch.randn(gshape, generator=g, device=device, dtype=torch.float32).mul_(0.5).add_(7.5)
    bias = (-scale.float() * z).to(torch.bfloat16)
    return packed, scale, bias


def _int4_weight(shape, std, g, device):
    """Random symmetric int4 weight: packed codes U{-7..7} and |N(0,std)|/7 scales."""
    *lead, K = shape
    assert K % GROUP == 0
    packed = torch.empty(tuple(lead) + (K // 2,), dtype=torch.uint8, device=device)
    rows = packed.view(-1, K // 2)
    step = 1 << 14
    flat_n = rows.shape[0]
    for r0 in range(0, flat_n, step):
        r1 = min(flat_n, r0 + step)
        codes = torch.randint(-7, 8, (r1 - r0, K), generator=g, device=device,
                              dtype=torch.int16)
        rows[r0:r1] = pack_int4(codes)
    scale = (torch.randn(tuple(lead) + (K // GROUP,), generator=g, device=device,
                         dtype=torch.float32).abs_().mul_(std / 7.0)).to(torch.bfloat16)
    return packed, scale


def make_x(wl: Workload, layer: int = 0, device="cpu", T: Optional[int] = None) -> torch.Tensor:
    T = wl.T if T is None else T
    return _normal_bf16((T, wl.shape.hidden), wl.x_std, _gen(wl.seed, "x", layer, device),
                        device, chunk_rows=1 << 14)


def make_layer(wl: Workload, layer: int = 0, device="cpu") -> dict:
    """All weights of one MoE layer, as torch tensors on `device`."""
    s = wl.shape
    H, E, I, Is = s.hidden, s.n_experts, s.inter, s.shared_inter
    std = wl.weight_std
    out = {}
    out["router_w"] = _normal_bf16((E, H), std, _gen(wl.seed, "router_w", layer, device), device)
    if wl.bias_std is not None:
        out["router_b"] = torch.randn((E,), generator=_gen(wl.seed, "router_b", layer, device),
                                      device=device, dtype=torch.float32).mul_(wl.bias_std)
    else:
        out["router_b"] = None
    if wl.wfmt == WFMT_BF16:
        out["gate_up"] = _normal_bf16((E, 2 * I, H), std, _gen(wl.seed, "gate_up", layer, device),
                                      device, chunk_rows=8)
        out["down"] = _normal_bf16((E, H, I), std, _gen(wl.seed, "down", layer, device),
                                   device, chunk_rows=16)
        out["sh_gate_up"] = _normal_bf16((2 * Is, H), std,
                                         _gen(wl.seed, "sh_gate_up", layer, device), device)
        out["sh_down"] = _normal_bf16((H, Is), std, _gen(wl.seed, "sh_down", layer, device), device)
        out["gate_up_scale"] = out["down_scale"] = None
        out["sh_gate_up_scale"] = out["sh_down_scale"] = None
    elif wl.wfmt == WFMT_INT4:
        out["gate_up"], out["gate_up_scale"] = _int4_weight(
            (E, 2 * I, H), std, _gen(wl.seed, "gate_up", layer, device), device)
        out["down"], out["down_scale"] = _int4_weight(
            (E, H, I), std, _gen(wl.seed, "down", layer, device), device)
        out["sh_gate_up"], out["sh_gate_up_scale"] = _int4_weight(
            (2 * Is, H), std, _gen(wl.seed, "sh_gate_up", layer, device), device)
        out["sh_down"], out["sh_down_scale"] = _int4_weight(
            (H, Is), std, _gen(wl.seed, "sh_down", layer, device), device)
    elif wl.wfmt == WFMT_INT4_AFFINE:
        for name, shape in (("gate_up", (E, 2 * I, H)), ("down", (E, H, I)),
                            ("sh_gate_up", (2 * Is, H)), ("sh_down", (H, Is))):
            out[name], out[name + "_scale"], out[name + "_bias"] = _int4_affine_weight(
                shape, std, _gen(wl.seed, name, layer, device), device)
    else:
        raise ValueError(wl.wfmt)
    out["sh_gate_w"] = _normal_bf16((H,), std, _gen(wl.seed, "sh_gate_w", layer, device), device)
    return out


def to_numpy(layer: dict) -> dict:
    """Host copies for the oracle: bf16 -> float32 (exact), uint8 stays uint8."""
    out = {}
    for k, v in layer.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.detach().float().cpu().numpy()
        else:
            out[k] = v.detach().cpu().numpy()
    return out


def expert_slice(layer: dict, experts) -> dict:
    """Subset of the routed-expert tensors (host copies), for sampled checks at full size."""
    idx = torch.as_tensor(list(experts), dtype=torch.long, device=layer["gate_up"].device)
    out = dict(layer)
    for k in ("gate_up", "gate_up_scale", "gate_up_bias", "down", "down_scale", "down_bias"):
        if layer.get(k) is not None:
            out[k] = layer[k].index_select(0, idx)
    return out
