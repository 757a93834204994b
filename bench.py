"""Benchmark of the sparse MoE layer on one GB300 (or N replicas).

One step = one prefill pass of the whole layer (router GEMM, top-k, placement:
histogram, scan, block map and scatter, gate/up+SwiGLU and down grouped GEMMs,
combine) over T=4096
synthetic tokens of the Qwen3.6-35B-A3B MoE shape (H=2048, 256 experts, top-8,
I=512, one shared expert, bf16, router bias ~N(0,1.5)), inputs resident in HBM,
L2 flushed between timed steps.  The same JSON line carries the batch-1 decode
latency (40 independent layers, weights far larger than L2, replayed as one
CUDA graph), the roofline of the dominant kernel of each path, the end-to-end
number through the host-buffer entry point, the fp64 CPU oracle timed on this
machine's cores, and the SM clocks seen during the run.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth  # noqa: E402

METRIC = "MoE-layer prefill tokens/s (T=4096) and batch-1 decode µs/layer; % of roofline"
L2_FLUSH_BYTES = 512 << 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi samples every 20 ms on a reader thread, each stamped with the
    host time it arrived; `mark_start` / `mark_end` bracket the timed region
    and `stop` keeps only the samples that fall inside it."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.perf_counter(), line))
        threading.Thread(target=reader, daemon=True).start()
        deadline = time.perf_counter() + 10.0
        while not self.lines and time.perf_counter() < deadline:   # sampling has begun
            time.sleep(0.01)

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        t0 = self.t0 if self.t0 is not None else -1e30
        t1 = self.t1 if self.t1 is not None else 1e30
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in list(self.lines):
            if not (t0 <= ts <= t1 + 0.02):
                continue
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"],
                    "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": float(max(power)),
                "window_s": (t1 - t0) if self.t0 is not None and self.t1 is not None else None}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# the kernels the roofline lines name, from one ncu capture of the current
# kernels (the summaries under profiles/): gate/up 705.0 + 33.8 MB at the
# T=4096 prefill workload, decode layer 57.77 + 0.51 MB (bf16),
# 16.21 + 0.00 MB (symmetric int4) and 17.11 + 0.00 MB (affine int4).
TRAFFIC_BYTES = {"gateup_swiglu_gemm": 738.9e6, "decode_layer": 58.29e6,
                 "decode_layer_int4_sym": 16.21e6, "decode_layer_int4_affine": 17.11e6}


# ------------------------------------------------------------- workload --
def algorithmic(s: moe_synth.Shape, T: int):
    H, E, k, I, Is = s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter
    gateup_flops = 2.0 * H * 2 * I * T * k + 2.0 * H * 2 * Is * T
    down_flops = 2.0 * I * H * T * k + 2.0 * Is * H * T
    router_flops = 2.0 * H * E * T
    return gateup_flops, down_flops, router_flops


def routing_bytes(s: moe_synth.Shape, T: int, k_split: int = 4):
    """Bytes each routing kernel must move at T tokens (what the step reads
    and writes, not what a cache hierarchy adds): router GEMM x, Wr and its
    split-K logit parts; top-k the parts and its outputs (indices, weights,
    per-32-token expert masks); placement the indices and masks in, counts,
    offsets, the two permutation arrays and the block list out, x and the
    shared gate's weights read once, the gates out, and x written k times in
    grouped order."""
    H, E, k = s.hidden, s.n_experts, s.top_k
    nblk = (T + 31) // 32
    x = T * H * 2
    parts = k_split * T * E * 4
    masks = nblk * E * 4
    return {
        "router_gemm": x + E * H * 2 + parts,
        "topk": parts + T * k * 8 + masks,
        "route_place": T * k * 4 + masks + 2 * E * 4 + 2 * T * k * 4 + x + H * 2 + T * 4
        + T * k * H * 2,
        "combine": (T * k + T) * H * 2 + T * k * 8 + T * 4 + x,
    }


def decode_bytes(s: moe_synth.Shape, int4: bool, affine: bool = False):
    H, E, k, I, Is = s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter
    if int4:
        ng = 2 if affine else 1   # scales, and biases for the affine format
        per = lambda rows, K: rows * K // 2 + ng * rows * (K // 64) * 2  # noqa: E731
    else:
        per = lambda rows, K: rows * K * 2  # noqa: E731
    routed_gu = k * per(2 * I, H)
    routed_dn = k * per(H, I)
    shared = per(2 * Is, H) + per(H, Is)
    router = E * H * 2 + H * 2
    return dict(routed_gateup=routed_gu, routed_down=routed_dn, shared=shared, router=router,
                expert_stream=routed_gu + routed_dn + shared,
                total=routed_gu + routed_dn + shared + router + 2 * H * 2)


def run_prefill(ctx, x, y, steps, warmup, flush, stream, clocks=None, prof_steps=20):
    """Times `steps` layer passes (CUDA events around each pass, L2 flushed
    before each), then runs `prof_steps` more passes with the library's
    per-kernel event timing on, so that those events do not sit inside the
    timed passes."""
    for _ in range(warmup):
        ctx.forward_prefill(0, x, y, stream=stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    launches0 = ctx.launch_count
    if clocks is not None:
        clocks.mark_start()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            ctx.forward_prefill(0, x, y, stream=stream)
            ends[i].record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark_end()
    launches = ctx.launch_count - launches0
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ctx.profile(True)
    with torch.cuda.stream(stream):
        for i in range(min(steps, prof_steps)):
            flush.zero_()
            ctx.forward_prefill(0, x, y, stream=stream)
    torch.cuda.synchronize()
    prof = ctx.profile_read()
    ctx.profile(False)
    return float(np.sum(ms)), prof, launches


def run_prefill_e2e(ctx, x_h, y_h, steps, warmup, flush, stream):
    """Wall time (ms, CUDA events on `stream`) of `steps` back-to-back calls
    from pinned host buffers: each call's input and output copies run on the
    library's copy streams, overlapping the neighbouring calls' compute, and
    the stream waits for the last output copy.  (No L2 flush: the inputs come
    from host memory, and one step streams 0.9 GB of weights, 7 times L2.)"""
    for _ in range(max(1, warmup // 2)):
        ctx.forward_prefill_host(0, x_h, y_h, stream=stream)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            ctx.forward_prefill_host(0, x_h, y_h, stream=stream)
        end.record(stream)
    torch.cuda.synchronize()
    return float(start.elapsed_time(end))


def bench_prefill_int4(args, dev, stream, flush, tf_burst, wl=moe_synth.PREFILL_INT4):
    """An int4 prefill workload at T=4096 (symmetric, or affine with a bias
    per group): weights are dequantised tile by tile inside the grouped GEMMs."""
    from sparse_moe_gb300 import MoEContext
    s = wl.shape
    ctx = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, n_layers=1,
                     max_chunk_rows=4096, wfmt=wl.wfmt, device=dev.index)
    w = moe_synth.make_layer(wl, device=dev)
    ctx.load_weights(0, w)
    x = moe_synth.make_x(wl, device=dev)
    y = torch.empty_like(x)
    steps = max(5, args.steps // 2)
    total_ms, prof, launches = run_prefill(ctx, x, y, steps, args.warmup, flush, stream)
    gu_f, dn_f, _ = algorithmic(s, wl.T)
    kern = {k: {"launches": v[0], "avg_us": v[1] * 1e3 / max(1, v[0])} for k, v in prof.items()}
    gu_us = kern.get("gateup_swiglu_gemm", {}).get("avg_us", float("nan"))
    dn_us = kern.get("down_gemm", {}).get("avg_us", float("nan"))
    out = {"workload": wl.name, "value": wl.T * steps / (total_ms * 1e-3), "unit": "tokens/s",
           "ms_per_step": total_ms / steps, "steps": steps,
           "gateup_TFLOPs": gu_f / (gu_us * 1e-6) / 1e12,
           "gateup_frac_of_bf16_peak": gu_f / (gu_us * 1e-6) / 1e12 / tf_burst,
           "down_TFLOPs": dn_f / (dn_us * 1e-6) / 1e12, "kernels_us": kern,
           "gpu_launches": launches}
    ctx.close()
    del w
    torch.cuda.empty_cache()
    return out


def _time_steps(fn, steps, warmup, flush, stream):
    """ms per call of fn() (one layer pass), CUDA events around each call on
    `stream`, L2 flushed before each."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in ev]))


def bench_ablations(args, dev, stream, flush):
    """The page's prefill ablations on GB300, each undoing one mechanism of the
    layer at the prompt length the page measured it at: routing kept on the GPU
    vs a host that waits for the routing before the grouped GEMMs ("Keep
    expert routing on the GPU", 512 tokens); tile shape from the expert's load
    vs a fixed tile ("Match tile size to expert load", 2K tokens: every block
    at the full 256-row MMA N, and blocks of at most 16 rows); weights expanded
    inside the GEMMs vs by a separate kernel into a bf16/fp16 array that the
    GEMMs read back ("Dequantize weights during matrix multiplication", 512
    tokens, the affine int4 format).  Layer time here, not the page's
    end-to-end prefill."""
    from sparse_moe_gb300 import MoEContext, dequant_int4, with_f16_down
    steps = max(10, min(args.steps, 40))
    out = {}

    def layer_ms(wl, env=None):
        old = {k: os.environ.get(k) for k in (env or {})}
        os.environ.update(env or {})
        try:
            s = wl.shape
            ctx = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter,
                             max_chunk_rows=4096, wfmt=wl.wfmt, device=dev.index)
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        w = moe_synth.make_layer(wl, device=dev)
        ctx.load_weights(0, with_f16_down(w) if wl.wfmt == moe_synth.WFMT_BF16 else w)
        x = moe_synth.make_x(wl, device=dev)
        y = torch.empty_like(x)
        ms = _time_steps(lambda: ctx.forward_prefill(0, x, y, stream=stream), steps, args.warmup,
                         flush, stream)
        ctx.close()
        return ms

    def entry(base_ms, abl_ms, what, page):
        return {"layer_ms": base_ms, "ablated_layer_ms": abl_ms, "ablated": what,
                "gain_of_mechanism": abl_ms / base_ms - 1.0, "page_end_to_end_gain": page}

    wl512 = moe_synth.sweep_workload(512)
    base512 = layer_ms(wl512)
    out["gpu_routing_vs_host_sync_T512"] = entry(
        base512, layer_ms(wl512, {"MOE_ABLATE_HOST_ROUTING": "1"}),
        "host waits for the routing (block count read back) before the grouped GEMMs", 0.89)
    wl2k = moe_synth.sweep_workload(2048)
    base2k = layer_ms(wl2k)
    out["adaptive_tile_vs_fixed_n256_T2048"] = entry(
        base2k, layer_ms(wl2k, {"MOE_ABLATE_TILE": "fixed256"}),
        "every block runs the full 256-row MMA N", 0.132)
    out["adaptive_tile_vs_16_row_blocks_T2048"] = entry(
        base2k, layer_ms(wl2k, {"MOE_ABLATE_TILE": "rows16"}),
        "blocks of at most 16 rows (the weights re-read per 16 rows; MMA N 32)", 0.132)

    # fused vs separate dequantisation, affine int4 at T=512
    wl4 = moe_synth.Workload("ablation_dequant_T512_int4affg64_bias1.5", moe_synth.QWEN, T=512,
                             wfmt=moe_synth.WFMT_INT4_AFFINE, bias_std=1.5, seed=512)
    fused = layer_ms(wl4)
    s4 = wl4.shape
    w4 = moe_synth.make_layer(wl4, device=dev)
    ctxb = MoEContext(s4.hidden, s4.n_experts, s4.top_k, s4.inter, s4.shared_inter,
                      max_chunk_rows=4096, device=dev.index)
    exp = {}
    for name in ("gate_up", "sh_gate_up", "down", "sh_down"):
        exp[name] = dequant_int4(w4[name], w4[name + "_scale"], w4[name + "_bias"])
    for name in ("down", "sh_down"):
        exp[name + "_f16"] = dequant_int4(w4[name], w4[name + "_scale"], w4[name + "_bias"],
                                          out_dtype=torch.float16)
    ctxb.load_weights(0, {"router_w": w4["router_w"], "router_b": w4["router_b"],
                          "sh_gate_w": w4["sh_gate_w"], **exp})
    x4 = moe_synth.make_x(wl4, device=dev)
    y4 = torch.empty_like(x4)
    from sparse_moe_gb300 import library, _abi
    lib = library()

    def separate():
        # expand every expert's weights, then run the bf16/fp16 layer on them
        h = ctypes.c_void_p(stream.cuda_stream)
        for name, dst in (("gate_up", exp["gate_up"]), ("sh_gate_up", exp["sh_gate_up"]),
                          ("down", exp["down_f16"]), ("sh_down", exp["sh_down_f16"])):
            c = w4[name]
            K = c.shape[-1] * 2
            st = lib.moe_dequant_int4(ctypes.c_void_p(c.data_ptr()),
                                      ctypes.c_void_p(w4[name + "_scale"].data_ptr()),
                                      ctypes.c_void_p(w4[name + "_bias"].data_ptr()),
                                      ctypes.c_void_p(dst.data_ptr()), c.numel() * 2 // K, K,
                                      _abi.MOE_W_INT4_AFFINE_G64,
                                      int(dst.dtype == torch.float16), h)
            assert st == 0
        ctxb.forward_prefill(0, x4, y4, stream=stream)

    out["fused_vs_separate_dequant_T512_int4_affine"] = entry(
        fused, _time_steps(separate, steps, args.warmup, flush, stream),
        "a separate kernel expands all expert weights (bf16 gate/up, fp16 down) that the "
        "bf16/fp16 GEMMs then read", 0.774)
    ctxb.close()
    del w4, exp
    torch.cuda.empty_cache()
    return out


def _sweep_point(T, dev, stream, flush, tf_burst, hbm, steps):
    """One prefill-path point of the sweep workload at T tokens (seed = T,
    router bias 1.5, 4096-row chunks)."""
    from sparse_moe_gb300 import MoEContext, with_f16_down
    wl = moe_synth.sweep_workload(T)
    s = wl.shape
    ctx = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, n_layers=1,
                     max_chunk_rows=4096, device=dev.index)
    w = moe_synth.make_layer(wl, device=dev)
    ctx.load_weights(0, with_f16_down(w))
    x = moe_synth.make_x(wl, device=dev)
    y = torch.empty_like(x)
    touched = 0
    for c0 in range(0, T, 4096):
        cnt = ctx.route(0, x[c0:c0 + 4096])["counts"]
        touched += int((cnt > 0).sum().item()) + 1   # + the shared expert
    for _ in range(2):
        ctx.forward_prefill(0, x, y, stream=stream)
    torch.cuda.synchronize()
    a = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    b = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.zero_()
            a[i].record(stream)
            ctx.forward_prefill(0, x, y, stream=stream)
            b[i].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in zip(a, b)]))
    gu_f, dn_f, rt_f = algorithmic(s, T)
    wbytes = touched * 3 * s.inter * s.hidden * 2 + s.n_experts * s.hidden * 2
    ctx.close()
    del w, x, y
    torch.cuda.empty_cache()
    return {"T": T, "tokens_per_s": T / (ms * 1e-3), "ms": ms, "chunks": (T + 4095) // 4096,
            "tensor_frac": (gu_f + dn_f + rt_f) / (ms * 1e-3) / 1e12 / tf_burst,
            "hbm_frac_expert_weights": wbytes / (ms * 1e-3) / 1e9 / hbm,
            "experts_touched_per_chunk": touched / ((T + 4095) // 4096)}


def bench_sweep(args, dev, stream, flush, tf_burst, hbm):
    """Prefill over the prompt-length sweep (T = 256 .. 128K, seed = T, router
    bias 1.5), long prompts in 4096-row chunks: tokens/s, and the fraction of
    the tensor peak (algorithmic FLOPs) and of the HBM peak (expert weights
    the chunks touch, each counted once per chunk) that the layer reaches."""
    return [_sweep_point(T, dev, stream, flush, tf_burst, hbm, 3 if T >= 32768 else 5)
            for T in moe_synth.SWEEP_T]


def _rows_point(T, dev, stream, flush, hbm, steps):
    """moe_forward_rows on the sweep workload's first T rows: layer time and
    the HBM fraction over the weights it must read (router, shared expert and
    the union of the selected experts, each once)."""
    from sparse_moe_gb300 import MoEContext
    wl = moe_synth.sweep_workload(T)
    s = wl.shape
    ctx = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, n_layers=1,
                     max_chunk_rows=16, device=dev.index)
    w = moe_synth.make_layer(wl, device=dev)
    ctx.load_weights(0, w)
    x = moe_synth.make_x(wl, device=dev)
    y = torch.empty_like(x)
    ctx.forward_rows(0, x, y, stream=stream)
    torch.cuda.synchronize()
    union = int(torch.unique(ctx.rows_routing(T)["topk_idx"]).numel())
    for _ in range(3):
        ctx.forward_rows(0, x, y, stream=stream)
    torch.cuda.synchronize()
    a = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    b = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.zero_()
            a[i].record(stream)
            ctx.forward_rows(0, x, y, stream=stream)
            b[i].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in zip(a, b)]))
    wbytes = (union + 1) * 3 * s.inter * s.hidden * 2 + s.n_experts * s.hidden * 2 + s.hidden * 2
    ctx.close()
    del w, x, y
    torch.cuda.empty_cache()
    return {"rows_ms": ms, "rows_hbm_frac": wbytes / (ms * 1e-3) / 1e9 / hbm, "union_experts": union,
            "rows_gpu_launches": 1}


def bench_small_m(args, dev, stream, flush, tf_burst, hbm):
    """Small row counts (2 - 16 rows, the page's speculative-verification
    shapes): the prefill path (grouped GEMMs at MMA N = 32) and the
    decode-style rows path (moe_forward_rows), each against the HBM time of
    the weights the rows need."""
    out = []
    for T in (2, 4, 8, 16):
        pt = _sweep_point(T, dev, stream, flush, tf_burst, hbm, 20)
        pt.update(_rows_point(T, dev, stream, flush, hbm, 20))
        out.append(pt)
    return out


def bench_decode(args, dev, stream, hbm, int4=None, wl=None):
    """40 independent decode layers replayed as one CUDA graph."""
    from sparse_moe_gb300 import MoEContext
    if wl is None:
        if int4 is None:
            int4 = args.decode_int4
        wl = moe_synth.DECODE_INT4 if int4 else moe_synth.DECODE_BF16
    int4 = wl.wfmt != moe_synth.WFMT_BF16
    s = wl.shape
    L = args.decode_layers or wl.n_layers
    ctx = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, n_layers=L,
                     max_chunk_rows=16, wfmt=wl.wfmt, device=dev.index)
    layers = []
    for l in range(L):
        w = moe_synth.make_layer(wl, layer=l, device=dev)
        ctx.load_weights(l, w)
        layers.append(w)
    xs = torch.stack([moe_synth.make_x(wl, layer=l, device=dev)[0] for l in range(L)])
    ys = torch.empty_like(xs)
    x_h = xs[0:1].cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    # eager warm-up, then a profiled eager pass for per-kernel times
    for l in range(L):
        ctx.forward_decode(l, xs[l:l + 1], ys[l:l + 1], stream=stream)
    torch.cuda.synchronize()
    ctx.profile(True)
    for _ in range(2):
        for l in range(L):
            ctx.forward_decode(l, xs[l:l + 1], ys[l:l + 1], stream=stream)
    torch.cuda.synchronize()
    # the expert-weight stream on its own: phase B of single launches, whose
    # CTAs stamp the global timer at its start and end while profiling is on
    phases = []
    for l in range(min(L, 10)):
        ctx.forward_decode(l, xs[l:l + 1], ys[l:l + 1], stream=stream)
        torch.cuda.synchronize()
        phases.append(ctx.decode_phase_read())
    prof = ctx.profile_read()
    ctx.profile(False)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                ctx.forward_decode(l, xs[l:l + 1], ys[l:l + 1], stream=stream)
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    reps = max(5, args.steps)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = ctx.launch_count
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us_layer = a.elapsed_time(b) * 1e3 / (reps * L)
    # the same L layers in one persistent launch (moe_forward_decode_layers):
    # a grid barrier between layers instead of a kernel boundary
    for _ in range(max(3, args.warmup)):
        ctx.forward_decode_layers(0, xs, ys, stream=stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            ctx.forward_decode_layers(0, xs, ys, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    us_layer_ml = a.elapsed_time(b) * 1e3 / (reps * L)
    # end to end from host memory: one token per layer call, copies included
    for _ in range(3):
        ctx.forward_decode_host(0, x_h, y_h, stream=stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    n_e2e = 200
    for i in range(n_e2e):
        ctx.forward_decode_host(i % L, x_h, y_h, stream=stream)
        stream.synchronize()
    e2e_us = (time.perf_counter() - t0) * 1e6 / n_e2e
    nb = decode_bytes(s, int4, affine=wl.wfmt == moe_synth.WFMT_INT4_AFFINE)
    b_bytes = nb["routed_gateup"] + nb["routed_down"]
    win = float(np.median([ph["window_us"] for ph in phases]))
    phase_b = {"bytes": b_bytes, "window_us": win,
               "median_cta_us": float(np.median([ph["median_us"] for ph in phases])),
               "GBps": b_bytes / (win * 1e-6) / 1e9,
               "frac_of_hbm": b_bytes / (win * 1e-6) / 1e9 / hbm,
               "how": "phase B of single eager launches (the k routed experts' gate/up rows, "
                      "their output-projection rows bulk-copied alongside), global-timer "
                      "stamps in every CTA, first start to last end; median of "
                      f"{len(phases)} launches"}
    lay = prof.get("decode_layer", (1, float("nan")))
    lay_us = lay[1] * 1e3 / max(1, lay[0])
    # one launch per layer: its average duration in the timed graph replays
    achieved = nb["total"] / (us_layer * 1e-6) / 1e9
    out = {
        "workload": wl.name, "value": us_layer, "unit": "us/layer",
        "tokens_per_s": 1e6 / (us_layer * L), "layers": L, "graph_replays": reps,
        "expert_stream_GBps": nb["expert_stream"] / (us_layer * 1e-6) / 1e9,
        "expert_stream_frac_of_hbm": nb["expert_stream"] / (us_layer * 1e-6) / 1e9 / hbm,
        "expert_stream_phase_b": phase_b,
        "bytes_per_layer": nb["total"],
        "roofline": {"kernel": "decode_layer", "bound": "hbm", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": (TRAFFIC_BYTES["decode_layer"] if not int4 else
                                 TRAFFIC_BYTES["decode_layer_int4_sym"]
                                 if wl.wfmt == moe_synth.WFMT_INT4 else
                                 TRAFFIC_BYTES["decode_layer_int4_affine"]),
                     "algorithmic_bytes_per_launch": nb["total"],
                     "launch_us_timed": us_layer,
                     "timing": "graph replays of L layers, CUDA events on the launch stream; "
                               "launch_us_eager: events around single eager launches",
                     "launch_us_eager": lay_us},
        "multi_layer": {
            "value": us_layer_ml, "unit": "us/layer",
            "how": f"moe_forward_decode_layers: all {L} layers in one persistent launch, "
                   "grid barrier between layers, next layer's shared weights fetched ahead",
            "roofline": {"kernel": "decode_layers", "bound": "hbm",
                         "achieved": nb["total"] / (us_layer_ml * 1e-6) / 1e9, "peak": hbm,
                         "unit": "GB/s",
                         "frac": nb["total"] / (us_layer_ml * 1e-6) / 1e9 / hbm}},
        "kernels_eager_us": {k: v[1] * 1e3 / max(1, v[0]) for k, v in prof.items()},
        "e2e": {"value": e2e_us, "unit": "us/token (one layer, host buffers, synchronous)",
                "h2d_bytes_per_step": s.hidden * 2, "d2h_bytes_per_step": s.hidden * 2},
        "gpu_launches_per_layer": (ctx.launch_count - launches0) // max(1, reps * L) or 1,
    }
    del g
    ctx.close()
    del layers
    torch.cuda.empty_cache()
    return out


def cpu_baseline_prefill(x_cpu, w_dev, k, min_seconds=10.0, max_passes=32):
    """The fp64 oracle, as it stands, over the whole prefill workload, repeated
    until about `min_seconds` of CPU work have been timed."""
    from oracle import moe_oracle as orc
    layer = moe_synth.to_numpy(w_dev)
    xs = x_cpu.float().numpy()
    t0 = time.perf_counter()
    passes = 0
    while passes < max_passes and (passes == 0 or time.perf_counter() - t0 < min_seconds):
        orc.moe_layer(xs, layer, k)
        passes += 1
    dt = time.perf_counter() - t0
    T = xs.shape[0]
    return {"value": T * passes / dt, "unit": "tokens/s", "cores": os.cpu_count(),
            "threads": torch.get_num_threads(), "kind": "oracle",
            "sample": f"fp64 oracle (router, top-k, grouping, all experts, shared expert) over all "
                      f"{T} tokens of the workload, {passes} pass(es), {dt:.1f} s",
            "seconds": dt}


def cpu_oracle_worker(threads: int) -> dict:
    """The fp64 oracle, as it stands, on bounded samples of each configured
    workload, timed in this process (started with the BLAS thread count set
    to `threads`).  Weights are regenerated on the host from the workloads'
    seeds (the host generator draws other numbers than the device one; the
    shapes, distributions and routing skew are the same)."""
    from oracle import moe_oracle as orc
    out = {"threads": threads}

    def timed(fn, min_s=0.5, max_reps=50):
        fn()   # first pass: warm caches and allocations
        t0 = time.perf_counter()
        n = 0
        while n < max_reps and (n == 0 or time.perf_counter() - t0 < min_s):
            fn()
            n += 1
        return (time.perf_counter() - t0) / n

    def host(wl):
        return moe_synth.to_numpy(moe_synth.make_layer(wl, device="cpu")), \
            moe_synth.make_x(wl, device="cpu").float().numpy()

    w, x = host(moe_synth.TINY_LAYER)
    dt = timed(lambda: orc.moe_layer(x, w, moe_synth.TINY.top_k))
    out["tiny_T16"] = {"tokens_per_s": 16 / dt, "sample": "all 16 tokens"}
    wl = moe_synth.PREFILL_BF16
    w, x = host(wl)
    k = wl.shape.top_k
    dt = timed(lambda: orc.moe_layer(x[:1], w, k))
    out["decode_bf16_T1"] = {"us_per_layer": dt * 1e6, "tokens_per_s_40_layers": 1.0 / (40 * dt),
                             "sample": "one token through one layer of the prefill workload's "
                                       "weights (8 routed experts + shared; the decode "
                                       "workload's shapes)"}
    S = 512
    dt = timed(lambda: orc.moe_layer(x[:S], w, k), min_s=0.0, max_reps=1)
    out["prefill_bf16_T4096"] = {"tokens_per_s": S / dt,
                                 "sample": f"first {S} tokens of the T=4096 workload"}
    lens = {}
    per_tok = None
    for T in moe_synth.SWEEP_T:
        if T <= 512:
            xs = moe_synth.make_x(moe_synth.sweep_workload(T), device="cpu").float().numpy()
            dts = timed(lambda: orc.moe_layer(xs, w, k), min_s=0.0, max_reps=1)
            per_tok = dts / T
            lens[str(T)] = {"seconds": dts, "tokens_per_s": T / dts, "how": "measured, all rows"}
        else:
            lens[str(T)] = {"seconds": T * per_tok, "tokens_per_s": 1.0 / per_tok,
                            "how": "extrapolated from the T=512 measurement (cost per token)"}
    out["prompt_sweep"] = lens
    del w
    wl4 = moe_synth.PREFILL_INT4
    w4, x4 = host(wl4)
    dt = timed(lambda: orc.moe_layer(x4[:1], w4, k))
    out["decode_int4_T1"] = {"us_per_layer": dt * 1e6, "sample": "one token, symmetric int4 G64"}
    S = 256
    dt = timed(lambda: orc.moe_layer(x4[:S], w4, k), min_s=0.0, max_reps=1)
    out["prefill_int4_T4096"] = {"tokens_per_s": S / dt,
                                 "sample": f"first {S} tokens of the int4 T=4096 workload"}
    return out


def cpu_baselines_by_threads() -> dict:
    """cpu_oracle_worker with one thread and with all host cores, each in a
    subprocess whose BLAS thread count is fixed before numpy loads."""
    res = {}
    for threads in (1, os.cpu_count() or 1):
        env = dict(os.environ)
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[v] = str(threads)
        env["CUDA_VISIBLE_DEVICES"] = ""
        try:
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-worker",
                                str(threads)], env=env, capture_output=True, text=True,
                               timeout=600)
            res[f"threads_{threads}"] = json.loads(r.stdout.strip().splitlines()[-1])
        except Exception as e:   # reported, not fatal: the GPU numbers stand
            res[f"threads_{threads}"] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return res


def main_reference(args):
    """The oracle as the reference arm, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from oracle import moe_oracle as orc
    wl = moe_synth.PREFILL_BF16
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = moe_synth.to_numpy(moe_synth.make_layer(wl, device=dev))
    x = moe_synth.make_x(wl, device=dev).float().cpu().numpy()
    S = args.ref_sample
    # keep the whole run within a few minutes: shrink the per-step sample if
    # one step of S tokens would make K + W steps take longer than ~150 s
    t0 = time.perf_counter()
    orc.moe_layer(x[:S], w, wl.shape.top_k)
    t_step = time.perf_counter() - t0
    while S > 16 and t_step * (args.steps + args.warmup) > 150.0:
        S //= 2
        t0 = time.perf_counter()
        orc.moe_layer(x[:S], w, wl.shape.top_k)
        t_step = time.perf_counter() - t0
    for i in range(args.warmup):
        orc.moe_layer(x[(i * S) % wl.T:(i * S) % wl.T + S], w, wl.shape.top_k)
    t0 = time.perf_counter()
    for i in range(args.steps):
        s0 = (i * S) % wl.T
        orc.moe_layer(x[s0:s0 + S], w, wl.shape.top_k)
    dt = time.perf_counter() - t0
    value = args.steps * S / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "sample_tokens_per_step": S},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{S} consecutive tokens of the T={wl.T} workload per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def replicas_rate(total_ms, world, tokens_per_step, steps, device):
    """Whole-job rate of `world` independent replicas: the slowest rank's
    timed region (max over ranks) and all ranks' tokens over it.  Returns
    (max total ms, tokens/s)."""
    if world > 1:
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, world * tokens_per_step * steps / (total_ms * 1e-3)


def main(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm, tf_burst, tf_sust, peak_src = peaks()

    if args.skip_prefill:
        # decode only (a diagnostic mode: e.g. a small decode case for a profiler)
        out = bench_decode(args, dev, torch.cuda.Stream(device=dev), hbm,
                           wl=moe_synth.DECODE_INT4_AFFINE if args.decode_affine else None)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": out["value"], "unit": out["unit"],
                              "n_gpus": world, "higher_is_better": False, "decode": out}))
        return 0

    from sparse_moe_gb300 import MoEContext, with_f16_down
    wl = moe_synth.PREFILL_BF16
    s = wl.shape
    ctx = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, n_layers=1,
                     max_chunk_rows=4096, device=local)
    w = moe_synth.make_layer(wl, device=dev)
    # fp16 copies of the down weights, made once at load (outside the timed
    # region): the down GEMM then skips its in-shared-memory conversion
    ctx.load_weights(0, with_f16_down(w))
    x = moe_synth.make_x(wl, device=dev)
    y = torch.empty_like(x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total_ms, prof, launches = run_prefill(ctx, x, y, args.steps, args.warmup, flush, stream,
                                           clocks)
    torch.cuda.synchronize()
    total_ms, value = replicas_rate(total_ms, world, wl.T, args.steps, dev)
    clk = clocks.stop()
    ms_step = total_ms / args.steps

    gu_f, dn_f, rt_f = algorithmic(s, wl.T)
    kern = {k: {"launches": v[0], "avg_us": v[1] * 1e3 / max(1, v[0])} for k, v in prof.items()}
    # achieved bandwidth of the HBM/latency-bound kernels (algorithmic bytes
    # per launch over the launch's CUDA-event time)
    for name, nbytes in routing_bytes(s, wl.T).items():
        if name in kern:
            kern[name]["algorithmic_bytes"] = nbytes
            kern[name]["achieved_GBps"] = nbytes / (kern[name]["avg_us"] * 1e-6) / 1e9
            kern[name]["frac_of_hbm"] = kern[name]["achieved_GBps"] / hbm
    gu_us = kern.get("gateup_swiglu_gemm", {}).get("avg_us", float("nan"))
    dn_us = kern.get("down_gemm", {}).get("avg_us", float("nan"))
    achieved = gu_f / (gu_us * 1e-6) / 1e12
    roofline = {"kernel": "gateup_swiglu_gemm", "bound": "tensor", "achieved": achieved,
                "peak": tf_burst, "unit": "TFLOP/s", "frac": achieved / tf_burst,
                "traffic": TRAFFIC_BYTES["gateup_swiglu_gemm"],
                "peak_source": f"{peak_src} bf16 burst",
                "timing": "CUDA events around each launch on the launch stream, over passes "
                          "run right after the timed passes (L2 flushed before each)",
                "algorithmic_flops_per_launch": gu_f,
                "down_gemm_TFLOPs": dn_f / (dn_us * 1e-6) / 1e12,
                "grouped_gemms_frac": (gu_f + dn_f) / ((gu_us + dn_us) * 1e-6) / 1e12 / tf_burst}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "hidden": s.hidden, "experts": s.n_experts,
                   "top_k": s.top_k, "inter": s.inter, "shared_inter": s.shared_inter,
                   "router_bias_std": wl.bias_std, "parallelism": f"replicas{world}",
                   "down_weights": "bf16 plus fp16 copies made once at load",
                   "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)"},
        "roofline": roofline,
        "kernels_us": kern,
        "gpu_launches": launches,
        "clocks": clk,
    }

    if rank == 0 and not args.skip_int4:
        # the same layer with only the bf16 down weights (no fp16 copies): the
        # down GEMM then converts each weight tile in shared memory
        ctx_b = MoEContext(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, n_layers=1,
                           max_chunk_rows=4096, device=local)
        ctx_b.load_weights(0, w)
        steps_b = max(5, args.steps // 4)
        tot_b, prof_b, _ = run_prefill(ctx_b, x, y, steps_b, args.warmup, flush, stream)
        dn_b = prof_b.get("down_gemm", (1, float("nan")))
        line["prefill_bf16_down_only"] = {
            "value": wl.T * steps_b / (tot_b * 1e-3), "unit": "tokens/s",
            "ms_per_step": tot_b / steps_b, "steps": steps_b,
            "down_gemm_us": dn_b[1] * 1e3 / max(1, dn_b[0]),
            "how": "bf16 down weights only, converted to fp16 tile by tile in the GEMM"}
        ctx_b.close()
    if rank == 0 and not args.skip_e2e:
        x_h = x.cpu().pin_memory()
        y_h = torch.empty_like(x_h).pin_memory()
        e2e_ms = run_prefill_e2e(ctx, x_h, y_h, args.steps, args.warmup, flush, stream)
        line["e2e"] = {"value": wl.T * args.steps / (e2e_ms * 1e-3), "unit": "tokens/s",
                       "h2d_bytes_per_step": wl.T * s.hidden * 2,
                       "d2h_bytes_per_step": wl.T * s.hidden * 2,
                       "timing": "wall time of the timed steps as back-to-back "
                                 "moe_forward_prefill_host calls (pinned host buffers)"}
    if rank == 0 and not args.skip_decode:
        line["decode"] = bench_decode(args, dev, stream, hbm)
    if rank == 0 and not args.skip_sweep:
        line["sweep"] = bench_sweep(args, dev, stream, flush, tf_burst, hbm)
        line["small_m"] = bench_small_m(args, dev, stream, flush, tf_burst, hbm)
    if rank == 0 and not args.skip_ablations:
        line["ablations"] = bench_ablations(args, dev, stream, flush)
    if rank == 0 and not args.skip_int4:
        line["prefill_int4"] = bench_prefill_int4(args, dev, stream, flush, tf_burst)
        line["prefill_int4_affine"] = bench_prefill_int4(args, dev, stream, flush, tf_burst,
                                                         wl=moe_synth.PREFILL_INT4_AFFINE)
        if not args.skip_decode and not args.decode_int4:
            line["decode_int4"] = bench_decode(args, dev, stream, hbm, int4=True)
            line["decode_int4_affine"] = bench_decode(args, dev, stream, hbm,
                                                      wl=moe_synth.DECODE_INT4_AFFINE)
    if rank == 0 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline_prefill(x.cpu(), w, s.top_k)
        if not args.skip_cpu_configs:
            line["cpu_baseline"]["per_config"] = cpu_baselines_by_threads()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-sample", type=int, default=128,
                    help="tokens per step of the reference arm (the oracle on the host cores)")
    ap.add_argument("--decode-int4", action="store_true")
    ap.add_argument("--decode-affine", action="store_true",
                    help="with --skip-prefill: the affine int4 decode workload")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-sweep", action="store_true",
                    help="skip the prompt-length sweep (T = 256 .. 128K)")
    ap.add_argument("--skip-ablations", action="store_true",
                    help="skip the ablations (GPU routing, tile shape, fused dequantisation)")
    ap.add_argument("--skip-int4", action="store_true",
                    help="skip the int4 prefill and decode measurements")
    ap.add_argument("--skip-prefill", action="store_true",
                    help="decode measurements only (diagnostic; not the benchmark line)")
    ap.add_argument("--decode-layers", type=int, default=0,
                    help="layers in the decode graph (default: the workload's 40)")
    ap.add_argument("--cpu-oracle-worker", type=int, default=0,
                    help=argparse.SUPPRESS)   # internal: one thread setting of the CPU baseline
    ap.add_argument("--skip-cpu-configs", action="store_true",
                    help="skip the per-configuration oracle timings (1 thread and all cores)")
    a = ap.parse_args()
    if a.cpu_oracle_worker:
        print(json.dumps(cpu_oracle_worker(a.cpu_oracle_worker)))
        sys.exit(0)
    if a.warmup < 3 and a.impl == "ours":
        a.warmup = 3
    sys.exit(main_reference(a) if a.impl == "reference" else main(a))
