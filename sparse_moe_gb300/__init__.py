"""GB300 (sm_103a) sparse mixture-of-experts layer.

A thin Python binding over the C ABI in include/sparse_moe.h.  Every step of
the layer runs in the library's CUDA kernels; this module only marshals
arguments.  PyTorch supplies device memory and the current stream.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _abi

__all__ = ["MoEError", "MoEContext", "library", "WFMT", "convert_bf16_to_f16",
           "with_f16_down", "dequant_int4"]

WFMT = {"bf16": _abi.MOE_W_BF16, "int4_sym_g64": _abi.MOE_W_INT4_SYM_G64,
        "int4_affine_g64": _abi.MOE_W_INT4_AFFINE_G64}


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


def library():
    """The loaded native library (built in-tree on first use)."""
    return _abi.load()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def convert_bf16_to_f16(src: torch.Tensor, stream=None) -> torch.Tensor:
    """fp16 copy of a contiguous bf16 CUDA tensor, written by the library's
    conversion kernel (round to nearest even)."""
    if src.dtype != torch.bfloat16 or not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous bf16 CUDA tensor")
    dst = torch.empty(src.shape, dtype=torch.float16, device=src.device)
    st = library().moe_convert_bf16_to_f16(_ptr(src), _ptr(dst), src.numel(),
                                           _stream_handle(stream, src.device))
    if st != 0:
        raise MoEError(st, "moe_convert_bf16_to_f16")
    return dst


def dequant_int4(codes: torch.Tensor, scale: torch.Tensor, bias: Optional[torch.Tensor] = None,
                 out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """Expanded copy of int4 weights (codes uint8 [..., K/2], bf16 scale and,
    for the affine format, bias [..., K/64]) in bf16 or fp16, rounded as the
    grouped GEMMs round them; written by the library's kernel."""
    K = codes.shape[-1] * 2
    rows = codes.numel() * 2 // K
    dst = torch.empty(tuple(codes.shape[:-1]) + (K,), dtype=out_dtype, device=codes.device)
    fmt = _abi.MOE_W_INT4_AFFINE_G64 if bias is not None else _abi.MOE_W_INT4_SYM_G64
    st = library().moe_dequant_int4(_ptr(codes), _ptr(scale), _ptr(bias), _ptr(dst), rows, K, fmt,
                                    int(out_dtype == torch.float16),
                                    _stream_handle(stream, codes.device))
    if st != 0:
        raise MoEError(st, "moe_dequant_int4")
    return dst


def with_f16_down(w: dict, stream=None) -> dict:
    """`w` plus the optional fp16 copies of the bf16 down projections
    (down_f16, sh_down_f16) that let the prefill down GEMM skip its in-kernel
    weight conversion."""
    out = dict(w)
    out["down_f16"] = convert_bf16_to_f16(w["down"], stream)
    out["sh_down_f16"] = convert_bf16_to_f16(w["sh_down"], stream)
    return out


class MoEContext:
    """One layer shape, `n_layers` weight slots, and the workspace they share."""

    def __init__(self, hidden: int, n_experts: int, top_k: int, inter: int, shared_inter: int,
                 n_layers: int = 1, max_chunk_rows: int = 4096, wfmt: str = "bf16",
                 device: int = 0):
        self.lib = library()
        self.cfg = _abi.MoeConfig(hidden, n_experts, top_k, inter, shared_inter, n_layers,
                                  max_chunk_rows, WFMT[wfmt])
        self.hidden, self.n_experts, self.top_k = hidden, n_experts, top_k
        self.inter, self.shared_inter = inter, shared_inter
        self.max_chunk_rows = max_chunk_rows
        self.wfmt = wfmt
        self.device = torch.device("cuda", device)
        nbytes = ctypes.c_size_t()
        self._check(self.lib.moe_workspace_size(ctypes.byref(self.cfg), ctypes.byref(nbytes)),
                    "moe_workspace_size", ctx=False)
        self.workspace = torch.empty(nbytes.value + 256, dtype=torch.uint8, device=self.device)
        base = self.workspace.data_ptr()
        self._ws_ptr = (base + 255) // 256 * 256
        h = ctypes.c_void_p()
        self._check(self.lib.moe_ctx_create(ctypes.byref(self.cfg), device,
                                            ctypes.c_void_p(self._ws_ptr),
                                            ctypes.c_size_t(nbytes.value), ctypes.byref(h)),
                    "moe_ctx_create", ctx=False)
        self.handle = h
        self._weights = {}

    # ------------------------------------------------------------ helpers --
    def _check(self, st: int, what: str, ctx: bool = True):
        if st != _abi.MOE_OK:
            detail = ""
            if ctx and getattr(self, "handle", None):
                detail = self.lib.moe_last_error(self.handle).decode()
            name = self.lib.moe_status_string(st).decode()
            raise MoEError(st, f"{what}: {name}" + (f": {detail}" if detail else ""))

    def close(self):
        if getattr(self, "handle", None):
            self.lib.moe_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ weights --
    def load_weights(self, layer: int, w: dict):
        """`w` holds device tensors in the layout of include/sparse_moe.h
        (keys: router_w, router_b, gate_up, gate_up_scale, down, down_scale,
        sh_gate_up, sh_gate_up_scale, sh_down, sh_down_scale, sh_gate_w, the
        optional down_f16, sh_down_f16, and for affine int4 gate_up_bias,
        down_bias, sh_gate_up_bias, sh_down_bias).
        The context borrows them; a reference is kept here."""
        for k, v in w.items():
            if v is not None and (not v.is_cuda or not v.is_contiguous()):
                raise ValueError(f"{k} must be a contiguous CUDA tensor")
        mw = _abi.MoeWeights(*[_ptr(w.get(n)) for n, _ in _abi.MoeWeights._fields_])
        self._check(self.lib.moe_load_weights(self.handle, layer, ctypes.byref(mw)),
                    "moe_load_weights")
        self._weights[layer] = w

    # ------------------------------------------------------------ compute --
    def route(self, layer: int, x: torch.Tensor, stream=None, want_logits: bool = True) -> dict:
        T = x.shape[0]
        dev = self.device
        E, k = self.n_experts, self.top_k
        out = dict(
            logits=torch.empty((T, E), dtype=torch.float32, device=dev) if want_logits else None,
            topk_idx=torch.empty((T, k), dtype=torch.int32, device=dev),
            topk_w=torch.empty((T, k), dtype=torch.float32, device=dev),
            counts=torch.empty((E,), dtype=torch.int32, device=dev),
            offsets=torch.empty((E + 1,), dtype=torch.int32, device=dev),
            sorted_rows=torch.empty((T * k,), dtype=torch.int32, device=dev),
            pos_of_assign=torch.empty((T * k,), dtype=torch.int32, device=dev),
        )
        st = self.lib.moe_route(self.handle, layer, _ptr(x), T, _ptr(out["logits"]),
                                _ptr(out["topk_idx"]), _ptr(out["topk_w"]), _ptr(out["counts"]),
                                _ptr(out["offsets"]), _ptr(out["sorted_rows"]),
                                _ptr(out["pos_of_assign"]), _stream_handle(stream, dev))
        self._check(st, "moe_route")
        return out

    def forward_prefill(self, layer: int, x: torch.Tensor, y: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty_like(x)
        st = self.lib.moe_forward_prefill(self.handle, layer, _ptr(x), x.shape[0], _ptr(y),
                                          _stream_handle(stream, self.device))
        self._check(st, "moe_forward_prefill")
        return y

    def forward_decode(self, layer: int, x: torch.Tensor, y: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty_like(x)
        st = self.lib.moe_forward_decode(self.handle, layer, _ptr(x), _ptr(y),
                                         _stream_handle(stream, self.device))
        self._check(st, "moe_forward_decode")
        return y

    def forward_decode_layers(self, first_layer: int, x: torch.Tensor, y: torch.Tensor,
                              chained: bool = False, stream=None) -> torch.Tensor:
        """Layers first_layer .. first_layer + n - 1 in one launch per up to 48
        layers.  Independent inputs: x and y are [n, H] (layer l reads x[l],
        writes y[l]).  chained=True: y is [n, H] and x is [1, H]; layer 0 reads
        x, layer l > 0 reads y[l - 1]."""
        H = self.hidden
        if chained:
            n = y.shape[0]
            buf = torch.empty((n + 1, H), dtype=torch.bfloat16, device=y.device)
            buf[0].copy_(x.reshape(H))
            st = self.lib.moe_forward_decode_layers(self.handle, first_layer, n, _ptr(buf), H,
                                                    ctypes.c_void_p(buf[1:].data_ptr()), H,
                                                    _stream_handle(stream, self.device))
            self._check(st, "moe_forward_decode_layers")
            y.copy_(buf[1:])
            return y
        n = x.shape[0]
        st = self.lib.moe_forward_decode_layers(self.handle, first_layer, n, _ptr(x), H, _ptr(y), H,
                                                _stream_handle(stream, self.device))
        self._check(st, "moe_forward_decode_layers")
        return y

    def forward_rows(self, layer: int, x: torch.Tensor, y: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
        """y[T, H] for x[T, H] (device bf16, 1 <= T <= 16) through the
        decode-style path that reads each needed weight row once for all T
        rows (moe_forward_rows)."""
        if y is None:
            y = torch.empty_like(x)
        st = self.lib.moe_forward_rows(self.handle, layer, _ptr(x), x.shape[0], _ptr(y),
                                       _stream_handle(stream, self.device))
        self._check(st, "moe_forward_rows")
        return y

    def rows_routing(self, T: int, stream=None) -> dict:
        """Routing of the last forward_rows call (T rows)."""
        dev = self.device
        out = dict(logits=torch.empty((T, self.n_experts), dtype=torch.float32, device=dev),
                   topk_idx=torch.empty((T, self.top_k), dtype=torch.int32, device=dev),
                   topk_w=torch.empty((T, self.top_k), dtype=torch.float32, device=dev))
        st = self.lib.moe_rows_routing(self.handle, _ptr(out["logits"]), _ptr(out["topk_idx"]),
                                       _ptr(out["topk_w"]), _stream_handle(stream, dev))
        self._check(st, "moe_rows_routing")
        return out

    def decode_routing(self, stream=None) -> dict:
        dev = self.device
        out = dict(logits=torch.empty((self.n_experts,), dtype=torch.float32, device=dev),
                   topk_idx=torch.empty((self.top_k,), dtype=torch.int32, device=dev),
                   topk_w=torch.empty((self.top_k,), dtype=torch.float32, device=dev))
        st = self.lib.moe_decode_routing(self.handle, _ptr(out["logits"]), _ptr(out["topk_idx"]),
                                         _ptr(out["topk_w"]), _stream_handle(stream, dev))
        self._check(st, "moe_decode_routing")
        return out

    def forward_prefill_host(self, layer: int, x_host: torch.Tensor, y_host: torch.Tensor,
                             stream=None):
        """x_host, y_host: CPU bf16 [T, H] (pinned for asynchronous copies)."""
        st = self.lib.moe_forward_prefill_host(self.handle, layer, _ptr(x_host), x_host.shape[0],
                                               _ptr(y_host), _stream_handle(stream, self.device))
        self._check(st, "moe_forward_prefill_host")

    def forward_decode_host(self, layer: int, x_host: torch.Tensor, y_host: torch.Tensor,
                            stream=None):
        st = self.lib.moe_forward_decode_host(self.handle, layer, _ptr(x_host), _ptr(y_host),
                                              _stream_handle(stream, self.device))
        self._check(st, "moe_forward_decode_host")

    def check_device(self) -> int:
        code = ctypes.c_int32(0)
        st = self.lib.moe_check_device(self.handle, ctypes.byref(code))
        self._check(st, "moe_check_device")
        return code.value

    def profile(self, on: bool):
        self._check(self.lib.moe_profile_enable(self.handle, int(on)), "moe_profile_enable")

    def profile_read(self) -> dict:
        arr = (_abi.MoeKernelStat * 32)()
        n = ctypes.c_int(0)
        self._check(self.lib.moe_profile_read(self.handle, arr, 32, ctypes.byref(n)),
                    "moe_profile_read")
        return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms)
                for i in range(min(n.value, 32))}

    def decode_phase_read(self) -> dict:
        """Phase B of the last decode launched while profiling was on: the
        span from the first CTA's start to the last CTA's end, and the median
        CTA's duration (µs)."""
        win = ctypes.c_double(0.0)
        med = ctypes.c_double(0.0)
        self._check(self.lib.moe_decode_phase_read(self.handle, ctypes.byref(win), ctypes.byref(med)),
                    "moe_decode_phase_read")
        return {"window_us": win.value, "median_us": med.value}

    @property
    def launch_count(self) -> int:
        return int(self.lib.moe_launch_count(self.handle))
