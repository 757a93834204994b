"""The allocation-free decode entry point (for callers that cannot allocate
device memory, so cannot hand a context its workspace) must give the same
output as the context-based decode, call after call, through the C ABI: it
runs the same kernel on the same inputs, so the outputs must be equal bit
for bit.  One case is also checked against the fp64 oracle.
This file is collected last so that, if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_layer_close, host_layer, make_ctx
from oracle import moe_oracle as orc
from sparse_moe_gb300 import _abi

pytestmark = pytest.mark.gpu

WFMT = {moe_synth.WFMT_BF16: _abi.MOE_W_BF16, moe_synth.WFMT_INT4: _abi.MOE_W_INT4_SYM_G64,
        moe_synth.WFMT_INT4_AFFINE: _abi.MOE_W_INT4_AFFINE_G64}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("wl", [moe_synth.Workload("na_tiny", moe_synth.TINY, T=1, seed=21),
                                moe_synth.DECODE_BF16, moe_synth.DECODE_INT4,
                                moe_synth.DECODE_INT4_AFFINE],
                         ids=["tiny", "qwen_bf16", "qwen_int4", "qwen_int4_affine"])
def test_noalloc_decode_matches_context_decode(wl):
    lib = _abi.load()
    ctx, (w,) = make_ctx(wl, max_chunk_rows=16)
    s = wl.shape
    cfg = _abi.MoeConfig(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, 1, 16,
                         WFMT[wl.wfmt])
    mw = _abi.MoeWeights(*[_ptr(w.get(n)) for n, _ in _abi.MoeWeights._fields_])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):                       # two calls in a row share the scratch
        x = moe_synth.make_x(wl, layer=call, device="cuda")
        y_ref = ctx.forward_decode(0, x)
        y = torch.full_like(x, float("nan"))
        st = lib.moe_forward_decode_noalloc(ctypes.byref(cfg), ctypes.byref(mw), _ptr(x), _ptr(y),
                                            stream)
        assert st == _abi.MOE_OK, lib.moe_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), f"call {call}: differs from moe_forward_decode"
        if call == 1 and wl.shape == moe_synth.TINY:
            # the same output against the oracle, routed from the context
            # decode's logits (equal outputs imply the same selection)
            lg = ctx.decode_routing()["logits"].cpu().numpy()[None, :]
            ref = orc.moe_layer(x.float().cpu().numpy(), host_layer(w), s.top_k, logits=lg)
            assert_layer_close(y.float().cpu().numpy(), ref, what="no-alloc decode")
    # no bounded wait ran out: the entry point's status word reads clear
    code = ctypes.c_int32(-1)
    assert lib.moe_check_device(None, ctypes.byref(code)) == _abi.MOE_OK
    assert code.value == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = _abi.load()
    cfg = _abi.MoeConfig(2048, 256, 32, 4096, 4096, 1, 16, _abi.MOE_W_BF16)  # (k+1)*I*4 > 64 KiB
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = _ptr(dummy)
    mw = _abi.MoeWeights(p, None, p, None, p, None, p, None, p, None, p)
    st = lib.moe_forward_decode_noalloc(ctypes.byref(cfg), ctypes.byref(mw), p, p, None)
    assert st == _abi.MOE_ERR_WORKSPACE
