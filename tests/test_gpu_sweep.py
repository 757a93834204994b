"""Prompt-length sweep (T = 256 .. 128K, 4096-row chunks, router bias 1.5,
seed = T) against the fp64 oracle: routing of the sampled chunks bit for bit,
the layer output on sampled tokens (first, last, chunk boundaries, random).
Section "Bound temporary memory with prompt chunking": chunking must not
change the output, so every token is checked against the unchunked
definition."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_layer_close, check_routing, host_layer, make_ctx
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

CHUNK = 4096


@pytest.mark.parametrize("T", [256, 2048, 16384, 131072])
def test_sweep_length_matches_oracle(T):
    wl = moe_synth.sweep_workload(T)
    ctx, (w,) = make_ctx(wl, max_chunk_rows=CHUNK)
    x = moe_synth.make_x(wl, device="cuda")
    y = ctx.forward_prefill(0, x)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    nchunks = (T + CHUNK - 1) // CHUNK
    chunks = sorted({0, nchunks // 2, nchunks - 1})
    rng = np.random.default_rng(T)
    hl = host_layer(w)
    for c in chunks:
        c0, c1 = c * CHUNK, min(T, (c + 1) * CHUNK)
        xc = x[c0:c1]
        # routing of the whole chunk, bit for bit against the oracle's
        # re-selection from the GPU logits
        lg = check_routing(ctx, w, xc)
        n = c1 - c0
        local = np.unique(np.concatenate([[0, n - 1], rng.choice(n, min(n, 12), replace=False)]))
        ref = orc.moe_layer(xc.float().cpu().numpy(), hl, ctx.top_k, logits=lg, tokens=local)
        got = y[c0 + torch.as_tensor(local, device="cuda")].float().cpu().numpy()
        assert_layer_close(got, ref, what=f"T={T} chunk {c}")
