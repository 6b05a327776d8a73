"""The allocation-free block entry point against the workspace one.

h3dit_block_forward_noalloc exists for callers that cannot allocate device
memory or pass a workspace (a host program whose own allocator owns all
device memory, a serving loop that must not call cudaMalloc).  It runs the
same block with the library's built-in scratch.  Two calls in a row, on
different inputs, must each match h3dit_block_forward on the same inputs
within the block tolerances used elsewhere in the tests; the second call
also shows that whatever the first call left in the shared scratch does not
leak into the result.  A shape too large for the scratch must be refused.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_bf16, dev_f32, host, max_abs, rel_l2, shape_of

pytestmark = pytest.mark.gpu


def _inputs(seed):
    w = synth.WORKLOADS["tiny_block"]
    n = w.n_tokens
    wt = {k: dev_bf16(v) for k, v in synth.host_block_weights(w.d, w.ffn, seed=seed).items()}
    bw = H.block_weights(wt["w_qkv"], wt["w_o"], wt["w1"], wt["w2"])
    mod = dev_f32(synth.host_mod(w.d, seed=seed))
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    x = synth.host_activations(n, w.d, seed=seed + 100)
    return w, n, wt, bw, mod, pos, x


def test_noalloc_matches_workspace_entry_two_calls():
    for seed in (11, 12):
        w, n, wt, bw, mod, pos, x = _inputs(seed)
        shape = shape_of(w)
        # existing entry point, caller workspace
        x_ref = dev_bf16(x)
        nbytes = H.h3dit_workspace_size(shape, n)
        ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
        H.h3dit_block_forward(shape, bw, mod, x_ref, pos, n, ws, nbytes)
        H.h3dit_check_device_error()
        # allocation-free entry point
        x_na = dev_bf16(x)
        H.h3dit_block_forward_noalloc(shape, bw, mod, x_na, pos, n)
        H.h3dit_check_device_error()
        got, ref = host(x_na), host(x_ref)
        r, m = rel_l2(got, ref), max_abs(got, ref)
        rb = rel_l2(got - x, ref - x)
        assert r <= 1e-2 and m <= 5e-2 and rb <= 2e-2, f"call seed {seed}: rel_l2={r:.2e} max_abs={m:.2e} branch={rb:.2e}"


def test_noalloc_refuses_shapes_beyond_its_scratch():
    w = synth.WORKLOADS["block_512"]
    shape = shape_of(w)
    need = H.h3dit_workspace_size(shape, w.n_tokens)
    assert need > 64 << 20
    x = torch.zeros((8, w.d), device="cuda", dtype=torch.bfloat16)
    dummy = H.block_weights(x, x, x, x)
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_block_forward_noalloc(shape, dummy, x, x, x, w.n_tokens)
    assert e.value.status == H.E_NOMEM
    assert "scratch" in str(e.value)
