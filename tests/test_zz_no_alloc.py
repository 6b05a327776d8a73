"""The allocation-free block entry point against the workspace one.

h3dit_block_forward_noalloc exists for callers that cannot allocate device
memory or pass a workspace (a host program whose own allocator owns all
device memory, a serving loop that must not call cudaMalloc).  It runs the
same block with the library's built-in scratch.  Both entry points launch the
same kernels on the same inputs, and those kernels have no atomics and no
order-dependent reductions across CTAs, so every call must give the workspace
entry point's output bit for bit.  Two calls in a row, on different inputs,
show that whatever the first call left in the shared scratch does not leak
into the second; this is run on the BF16 block and on the dynamic-int8 block,
whose scratch also holds the activation scales and the int8 codes.  Shapes too
large for the scratch are refused, after the ordinary argument checks.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_bf16, dev_f32, host, max_abs, rel_l2, shape_of

pytestmark = pytest.mark.gpu


def _codes_dev(q):
    return torch.from_numpy(np.ascontiguousarray(q, np.float32)).to("cuda").to(torch.bfloat16)


def _inputs(seed, int8):
    w = synth.WORKLOADS["tiny_block"]
    n = w.n_tokens
    wt = synth.host_block_weights(w.d, w.ffn, seed=seed)
    keep = []
    if int8:
        dev = {}
        for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"),
                             ("w2", "q2", "s2")):
            q, s = O.quantize_weight(wt[name])
            dev[qn], dev[sn] = _codes_dev(q), dev_f32(s[:, 0])
        keep.append(dev)
        bw = H.block_weights(dev["q_qkv"], dev["q_o"], dev["q1"], dev["q2"], dev["s_qkv"], dev["s_o"], dev["s1"],
                             dev["s2"])
    else:
        dev = {k: dev_bf16(v) for k, v in wt.items()}
        keep.append(dev)
        bw = H.block_weights(dev["w_qkv"], dev["w_o"], dev["w1"], dev["w2"])
    mod = dev_f32(synth.host_mod(w.d, seed=seed))
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    x = synth.host_activations(n, w.d, seed=seed + 100)
    return w, n, keep, bw, mod, pos, x


@pytest.mark.parametrize("precision", [H.BF16, H.INT8])
def test_noalloc_matches_workspace_entry_two_calls(precision):
    for seed in (11, 12):
        w, n, keep, bw, mod, pos, x = _inputs(seed, precision == H.INT8)
        shape = shape_of(w, precision)
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
        if not torch.equal(x_na, x_ref):
            got, ref = host(x_na), host(x_ref)
            pytest.fail(f"call seed {seed}: not bit-identical to the workspace entry point "
                        f"(rel_l2={rel_l2(got, ref):.2e} max_abs={max_abs(got, ref):.2e}, "
                        f"{int((x_na != x_ref).sum())} elements differ)")
        # and the call did compute the block (the branch is not zero)
        assert rel_l2(host(x_na), x) > 1e-3


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
    # argument errors are reported as such, whatever the size
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_block_forward_noalloc(shape, dummy, x, None, x, w.n_tokens)
    assert e.value.status == H.E_INVAL
