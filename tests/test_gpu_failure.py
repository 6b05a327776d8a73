"""Failure paths on the GPU, driven without faulting or hanging it.

* A stalled pipeline: the wait limit is shortened to milliseconds and the
  next projection's first CTA is told to stop loading before one k-block, so
  the tensor-core thread's bounded wait on that stage runs out with no copy
  in flight.  The launch must end by itself, h3dit_check_device_error must
  report E_TIMEOUT (once: the word is cleared), and the next ordinary calls
  must give correct results on the same context.
* Poisoned workspaces: the activation arenas are aliased by lifetime
  ([linlog] "DiT 融合内核": activation-buffer aliasing), so a read of an
  arena byte before it is written would pick up a previous tensor.  Filling
  the workspace with NaN bit patterns (0xFF bytes: BF16 0xFFFF, fp32
  0xFFFFFFFF) before a block, an int8 block and a reduced step must give
  outputs bit-identical to a zero-filled workspace.
"""
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_bf16, dev_f32, host, max_abs, oracle_cfg, rel_l2, shape_of

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_block"]


def _linear_case(m, n, k, seed):
    a = synth.host_activations(m, k, seed=seed)
    b = synth.host_activations(n, k, seed=seed + 1) * np.float32(0.05)
    b = synth.to_bf16_values(b)
    return a, b


def _linear_ok(got, a, b):
    ref = O.bf16_round(np.asarray(a, np.float64) @ np.asarray(b, np.float64).T)
    return rel_l2(got, ref) <= 5e-3 and max_abs(got, ref) <= 2.0 ** -7 * float(np.max(np.abs(ref))) + 1e-6


def test_stalled_projection_times_out_and_the_context_recovers():
    m, n, k = 1000, 512, 1024
    a, b = _linear_case(m, n, k, seed=3)
    ad, bd = dev_bf16(a), dev_bf16(b)
    c = torch.zeros((m, n), device="cuda", dtype=torch.bfloat16)
    H.h3dit_check_device_error()          # start from a clear error word
    try:
        H.h3dit_test_set_wait_limit(5_000_000)      # 5 ms
        H.h3dit_test_stall_next_gemm(3)
        H.h3dit_linear(ad, bd, m, n, k, 0, c)
        with pytest.raises(H.H3DitError) as e:
            H.h3dit_check_device_error()
        assert e.value.status == H.E_TIMEOUT
        # the word was cleared by that read
        H.h3dit_check_device_error()
        # a stall inside a whole block: the QKV projection stops at k-block 1
        w = TINY
        nt = w.n_tokens
        shape = shape_of(w)
        wt = {kk: dev_bf16(v) for kk, v in synth.host_block_weights(w.d, w.ffn, seed=9).items()}
        bw = H.block_weights(wt["w_qkv"], wt["w_o"], wt["w1"], wt["w2"])
        mod = dev_f32(synth.host_mod(w.d, seed=9))
        pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
        x = synth.host_activations(nt, w.d, seed=9)
        nbytes = H.h3dit_workspace_size(shape, nt)
        ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
        xs = dev_bf16(x)
        H.h3dit_test_stall_next_gemm(1)
        H.h3dit_block_forward(shape, bw, mod, xs, pos, nt, ws, nbytes)
        with pytest.raises(H.H3DitError) as e:
            H.h3dit_check_device_error()
        assert e.value.status == H.E_TIMEOUT
    finally:
        H.h3dit_test_stall_next_gemm(-1)
        H.h3dit_test_set_wait_limit(0)
    # ordinary calls on the same context give the right results
    c2 = torch.zeros_like(c)
    H.h3dit_linear(ad, bd, m, n, k, 0, c2)
    H.h3dit_check_device_error()
    assert _linear_ok(host(c2), a, b)
    xr = dev_bf16(x)
    H.h3dit_block_forward(shape, bw, mod, xr, pos, nt, ws, nbytes)
    H.h3dit_check_device_error()
    cfg = oracle_cfg(w)
    wh = {kk: v.float().cpu().numpy() for kk, v in wt.items()}
    ref_bf = O.block_forward(x, wh, host(mod), host(pos), cfg, bf16_storage=True)
    got = host(xr)
    assert rel_l2(got, ref_bf) <= 1e-2 and rel_l2(got - x, ref_bf - x) <= 2e-2


def _fill(ws, byte):
    ws.fill_(byte)
    torch.cuda.synchronize()


def _block_both(shape, bw, mod, pos, x, n):
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    outs = []
    for byte in (0x00, 0xFF):
        _fill(ws, byte)
        xd = dev_bf16(x)
        H.h3dit_block_forward(shape, bw, mod, xd, pos, n, ws, nbytes)
        H.h3dit_check_device_error()
        outs.append(xd)
    return outs


@pytest.mark.parametrize("n", [256, 77])
def test_poisoned_workspace_block_bf16(n):
    w = TINY
    shape = shape_of(w)
    wt = {k: dev_bf16(v) for k, v in synth.host_block_weights(w.d, w.ffn, seed=21).items()}
    bw = H.block_weights(wt["w_qkv"], wt["w_o"], wt["w1"], wt["w2"])
    mod = dev_f32(synth.host_mod(w.d, seed=21))
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio)[:n])
    x = synth.host_activations(n, w.d, seed=21)
    zero, poison = _block_both(shape, bw, mod, pos, x, n)
    assert torch.equal(zero, poison)
    assert not torch.isnan(poison.float()).any()


def test_poisoned_workspace_block_int8():
    w = TINY
    n = w.n_tokens
    shape = shape_of(w, H.INT8)
    wt = synth.host_block_weights(w.d, w.ffn, seed=22)
    dev = {}
    for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"), ("w2", "q2", "s2")):
        q, s = O.quantize_weight(wt[name])
        dev[qn], dev[sn] = dev_bf16(q.astype(np.float32)), dev_f32(s[:, 0])
    bw = H.block_weights(dev["q_qkv"], dev["q_o"], dev["q1"], dev["q2"], dev["s_qkv"], dev["s_o"], dev["s1"], dev["s2"])
    mod = dev_f32(synth.host_mod(w.d, seed=22))
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    x = synth.host_activations(n, w.d, seed=22)
    zero, poison = _block_both(shape, bw, mod, pos, x, n)
    assert torch.equal(zero, poison)
    assert not torch.isnan(poison.float()).any()


def test_poisoned_workspace_reduced_step():
    w = TINY
    n = w.n_tokens
    nb = 5
    shape = shape_of(w)
    devs = []
    for b in range(nb):
        wt = {k: dev_bf16(v) for k, v in synth.host_block_weights(w.d, w.ffn, seed=23, block=b).items()}
        devs.append((wt, H.block_weights(wt["w_qkv"], wt["w_o"], wt["w1"], wt["w2"])))
    mods = dev_f32(np.stack([synth.host_mod(w.d, seed=23, block=b) for b in range(nb)]))
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    x = synth.host_activations(n, w.d, seed=23)
    T, Hh, W = w.video
    tr = H.reduction(H.video_grid(0, T, Hh, W), 1, 3)
    nbytes = H.h3dit_workspace_size(shape, n, tr)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    outs = []
    for byte in (0x00, 0xFF):
        _fill(ws, byte)
        xd = dev_bf16(x)
        H.h3dit_step_forward(shape, [d[1] for d in devs], mods, xd, pos, n, tr, ws, nbytes)
        H.h3dit_check_device_error()
        outs.append(xd)
    assert torch.equal(outs[0], outs[1])
    assert not torch.isnan(outs[1].float()).any()
