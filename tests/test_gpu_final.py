"""The final layer on the GPU through the C ABI against the oracle ([linlog]
"DiT 融合内核": the audio and video heads normalise their rows of the residual
stream in place with their own AdaLN vectors, and the BF16 head applies the
AdaLN while loading its projection tiles).

Tolerance: each output is one BF16 rounding of an fp32 dot product of d BF16
operands that the oracle also rounds (the normalised row), so relative L2
<= 5e-3 and max-abs <= 2^-7 max|ref| against the oracle with BF16 storage;
against the pure fp64 oracle relative L2 <= 1e-2 (the BF16 rounding of the
normalised operand adds 2^-9 relative per term)."""
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_bf16, dev_f32, host, max_abs, rel_l2, shape_of

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_block"]


def _run(w, x, specs, seed):
    """specs: list of (row_start, rows, c_out); returns (outputs, oracle inputs)."""
    n = x.shape[0]
    shape = shape_of(w)
    xd = dev_bf16(x)
    heads, keep, hosts = [], [], []
    for k, (r0, rows, c) in enumerate(specs):
        mod = synth.host_mod(w.d, seed=seed, block=50 + k, std=0.3)
        wt = synth.host_block_weights(w.d, c, seed=seed, block=60 + k)["w1"]   # [c][d], N(0, 0.02)
        sh, sc, wd = dev_f32(mod[0]), dev_f32(mod[1]), dev_bf16(wt)
        out = torch.empty((rows, c), device="cuda", dtype=torch.bfloat16)
        heads.append(H.final_head(r0, rows, sh, sc, wd, c, out))
        keep += [sh, sc, wd, out]
        hosts.append((r0, rows, mod[0], mod[1], wt, out))
    H.h3dit_final_layer(shape, xd, n, heads)
    H.h3dit_check_device_error()
    return hosts


def _check(x, hosts, eps):
    for r0, rows, sh, sc, wt, out in hosts:
        got = host(out)
        ref_bf = O.final_head(x, r0, rows, sh, sc, wt, eps, bf16_storage=True)
        ref = O.final_head(x, r0, rows, sh, sc, wt, eps)
        assert rel_l2(got, ref_bf) <= 5e-3
        assert max_abs(got, ref_bf) <= 2.0 ** -7 * float(np.max(np.abs(ref_bf))) + 1e-6
        assert rel_l2(got, ref) <= 1e-2


def test_final_layer_video_and_audio_heads():
    w = TINY
    n = w.n_tokens
    x = synth.host_activations(n, w.d, seed=41, std=2.0)
    # video rows 0..191 (c_out 64), audio rows 240..255 (c_out 32)
    hosts = _run(w, x, [(0, 192, 64), (240, 16, 32)], seed=41)
    _check(x, hosts, w.eps)


@pytest.mark.parametrize("r0,rows,c", [(0, 1, 16), (3, 129, 256), (100, 156, 48)])
def test_final_layer_ragged_heads(r0, rows, c):
    w = TINY
    n = w.n_tokens
    x = synth.host_activations(n, w.d, seed=42 + rows, std=3.0)
    hosts = _run(w, x, [(r0, rows, c)], seed=42 + rows)
    _check(x, hosts, w.eps)


@pytest.mark.parametrize("rows", [5120, 9728])
def test_final_layer_cluster_splits(rows):
    """Enough 128-row tiles that the head kernel splits d over 3 CTAs (40
    tiles, uneven k-block ranges at d = 256) or does not split (76 tiles)."""
    w = TINY
    x = synth.host_activations(rows + 8, w.d, seed=45, std=2.0)
    hosts = _run(w, x, [(5, rows, 64)], seed=45)
    _check(x, hosts, w.eps)


@pytest.mark.slow
def test_final_layer_512_class_sampled_rows():
    """Video rows 0..6143 and audio rows 6656..6911 of the 512-class stream."""
    w = synth.WORKLOADS["block_512"]
    n = w.n_tokens
    x = synth.device_activations(n, w.d, seed=43)
    xh = host(x)
    hosts = _run(w, xh, [(0, 6144, 64), (6656, 256, 64)], seed=43)
    rows = [0, 127, 128, 3000, 6143]
    for (r0, nr, sh, sc, wt, out), sel in zip(hosts, (rows, [0, 100, 255])):
        got = host(out)[sel]
        ref_bf = np.stack([O.final_head(xh, r0 + i, 1, sh, sc, wt, w.eps, bf16_storage=True)[0] for i in sel])
        assert rel_l2(got, ref_bf) <= 5e-3
        assert max_abs(got, ref_bf) <= 2.0 ** -7 * float(np.max(np.abs(ref_bf))) + 1e-6


def test_final_layer_errors():
    w = TINY
    n = w.n_tokens
    shape = shape_of(w)
    x = dev_bf16(synth.host_activations(n, w.d, seed=44))
    v = dev_f32(np.zeros(w.d, np.float32))
    wt = dev_bf16(np.zeros((256, w.d), np.float32))
    out = torch.empty((256, 256), device="cuda", dtype=torch.bfloat16)
    for spec, status in (((0, 16, 24), H.E_UNSUPPORTED), ((0, 16, 272), H.E_UNSUPPORTED),
                         ((200, 100, 32), H.E_INVAL), ((0, 0, 32), H.E_INVAL)):
        with pytest.raises(H.H3DitError) as e:
            H.h3dit_final_layer(shape, x, n, [H.final_head(spec[0], spec[1], v, v, wt, spec[2], out)])
        assert e.value.status == status


def test_final_layer_enqueued_behind_a_step_reads_the_step_output():
    """Both final-layer launches may be scheduled before the kernel ahead of
    them on the stream has finished (programmatic dependent launch): the
    statistics launch waits for it before reading x, and the head kernel's
    transform warps wait for the statistics before reading them.  Enqueued
    straight behind a 4-block step, with no host synchronisation between,
    the layer gives exactly what it gives on the step's output afterwards."""
    w = TINY
    n = w.n_tokens
    shape = shape_of(w)
    nb = 4
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    x = dev_bf16(synth.host_activations(n, w.d, seed=71))
    devs = [{k: dev_bf16(v) for k, v in synth.host_block_weights(w.d, w.ffn, seed=71, block=b).items()}
            for b in range(nb)]
    bws = [H.block_weights(dv["w_qkv"], dv["w_o"], dv["w1"], dv["w2"]) for dv in devs]
    mods = dev_f32(np.stack([synth.host_mod(w.d, seed=71, block=b) for b in range(nb)]))
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    specs = [(0, 192, 64), (240, 16, 32)]
    params = []
    for k, (r0, rows, c) in enumerate(specs):
        mod = synth.host_mod(w.d, seed=71, block=50 + k, std=0.3)
        wt = synth.host_block_weights(w.d, c, seed=71, block=60 + k)["w1"]
        params.append((r0, rows, c, dev_f32(mod[0]), dev_f32(mod[1]), dev_bf16(wt)))

    def heads():
        hs, outs = [], []
        for r0, rows, c, sh, sc, wd in params:
            out = torch.full((rows, c), float("nan"), device="cuda", dtype=torch.bfloat16)
            hs.append(H.final_head(r0, rows, sh, sc, wd, c, out))
            outs.append(out)
        return hs, outs

    heads_a, outs_a = heads()
    heads_b, outs_b = heads()
    torch.cuda.synchronize()
    H.h3dit_step_forward(shape, bws, mods, x, pos, n, None, ws, nbytes)
    H.h3dit_final_layer(shape, x, n, heads_a)
    torch.cuda.synchronize()
    H.h3dit_check_device_error()
    x_after = x.clone()
    torch.cuda.synchronize()
    H.h3dit_final_layer(shape, x_after, n, heads_b)
    H.h3dit_check_device_error()
    for a, b in zip(outs_a, outs_b):
        assert torch.equal(a, b)
        assert not torch.isnan(a.float()).any()
    xh = host(x_after)
    for (r0, rows, c, sh, sc, wd), out in zip(params, outs_b):
        ref_bf = O.final_head(xh, r0, rows, host(sh), host(sc), host(wd), w.eps, bf16_storage=True)
        assert rel_l2(host(out), ref_bf) <= 5e-3
