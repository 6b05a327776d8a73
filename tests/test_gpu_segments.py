"""Per-segment AdaLN modulation on the GPU through the C ABI against the
oracle ([linlog] "音频处理": the reference audio is conditioned at its own
timestep, so its precomputed AdaLN vectors differ from the video's).

The tiny workload's video (192 tokens), text (48) and audio (16) get three
different modulation sets.  Checked: the block against the oracle with the
per-token modulation; one segment equal to h3dit_block_forward bit for bit;
the int8 block with segments; a reduced step whose segment boundaries move
with the pairing; malformed tables refused."""
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_bf16, dev_f32, host, oracle_cfg, rel_l2, shape_of
from tests.test_gpu_block import assert_block

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_block"]
STARTS = [0, 192, 240]          # video, text, audio


def _seg_mods(seed, nseg=3, d=TINY.d, std=0.3):
    return np.stack([synth.host_mod(d, seed=seed, block=100 + k, std=std) for k in range(nseg)])


def _dev_weights(wt):
    dev = {k: dev_bf16(v) for k, v in wt.items()}
    return dev, H.block_weights(dev["w_qkv"], dev["w_o"], dev["w1"], dev["w2"])


def test_block_three_segments():
    w = TINY
    n = w.n_tokens
    shape = shape_of(w)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=31)
    wt = synth.host_block_weights(w.d, w.ffn, seed=31)
    mods = _seg_mods(31)
    dev, bw = _dev_weights(wt)
    xd = dev_bf16(x)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_block_forward_seg(shape, bw, dev_f32(mods), H.segments(STARTS), xd, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(xd)
    per_row = O.segment_mod(mods, STARTS, n)
    cfg = oracle_cfg(w)
    ref = O.block_forward(x, wt, per_row, pos, cfg)
    ref_bf = O.block_forward(x, wt, per_row, pos, cfg, bf16_storage=True)
    assert_block(got, x, ref, ref_bf)
    # the single-set block differs: the segments really apply
    one = O.block_forward(x, wt, mods[0], pos, cfg, bf16_storage=True)
    assert rel_l2(got[200:] - x[200:], one[200:] - x[200:]) > 0.1


def test_one_segment_equals_plain_block():
    w = TINY
    n = w.n_tokens
    shape = shape_of(w)
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    x = synth.host_activations(n, w.d, seed=32)
    wt = synth.host_block_weights(w.d, w.ffn, seed=32)
    mod = synth.host_mod(w.d, seed=32)
    dev, bw = _dev_weights(wt)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    a = dev_bf16(x)
    H.h3dit_block_forward(shape, bw, dev_f32(mod), a, pos, n, ws, nbytes)
    b = dev_bf16(x)
    H.h3dit_block_forward_seg(shape, bw, dev_f32(mod[None]), H.segments([0]), b, pos, n, ws, nbytes)
    H.h3dit_check_device_error()
    assert torch.equal(a, b)


def test_int8_block_three_segments():
    from tests.test_gpu_int8 import _int8_weights
    w = TINY
    n = w.n_tokens
    shape = shape_of(w, H.INT8)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=33)
    wt = synth.host_block_weights(w.d, w.ffn, seed=33)
    mods = _seg_mods(33)
    hw, _, bw = _int8_weights(wt)
    xd = dev_bf16(x)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_block_forward_seg(shape, bw, dev_f32(mods), H.segments(STARTS), xd, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(xd)
    per_row = O.segment_mod(mods, STARTS, n)
    cfg = oracle_cfg(w)
    ref_bf = O.block_forward_int8(x, hw, per_row, pos, cfg, bf16_storage=True)
    ref64 = O.block_forward_int8(x, hw, per_row, pos, cfg, bf16_storage=False)
    assert_block(got, x, ref64, ref_bf)


def test_reduced_step_with_segments():
    """3 blocks, pairing after block 0 and restore before block 2: the text
    and audio boundaries move up by the 96 rows the pairing removes."""
    w = TINY
    n = w.n_tokens
    shape = shape_of(w)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=34)
    nb = 3
    wts = [synth.host_block_weights(w.d, w.ffn, seed=34, block=b) for b in range(nb)]
    mods = np.stack([_seg_mods(34 + 10 * b) for b in range(nb)])      # [nb][3][6][d]
    devs = [_dev_weights(t) for t in wts]
    T, Hh, W = w.video
    tr = H.reduction(H.video_grid(0, T, Hh, W), 0, 2)
    nbytes = H.h3dit_workspace_size(shape, n, tr)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    xd = dev_bf16(x)
    H.h3dit_step_forward_seg(shape, [d_[1] for d_ in devs], dev_f32(mods), H.segments(STARTS), xd, dev_f32(pos), n,
                             tr, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(xd)
    cfg = oracle_cfg(w)
    per_row = [O.segment_mod(mods[b], STARTS, n) for b in range(nb)]
    red = O.Reduction(O.VideoGrid(0, T, Hh, W), 0, 2)
    ref_bf = O.step_forward(x, wts, per_row, pos, cfg, reduction=red, bf16_storage=True)
    ref = O.step_forward(x, wts, per_row, pos, cfg, reduction=red)
    assert rel_l2(got, ref_bf) <= 1e-2 * nb and rel_l2(got - x, ref_bf - x) <= 2e-2 * nb
    assert rel_l2(got, ref) <= 1e-2 * nb


def test_malformed_segments_refused():
    w = TINY
    n = w.n_tokens
    shape = shape_of(w)
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    wt = synth.host_block_weights(w.d, w.ffn, seed=35)
    dev, bw = _dev_weights(wt)
    mods = dev_f32(_seg_mods(35, nseg=4))
    xd = dev_bf16(synth.host_activations(n, w.d, seed=35))
    T, Hh, W = w.video
    tr = H.reduction(H.video_grid(0, T, Hh, W), 0, 2)
    nbytes = H.h3dit_workspace_size(shape, n, tr)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    bad = [[5, 100], [0, 300], [0, 100, 50]]
    for starts in bad:
        with pytest.raises(H.H3DitError) as e:
            H.h3dit_block_forward_seg(shape, bw, mods, H.segments(starts), xd, pos, n, ws, nbytes)
        assert e.value.status == H.E_INVAL
    sg = H.Segments()
    sg.count = 5
    with pytest.raises(H.H3DitError):
        H.h3dit_block_forward_seg(shape, bw, mods, sg, xd, pos, n, ws, nbytes)
    # a boundary inside the paired video grid
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_step_forward_seg(shape, [bw], mods, H.segments([0, 100]), xd, pos, n, tr, ws, nbytes)
    assert e.value.status == H.E_INVAL and "inside" in H.lib().h3dit_last_error().decode()


def test_int8_reduced_step_with_segments():
    from tests.test_gpu_int8 import _int8_weights
    w = TINY
    n = w.n_tokens
    shape = shape_of(w, H.INT8)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=36)
    nb = 3
    wts = [synth.host_block_weights(w.d, w.ffn, seed=36, block=b) for b in range(nb)]
    packs = [_int8_weights(t) for t in wts]
    mods = np.stack([_seg_mods(36 + 10 * b) for b in range(nb)])
    T, Hh, W = w.video
    tr = H.reduction(H.video_grid(0, T, Hh, W), 0, 2)
    nbytes = H.h3dit_workspace_size(shape, n, tr)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    xd = dev_bf16(x)
    H.h3dit_step_forward_seg(shape, [p[2] for p in packs], dev_f32(mods), H.segments(STARTS), xd, dev_f32(pos), n,
                             tr, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(xd)
    cfg = oracle_cfg(w)
    per_row = [O.segment_mod(mods[b], STARTS, n) for b in range(nb)]
    red = O.Reduction(O.VideoGrid(0, T, Hh, W), 0, 2)
    ref_bf = O.step_forward(x, [p[0] for p in packs], per_row, pos, cfg, reduction=red, bf16_storage=True, int8=True)
    assert rel_l2(got, ref_bf) <= 1e-2 * nb and rel_l2(got - x, ref_bf - x) <= 2e-2 * nb
