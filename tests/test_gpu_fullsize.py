"""Parity at the full workload sizes, in the launch configuration the bench
times, on outputs the oracle can evaluate row by row.

* One BF16 block at the 512x512x22-frame class (d 5120, 40 x 128 heads,
  F 20480, N 6912): the oracle evaluates every token's keys and values and
  then the block output of sampled query rows from several tiles and every
  modality.
* The same block on the dynamic-int8 path (weights quantised per output
  channel by the oracle), sampled rows against the oracle's int8 block; and
  the int8 GEMM's int32 accumulators at the QKV and FC2 shapes, sampled rows
  bit-exact.
* The 50-block step at the 864x480 class (N 10488), with and without token
  reduction: all gates are zero except in one block, so the step output is
  that single block applied to the step input (zero-gate blocks leave the
  residual bit-exact), and the oracle checks sampled rows of it on both
  sides of the video-row, modality and tile boundaries.  The live block is
  each of 0, 3, 4, 39, 40 and 49: the ends of the step and the blocks on
  either side of the reduce (after block 3) and restore (before block 40)
  points, where the fused hand-over of the next block's AdaLN is switched
  off.  This pins the per-block weight and modulation indexing, the fused
  hand-over and the reduce/restore boundaries at full size.
"""
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_f32, host, max_abs, oracle_cfg, rel_l2, shape_of
from tests.test_gpu_block import assert_block

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _host_w(dev):
    return {k: v.float().cpu().numpy() for k, v in dev.items()}


def _bw(dev):
    return H.block_weights(dev["w_qkv"], dev["w_o"], dev["w1"], dev["w2"])


def test_block_512_sampled_rows():
    w = synth.WORKLOADS["block_512"]
    n = w.n_tokens
    shape = shape_of(w)
    dev = synth.device_block_weights(w.d, w.ffn, seed=0, block=0)
    mods = synth.device_mods(1, w.d, seed=0)
    x = synth.device_activations(n, w.d, seed=0)
    x_in = host(x)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_block_forward(shape, _bw(dev), mods, x, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(x)
    rows = [0, 127, 128, 1000, 4095, 6143, 6144, 6500, 6655, 6656, 6911]
    wh, mh, cfg = _host_w(dev), host(mods[0]), oracle_cfg(w)
    ref = O.block_forward(x_in, wh, mh, pos, cfg, rows=rows)
    ref_bf = O.block_forward(x_in, wh, mh, pos, cfg, rows=rows, bf16_storage=True)
    assert_block(got[rows], x_in[rows], ref, ref_bf)


def _codes_dev(q):
    return torch.from_numpy(np.ascontiguousarray(q, np.float32)).to("cuda").to(torch.bfloat16)


def test_int8_gemm_accumulators_full_size_sampled_rows():
    """The QKV and FC2 shapes of the 512 class (6912 x 15360 x 5120 and
    6912 x 5120 x 20480): int32 accumulators of sampled rows bit-exact."""
    rows = [0, 127, 128, 3333, 6143, 6144, 6911]
    for (m, n, k) in ((6912, 15360, 5120), (6912, 5120, 20480)):
        a = synth.host_int8((m, k), seed=k, stream=21)
        b = synth.host_int8((n, k), seed=k, stream=22)
        acc = torch.empty((m, n), device="cuda", dtype=torch.int32)
        H.h3dit_linear_i8_acc(_codes_dev(a), _codes_dev(b), m, n, k, acc)
        H.h3dit_check_device_error()
        got = acc[rows].cpu().numpy().astype(np.int64)
        del acc
        assert np.array_equal(got, O.gemm_int(a[rows], b))


def test_int8_block_512_sampled_rows():
    w = synth.WORKLOADS["block_512_int8"]
    n = w.n_tokens
    shape = shape_of(w, H.INT8)
    dev = synth.device_block_weights(w.d, w.ffn, seed=0, block=0)
    wh = _host_w(dev)
    del dev
    hw, bwd = {}, {}
    for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"), ("w2", "q2", "s2")):
        q, s = O.quantize_weight(wh[name])
        hw[qn], hw[sn] = q, s[:, 0]
        bwd[qn], bwd[sn] = _codes_dev(q), dev_f32(s[:, 0])
    bw = H.block_weights(bwd["q_qkv"], bwd["q_o"], bwd["q1"], bwd["q2"], bwd["s_qkv"], bwd["s_o"], bwd["s1"], bwd["s2"])
    mods = synth.device_mods(1, w.d, seed=0)
    x = synth.device_activations(n, w.d, seed=0)
    x_in = host(x)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_block_forward(shape, bw, mods, x, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(x)
    rows = [0, 127, 128, 1000, 4095, 6143, 6144, 6500, 6655, 6656, 6911]
    mh, cfg = host(mods[0]), oracle_cfg(w)
    ref_bf = O.block_forward_int8(x_in, hw, mh, pos, cfg, bf16_storage=True, rows=rows)
    ref64 = O.block_forward_int8(x_in, hw, mh, pos, cfg, bf16_storage=False, rows=rows)
    assert_block(got[rows], x_in[rows], ref64, ref_bf)


# The live block sits at each boundary of the step: the first and last
# blocks, the last block before the reduction (3), the first and last
# reduced blocks (4, 39) and the first block after the restore (40).  At 3 and
# 39 the fused hand-over of the next block's AdaLN is switched off ([linlog]
# "DiT 融合内核": the next block's AdaLN is emitted only at boundaries without
# token reduction), so these cases pin that switch at full size.
LIVE_BLOCKS = [0, 3, 4, 39, 40, 49]
FULL_ROWS = [0, 1, 53, 54, 127, 128, 5000, 9719, 9720, 10231, 10232, 10487]
RED_ROWS = [0, 26, 27, 2000, 4859, 4860, 5371, 5372, 5627]


@pytest.mark.parametrize("reduce", [False, True])
@pytest.mark.parametrize("live", LIVE_BLOCKS)
def test_step_864_single_live_block(reduce, live):
    w = synth.WORKLOADS["step_864_tr" if reduce else "step_864"]
    n = w.n_tokens
    nb = w.n_blocks
    after, before = w.reduction if reduce else (None, None)
    shape = shape_of(w)
    devs = [synth.device_block_weights(w.d, w.ffn, seed=w.seed, block=b) for b in range(nb)]
    mods = synth.device_mods(nb, w.d, seed=w.seed)
    gates = torch.zeros((nb, w.d), device="cuda")
    mods[:, 2] = gates
    mods[:, 5] = gates
    g = torch.Generator(device="cuda")
    g.manual_seed(4242 + live)
    mods[live, 2] = torch.randn(w.d, device="cuda", generator=g) * 0.5
    mods[live, 5] = torch.randn(w.d, device="cuda", generator=g) * 0.5
    x = synth.device_activations(n, w.d, seed=w.seed)
    x_in = host(x)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    T, Hh, W = w.video
    tr = H.reduction(H.video_grid(0, T, Hh, W), after, before) if reduce else None
    nbytes = H.h3dit_workspace_size(shape, n, tr)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_step_forward(shape, [_bw(d) for d in devs], mods, x, dev_f32(pos), n, tr, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(x)
    del ws
    cfg = oracle_cfg(w)
    wl = _host_w(devs[live])
    ml = host(mods[live])
    del devs
    torch.cuda.empty_cache()
    in_reduced = reduce and after < live < before
    if not in_reduced:
        # before the reduction, or after the restore: the reduce / restore
        # pair with no update in between gives back the side copy bit for
        # bit, so the step output is the live block on the full stream
        rows = FULL_ROWS
        ref = O.block_forward(x_in, wl, ml, pos, cfg, rows=rows)
        ref_bf = O.block_forward(x_in, wl, ml, pos, cfg, rows=rows, bf16_storage=True)
        assert_block(got[rows], x_in[rows], ref, ref_bf)
        assert np.isfinite(got).all()
        return
    g = O.VideoGrid(0, T, Hh, W)
    pos_red = O.reduced_positions(pos, g)
    wr = (W + 1) // 2
    refs = []
    for storage in (False, True):
        x_red, _ = O.token_reduce(x_in, g, bf16_storage=storage)
        y = O.block_forward(x_red, wl, ml, pos_red, cfg, rows=RED_ROWS, bf16_storage=storage)
        full_rows, ref_rows = [], []
        for p, yp in zip(RED_ROWS, y):
            if p < T * Hh * wr:
                i0 = (p // wr) * W + 2 * (p % wr)
                for i in (i0, i0 + 1):
                    full_rows.append(i)
                    v = x_in[i] + (yp - x_red[p])
                    ref_rows.append(O.bf16_round(v) if storage else v)
            else:
                i = p + T * Hh * (W - wr)
                full_rows.append(i)
                ref_rows.append(yp)
        refs.append(np.stack(ref_rows))
    assert_block(got[full_rows], x_in[full_rows], refs[0], refs[1], roundings=2)
