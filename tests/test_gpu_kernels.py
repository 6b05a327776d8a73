"""Kernel-level parity on the GPU: every step of the block through the C ABI
against the fp64 oracle on the same seeded inputs, at sizes spanning several
tiles with ragged tails.

Tolerances (fp32 accumulation, BF16 storage): a stored BF16 value carries a
relative rounding error of at most 2^-9, so single-step outputs are held to
relative L2 <= 5e-3 and max-abs <= 2^-7 of the reference's max magnitude
(plus the accumulation error of fp32 over K terms, far below that).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_bf16, dev_f32, host, max_abs, oracle_cfg, rel_l2, shape_of

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_block"]


def _close(got, ref, rel=5e-3, amax_frac=2.0 ** -7):
    r = rel_l2(got, ref)
    m = max_abs(got, ref)
    bound = amax_frac * float(np.max(np.abs(ref))) + 1e-6
    assert r <= rel and m <= bound, f"rel_l2={r:.3e} (<= {rel}) max_abs={m:.3e} (<= {bound:.3e})"


@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (1, 256, 64), (7, 512, 128), (129, 256, 320),
                                   (300, 768, 256), (1000, 1024, 512)])
@pytest.mark.parametrize("act", [0, 1])
def test_linear(m, n, k, act):
    a = synth.host_activations(m, k, seed=m * 7 + k)
    b = synth.to_bf16_values(synth.host_uniform((n, k), 5, n + k, -0.1, 0.1))
    c = torch.empty((m, n), device="cuda", dtype=torch.bfloat16)
    H.h3dit_linear(dev_bf16(a), dev_bf16(b), m, n, k, act, c)
    torch.cuda.synchronize()
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    if act:
        ref = O.gelu_tanh(ref)
    _close(host(c), ref)


def test_linear_rejects_bad_shapes():
    a = torch.zeros((4, 64), device="cuda", dtype=torch.bfloat16)
    b = torch.zeros((100, 64), device="cuda", dtype=torch.bfloat16)
    c = torch.zeros((4, 100), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_linear(a, b, 4, 100, 64, 0, c)
    assert e.value.status == H.E_UNSUPPORTED


@pytest.mark.parametrize("n", [256, 77, 1])
def test_rope_table_and_qkv_project(n):
    w = TINY
    shape = shape_of(w)
    cfg = oracle_cfg(w)
    pos = synth.positions(w.video, w.n_text, w.n_audio)[:n]
    if n < len(pos):
        pos = pos + np.float32(0.25)   # off-grid positions
    h = synth.host_activations(n, w.d, seed=11)
    wt = synth.host_block_weights(w.d, w.ffn, seed=3)
    table = torch.empty((n, w.head_dim // 2, 2), device="cuda", dtype=torch.float32)
    H.h3dit_rope_table(shape, dev_f32(pos), n, table)
    ang = O.rope_angles(pos, cfg)
    _close(host(table)[..., 0], np.cos(ang), rel=1e-5, amax_frac=1e-5)
    _close(host(table)[..., 1], np.sin(ang), rel=1e-5, amax_frac=1e-5)
    vt_ld = (n + 63) // 64 * 64
    q = torch.empty((w.heads, n, w.head_dim), device="cuda", dtype=torch.bfloat16)
    k = torch.empty_like(q)
    vt = torch.zeros((w.heads, w.head_dim, vt_ld), device="cuda", dtype=torch.bfloat16)
    H.h3dit_qkv_project(shape, dev_bf16(h), dev_bf16(wt["w_qkv"]), table, n, q, k, vt, vt_ld)
    torch.cuda.synchronize()
    qkv = h.astype(np.float64) @ wt["w_qkv"].astype(np.float64).T
    d = w.d
    split = lambda t: t.reshape(n, w.heads, w.head_dim)
    q_ref = O.apply_rope(split(qkv[:, :d]), pos, cfg).transpose(1, 0, 2)
    k_ref = O.apply_rope(split(qkv[:, d:2 * d]), pos, cfg).transpose(1, 0, 2)
    v_ref = split(qkv[:, 2 * d:]).transpose(1, 2, 0)     # [H][Dh][n]
    _close(host(q), q_ref)
    _close(host(k), k_ref)
    _close(host(vt)[:, :, :n], v_ref)


@pytest.mark.parametrize("dh", [64, 128])
@pytest.mark.parametrize("n", [1, 100, 256, 300])
def test_attention(dh, n):
    heads = 2
    shape = H.BlockShape(heads * dh, heads, dh, 256, rope_sections=(dh // 4, 3 * dh // 8, 3 * dh // 8))
    r = np.random.default_rng(100 + n + dh)
    q = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32) * 1.5)
    k = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32) * 1.5)
    v = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32))
    vt_ld = (n + 63) // 64 * 64
    vt = np.zeros((heads, dh, vt_ld), np.float32)
    vt[:, :, :n] = v.transpose(0, 2, 1)
    o = torch.empty((n, heads * dh), device="cuda", dtype=torch.bfloat16)
    H.h3dit_attention(shape, dev_bf16(q), dev_bf16(k), dev_bf16(vt), vt_ld, n, o)
    H.h3dit_check_device_error()
    ref = O.attention(q, k, v).transpose(1, 0, 2).reshape(n, heads * dh)
    _close(host(o), ref, rel=1e-2, amax_frac=2.0 ** -6)


@pytest.mark.parametrize("mixed", [False, True])
def test_attention_large_logits_rescale(mixed):
    """Keys whose scores grow along the sequence force the running max to be
    raised (and O rescaled) at every tile.  ``mixed``: only every other query
    row sees the growth (the others score every key near 0), so within one
    warp some rows redo a tile with a new max while the rest keep theirs."""
    heads, dh, n = 1, 128, 1024
    shape = H.BlockShape(heads * dh, heads, dh, 256)
    r = np.random.default_rng(7)
    q = np.zeros((heads, n, dh), np.float32)
    q[..., 0] = 1.0
    if mixed:
        q[:, 1::2, 0] = 0.0
        q[:, 1::2, 1:] = r.standard_normal((heads, n // 2, dh - 1)).astype(np.float32)
    k = r.standard_normal((heads, n, dh)).astype(np.float32) * 0.1
    k[..., 0] = np.linspace(0, 1000, n, dtype=np.float32)   # scaled score rises ~16 (log2) per tile
    q, k = synth.to_bf16_values(q), synth.to_bf16_values(k)
    v = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32))
    vt = np.ascontiguousarray(v.transpose(0, 2, 1))
    o = torch.empty((n, dh), device="cuda", dtype=torch.bfloat16)
    H.h3dit_attention(shape, dev_bf16(q), dev_bf16(k), dev_bf16(vt), n, n, o)
    H.h3dit_check_device_error()
    ref = O.attention(q, k, v).transpose(1, 0, 2).reshape(n, dh)
    _close(host(o), ref, rel=1e-2, amax_frac=2.0 ** -6)


@pytest.mark.parametrize("n", [256, 5])
def test_adaln_and_gated_residual(n):
    w = TINY
    shape = shape_of(w)
    x = synth.host_activations(n, w.d, seed=21)
    br = synth.host_activations(n, w.d, seed=22)
    mod = synth.host_mod(w.d, seed=23)
    xd = dev_bf16(x)
    h = torch.empty_like(xd)
    H.h3dit_adaln(shape, xd, dev_f32(mod[0]), dev_f32(mod[1]), n, h)
    torch.cuda.synchronize()
    _close(host(h), O.adaln(x, mod[0], mod[1], w.eps), rel=5e-3)
    H.h3dit_gate_residual_adaln(shape, xd, dev_bf16(br), dev_f32(mod[2]), dev_f32(mod[3]), dev_f32(mod[4]), n, h)
    torch.cuda.synchronize()
    x1_ref = O.bf16_round(x.astype(np.float64) + mod[2].astype(np.float64) * br)
    # the stored residual is the fp32 result rounded once: within one BF16 step
    assert max_abs(host(xd), x1_ref) <= 2.0 ** -8 * float(np.max(np.abs(x1_ref)))
    _close(host(h), O.adaln(host(xd), mod[3], mod[4], w.eps), rel=5e-3)


_FUSION_SCRIPT = r"""
import sys, hashlib, numpy as np, torch
sys.path.insert(0, sys.argv[1])
from audio_diffusion_transformer_fwd_b300 import h3dit as H, synth
from tests.gpu_util import dev_bf16, dev_f32, shape_of
w = synth.WORKLOADS["tiny_block"]
x = dev_bf16(synth.host_activations(256, w.d, seed=31))
br = dev_bf16(synth.host_activations(256, w.d, seed=32))
mod = synth.host_mod(w.d, seed=33)
h = torch.empty_like(x)
H.h3dit_gate_residual_adaln(shape_of(w), x, br, dev_f32(mod[2]), dev_f32(mod[3]), dev_f32(mod[4]), 256, h)
torch.cuda.synchronize()
print(hashlib.sha256(x.view(torch.int16).cpu().numpy().tobytes() + h.view(torch.int16).cpu().numpy().tobytes()).hexdigest())
"""


def test_gated_adaln_fusion_is_bit_identical_to_stepwise():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for flag in ("0", "1"):
        env = dict(os.environ, H3DIT_DISABLE_GATED_ADALN=flag)
        r = subprocess.run([sys.executable, "-c", _FUSION_SCRIPT, root], env=env, capture_output=True, text=True,
                           timeout=300)
        assert r.returncode == 0, r.stderr
        outs.append(r.stdout.strip().splitlines()[-1])
    assert outs[0] == outs[1]


@pytest.mark.parametrize("rows,cols,group", [(5, 256, 256), (33, 2048, 1024), (4, 64, 8)])
def test_quantize_bit_exact(rows, cols, group):
    x = synth.host_activations(rows, cols, seed=rows + cols) * np.float32(3.0)
    x = synth.to_bf16_values(x)
    x[1, :group] = 0.0          # an all-zero group
    q = torch.empty((rows, cols), device="cuda", dtype=torch.int8)
    s = torch.empty((rows, cols // group), device="cuda", dtype=torch.float32)
    H.h3dit_quantize_act(dev_bf16(x), rows, cols, group, q, s)
    torch.cuda.synchronize()
    qr, sr = O.quantize_rows(x, group)
    assert np.array_equal(q.cpu().numpy(), qr)
    assert np.array_equal(s.cpu().numpy(), sr)


def test_quantize_weight_bit_exact():
    w = synth.host_block_weights(256, 1024, seed=9)["w1"]
    q = torch.empty(w.shape, device="cuda", dtype=torch.int8)
    s = torch.empty((w.shape[0],), device="cuda", dtype=torch.float32)
    H.h3dit_quantize_weight(dev_bf16(w), w.shape[0], w.shape[1], q, s)
    torch.cuda.synchronize()
    qr, sr = O.quantize_weight(w)
    assert np.array_equal(q.cpu().numpy(), qr) and np.array_equal(s.cpu().numpy(), sr[:, 0])


@pytest.mark.parametrize("grid,n_other", [((0, 2, 8, 12), 64), ((3, 2, 3, 5), 4), ((0, 6, 30, 54), 768)])
def test_token_reduce_restore_bit_exact(grid, n_other):
    off, T, Hh, W = grid
    n = off + T * Hh * W + n_other
    d = 256
    x = synth.host_activations(n, d, seed=n)
    g = H.video_grid(off, T, Hh, W)
    og = O.VideoGrid(off, T, Hh, W)
    nr = H.h3dit_reduced_tokens(n, g)
    assert nr == O.reduced_token_count(n, og)
    xd = dev_bf16(x)
    xr = torch.empty((nr, d), device="cuda", dtype=torch.bfloat16)
    side = torch.empty_like(xd)
    H.h3dit_token_reduce(xd, n, d, g, xr, side)
    red_ref, _ = O.token_reduce(x, og, bf16_storage=True)
    torch.cuda.synchronize()
    assert np.array_equal(host(xr), red_ref)
    assert torch.equal(side, xd)
    # zero update: identity, bit for bit (restore in place over the side copy)
    H.h3dit_token_restore(xr, side, n, d, g, side)
    torch.cuda.synchronize()
    assert torch.equal(side, xd)
    # a real update
    upd = synth.host_activations(nr, d, seed=n + 1) * np.float32(0.1)
    xr2 = synth.to_bf16_values(host(xr) + upd)
    out = torch.empty_like(xd)
    H.h3dit_token_restore(dev_bf16(xr2), xd, n, d, g, out)
    torch.cuda.synchronize()
    ref = O.token_restore(xr2, x, og, bf16_storage=True)
    assert max_abs(host(out), ref) <= 2.0 ** -7 * float(np.max(np.abs(ref)))
    assert np.mean(host(out) == ref) > 0.99
    # pair-mean positions
    pos = synth.positions((T, Hh, W), 0, 0)
    pos = np.concatenate([np.zeros((off, 3), np.float32), pos, np.ones((n_other, 3), np.float32)])
    pr = torch.empty((nr, 3), device="cuda", dtype=torch.float32)
    H.h3dit_reduced_positions(dev_f32(pos), n, g, pr)
    torch.cuda.synchronize()
    assert np.array_equal(pr.cpu().numpy(), O.reduced_positions(pos, og).astype(np.float32))


def test_abi_errors():
    shape = H.BlockShape(250, 2, 125, 1000)
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_workspace_size(shape, 10)
    assert e.value.status in (H.E_INVAL, H.E_UNSUPPORTED)
    assert "head" in H.lib().h3dit_last_error().decode() or "d " in H.lib().h3dit_last_error().decode()
    ok = shape_of(TINY)
    assert H.h3dit_workspace_size(ok, 256) > 0
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_block_forward(ok, H.block_weights(None, None, None, None), None, None, None, 256, None, 0)
    assert e.value.status == H.E_INVAL


@pytest.mark.parametrize("m,n,k,act", [(256, 256, 64, 0), (77, 256, 128, 1), (1, 512, 64, 0), (300, 768, 2048, 1),
                                       (1000, 512, 1024, 0), (513, 1024, 5120, 1)])
def test_pair_and_single_cta_projection_agree_bit_for_bit(monkeypatch, m, n, k, act):
    """The CTA-pair projection kernel (two SMs per 256 x 256 tile) and the
    single-CTA kernel (one SM per 128 x 256 tile) add the same products in
    the same order: their outputs are identical, ragged M tails included."""
    r = np.random.default_rng(m + n + k)
    a = dev_bf16(r.standard_normal((m, k)).astype(np.float32))
    b = dev_bf16(r.standard_normal((n, k)).astype(np.float32) * 0.05)
    out = []
    for single in ("1", "0"):
        monkeypatch.setenv("H3DIT_GEMM_SINGLE_CTA", single)
        c = torch.zeros((m, n), device="cuda", dtype=torch.bfloat16)
        H.h3dit_linear(a, b, m, n, k, act, c)
        H.h3dit_check_device_error()
        out.append(c)
    assert torch.equal(out[0], out[1])
    ref = O.bf16_round(host(a) @ host(b).T)
    if act:
        ref = O.bf16_round(O.gelu_tanh(host(a) @ host(b).T))
    assert rel_l2(host(out[1]), ref) <= 5e-3


@pytest.mark.parametrize("act", [0, 1])
def test_projection_tail_halves_equal_whole_tiles(monkeypatch, act):
    """81 tiles of 256 x 256 (27 x 3, ragged M) on the device's CTA pairs
    leave a short last wave, which the pair kernel runs as 256 x 128 halves
    (twice as many pairs busy).  Each output is the same k-ordered sum as in
    a whole tile, so the result equals whole tiles everywhere
    (H3DIT_GEMM_TAIL=0) bit for bit, every element written, and both follow
    the oracle; the single-CTA kernel agrees too."""
    m, n, k = 6900, 768, 320
    r = np.random.default_rng(61 + act)
    a = synth.to_bf16_values(r.standard_normal((m, k)).astype(np.float32))
    b = synth.to_bf16_values(r.standard_normal((n, k)).astype(np.float32) * 0.05)
    ad, bd = dev_bf16(a), dev_bf16(b)
    outs = []
    for tail, single in (("1", "0"), ("0", "0"), ("1", "1")):
        monkeypatch.setenv("H3DIT_GEMM_TAIL", tail)
        monkeypatch.setenv("H3DIT_GEMM_SINGLE_CTA", single)
        c = torch.full((m, n), float("nan"), device="cuda", dtype=torch.bfloat16)
        H.h3dit_linear(ad, bd, m, n, k, act, c)
        H.h3dit_check_device_error()
        outs.append(c)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    if act:
        ref = O.gelu_tanh(ref)
    _close(host(outs[0]), ref)


def test_qkv_projection_tail_halves_equal_whole_tiles(monkeypatch):
    """The QKV epilogue (RoPE, head-major Q/K, transposed V) on half tiles:
    6912 tokens, d 512 (162 tiles, a short last wave) give the same Q, K and
    V^T with and without the split."""
    n, d, heads, dh = 6912, 512, 4, 128
    shape = H.BlockShape(d, heads, dh, 4 * d)
    r = np.random.default_rng(63)
    h = dev_bf16(r.standard_normal((n, d)).astype(np.float32))
    w = dev_bf16(r.standard_normal((3 * d, d)).astype(np.float32) * 0.05)
    pos = dev_f32(synth.positions((6, 32, 32), 512, 256))
    table = torch.empty((n, dh // 2, 2), device="cuda", dtype=torch.float32)
    H.h3dit_rope_table(shape, pos, n, table)
    outs = []
    for tail in ("1", "0"):
        monkeypatch.setenv("H3DIT_GEMM_TAIL", tail)
        q = torch.full((heads, n, dh), float("nan"), device="cuda", dtype=torch.bfloat16)
        k = torch.full_like(q, float("nan"))
        vt = torch.full((heads, dh, n), float("nan"), device="cuda", dtype=torch.bfloat16)
        H.h3dit_qkv_project(shape, h, w, table, n, q, k, vt, n)
        H.h3dit_check_device_error()
        outs.append((q, k, vt))
    for x, y in zip(*outs):
        assert torch.equal(x, y)
        assert not torch.isnan(x.float()).any()


@pytest.mark.parametrize("heads,dh,n", [(40, 128, 1100), (64, 64, 600)])
def test_attention_split_tail_units(monkeypatch, heads, dh, n):
    """More 256-row units than SMs with a short last wave (200 units for
    40 heads x 1100 tokens; 192 for 64 x 600): the last wave's units run as
    CTA pairs that split the keys in two and combine (O, running max, row
    sum) through distributed shared memory.  Every output is written and
    follows the oracle; against whole units (H3DIT_ATTN_SPLIT=0) only the
    combine's rounding differs (within one BF16 step of the output)."""
    shape = H.BlockShape(heads * dh, heads, dh, 256, rope_sections=(dh // 4, 3 * dh // 8, 3 * dh // 8))
    r = np.random.default_rng(900 + n)
    q = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32) * 1.5)
    k = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32) * 1.5)
    v = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32))
    vt_ld = (n + 63) // 64 * 64
    vt = np.zeros((heads, dh, vt_ld), np.float32)
    vt[:, :, :n] = v.transpose(0, 2, 1)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(vt)
    outs = []
    for split in ("1", "0"):
        monkeypatch.setenv("H3DIT_ATTN_SPLIT", split)
        o = torch.full((n, heads * dh), float("nan"), device="cuda", dtype=torch.bfloat16)
        H.h3dit_attention(shape, qd, kd, vd, vt_ld, n, o)
        H.h3dit_check_device_error()
        outs.append(host(o))
    assert not np.isnan(outs[0]).any()
    ref = O.attention(q, k, v).transpose(1, 0, 2).reshape(n, heads * dh)
    for got in outs:
        _close(got, ref, rel=1e-2, amax_frac=2.0 ** -6)
    a, b = outs
    diff = np.abs(a - b)
    i = np.unravel_index(np.argmax(diff), diff.shape)
    assert rel_l2(a, b) <= 2e-3 and diff.max() <= 2.0 ** -7 * float(np.max(np.abs(b))), \
        f"rel_l2 {rel_l2(a, b):.3e}, max diff {diff.max():.3e} at {i}: {a[i]} vs {b[i]}, max|o| {np.max(np.abs(b)):.3e}"


def test_attention_persistent_units_equal_one_cta_per_unit(monkeypatch):
    """50 heads x 1536 tokens = 300 units: the full waves (296 units) run on
    148 persistent CTAs that walk two units each, counting every barrier
    phase on across units; the 4 left over run key-split.  Each output is
    the same computation as with one CTA per unit (H3DIT_ATTN_PERSIST=0),
    bit for bit, and follows the oracle (checked on three heads)."""
    heads, dh, n = 50, 128, 1536
    shape = H.BlockShape(heads * dh, heads, dh, 256)
    r = np.random.default_rng(77)
    q = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32) * 1.5)
    k = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32) * 1.5)
    v = synth.to_bf16_values(r.standard_normal((heads, n, dh)).astype(np.float32))
    vt = np.ascontiguousarray(v.transpose(0, 2, 1))
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(vt)
    outs = []
    for persist in ("1", "0"):
        monkeypatch.setenv("H3DIT_ATTN_PERSIST", persist)
        o = torch.full((n, heads * dh), float("nan"), device="cuda", dtype=torch.bfloat16)
        H.h3dit_attention(shape, qd, kd, vd, n, n, o)
        H.h3dit_check_device_error()
        outs.append(o)
    assert torch.equal(outs[0], outs[1])
    got = host(outs[0]).reshape(n, heads, dh)
    assert not np.isnan(got).any()
    for h in (0, 25, 49):
        ref = O.attention(q[h:h + 1], k[h:h + 1], v[h:h + 1])[0]
        _close(got[:, h], ref, rel=1e-2, amax_frac=2.0 ** -6)
