"""The dynamic-int8 block at full width (d 5120, 40 x 128 heads, F 20480),
run step by step through the C ABI, each step against the oracle fed that
step's GPU input ([linlog] "int8 量化：从 36 秒到 19 秒": dynamic per-token
activation scales, per-output-channel weight scales, one scale per 1024 FC2
input channels).

On 300 tokens (two full 128-row tiles and a ragged tail; video, text and
audio positions), in the order the block runs them:

* weights quantised per output channel on the GPU: codes and scales equal the
  oracle's bit for bit;
* AdaLN-1 + quantise: the codes and scales equal the oracle's quantiser
  applied to the GPU's own BF16 AdaLN output, bit for bit, and that output is
  the oracle's AdaLN to one BF16 rounding;
* QKV (int8) + RoPE, out-projection, FC1 + GELU and FC2 (int8, grouped):
  within relative L2 2e-3 of the oracle's identical scheme fed the same codes
  and scales; attention (BF16) within the single-kernel bound;
* the attention output and the FC1 output quantised per token and per
  (token, 1024 channels): codes and scales bit for bit, so quantising at the
  wrong granularity (a per-token scale where the group scale belongs, or the
  reverse) fails here at full width;
* the gated residuals: bit for bit against the BF16 rounding of x + g * branch;
* finally h3dit_block_forward on the same input equals the stepwise chain
  bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_f32, host, max_abs, oracle_cfg, rel_l2, shape_of

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

W = synth.WORKLOADS["block_512_int8"]
GROUP = 1024


def _codes_host(t):
    return host(t).astype(np.int64)


def _quantize_weight_gpu(wdev):
    """Per-output-channel int8 codes (widened to the BF16 operand form) and
    scales of one weight matrix, made on the GPU."""
    out, inp = wdev.shape
    q8 = torch.empty((out, inp), device="cuda", dtype=torch.int8)
    s = torch.empty((out,), device="cuda", dtype=torch.float32)
    H.h3dit_quantize_weight(wdev, out, inp, q8, s)
    q16 = torch.empty((out, inp), device="cuda", dtype=torch.bfloat16)
    H.h3dit_widen_codes(q8, out * inp, q16)
    return q8, q16, s


def _single_rounding_ok(got, ref):
    return rel_l2(got, ref) <= 5e-3 and max_abs(got, ref) <= 2.0 ** -7 * float(np.max(np.abs(ref))) + 1e-6


def test_int8_block_full_width_stepwise():
    d, F, Hh, Dh = W.d, W.ffn, W.heads, W.head_dim
    shape = shape_of(W, H.INT8)
    cfg = oracle_cfg(W)
    pos_all = synth.positions(W.video, W.n_text, W.n_audio)
    nv = W.n_video
    idx = list(range(0, 200)) + list(range(nv, nv + 50)) + list(range(nv + W.n_text, nv + W.n_text + 50))
    n = len(idx)
    pos = pos_all[idx]
    x_host = synth.host_activations(n, d, seed=31)
    mod = synth.host_mod(d, seed=31)
    shift1, scale1, gate1, shift2, scale2, gate2 = (dev_f32(mod[i]) for i in range(6))

    # ---- weights: quantised on the GPU, checked against the oracle's quantiser
    wdev = synth.device_block_weights(d, F, seed=31, block=0)
    qw, hw = {}, {}
    for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"), ("w2", "q2", "s2")):
        q8, q16, s = _quantize_weight_gpu(wdev[name])
        H.h3dit_check_device_error()
        qr, sr = O.quantize_weight(wdev[name].float().cpu().numpy())
        assert np.array_equal(q8.cpu().numpy(), qr), f"{name} weight codes"
        assert np.array_equal(s.cpu().numpy(), sr[:, 0]), f"{name} weight scales"
        hw[qn], hw[sn] = qr, sr[:, 0]
        qw[qn], qw[sn] = q16, s
        del q8
    del wdev
    torch.cuda.empty_cache()

    x = torch.from_numpy(x_host).to("cuda").to(torch.bfloat16)
    x_keep = x.clone()

    # ---- AdaLN-1 + quantise per token
    h_bf = torch.empty_like(x)
    H.h3dit_adaln(shape, x, shift1, scale1, n, h_bf)
    hq = torch.empty_like(x)
    hs = torch.empty(n, device="cuda", dtype=torch.float32)
    H.h3dit_adaln_quant(shape, x, shift1, scale1, n, hq, hs)
    H.h3dit_check_device_error()
    h_gpu = host(h_bf)
    qr, sr = O.quantize_rows(h_gpu)
    assert np.array_equal(_codes_host(hq), qr.astype(np.int64)), "AdaLN-1 codes"
    assert np.array_equal(hs.cpu().numpy(), sr[:, 0]), "AdaLN-1 scales"
    ref_h = O.adaln(x_host, mod[0], mod[1], W.eps)
    assert max_abs(h_gpu, ref_h) <= 2.0 ** -8 * float(np.max(np.abs(ref_h))) + 1e-6

    # ---- QKV (int8) with RoPE
    table = torch.empty((n, Dh // 2, 2), device="cuda", dtype=torch.float32)
    H.h3dit_rope_table(shape, dev_f32(pos), n, table)
    vt_ld = (n + 63) // 64 * 64
    q = torch.empty((Hh, n, Dh), device="cuda", dtype=torch.bfloat16)
    k = torch.empty_like(q)
    vt = torch.zeros((Hh, Dh, vt_ld), device="cuda", dtype=torch.bfloat16)
    H.h3dit_qkv_project_i8(shape, hq, hs, qw["q_qkv"], qw["s_qkv"], table, n, q, k, vt, vt_ld)
    H.h3dit_check_device_error()
    qkv = O.linear_int8(_codes_host(hq), hs.cpu().numpy(), hw["q_qkv"], hw["s_qkv"])
    tok = lambda t: t.reshape(n, Hh, Dh)
    refs = (O.apply_rope(tok(qkv[:, :d]), pos, cfg).transpose(1, 0, 2),
            O.apply_rope(tok(qkv[:, d:2 * d]), pos, cfg).transpose(1, 0, 2),
            tok(qkv[:, 2 * d:]).transpose(1, 2, 0))
    q_h, k_h, v_h = host(q), host(k), host(vt)[:, :, :n]
    for nm, got, ref in (("q", q_h, refs[0]), ("k", k_h, refs[1]), ("v", v_h, refs[2])):
        assert rel_l2(got, ref) <= 2e-3, f"QKV {nm} rel_l2 {rel_l2(got, ref):.2e}"

    # ---- attention (BF16), fed the GPU's q, k, v
    o = torch.empty((n, d), device="cuda", dtype=torch.bfloat16)
    H.h3dit_attention(shape, q, k, vt, vt_ld, n, o)
    H.h3dit_check_device_error()
    o_gpu = host(o)
    ref_o = O.attention(q_h, k_h, v_h.transpose(0, 2, 1)).transpose(1, 0, 2).reshape(n, d)
    assert _single_rounding_ok(o_gpu, ref_o), f"attention rel_l2 {rel_l2(o_gpu, ref_o):.2e}"

    # ---- o quantised per token, out-projection (int8)
    oq = torch.empty_like(o)
    os_ = torch.empty(n, device="cuda", dtype=torch.float32)
    H.h3dit_quantize_codes(o, n, d, d, oq, os_)
    H.h3dit_check_device_error()
    qr, sr = O.quantize_rows(o_gpu)
    assert np.array_equal(_codes_host(oq), qr.astype(np.int64)), "o codes"
    assert np.array_equal(os_.cpu().numpy(), sr[:, 0]), "o scales"
    a = torch.empty_like(o)
    H.h3dit_linear_i8(oq, os_, d, qw["q_o"], qw["s_o"], n, d, d, 0, a)
    H.h3dit_check_device_error()
    a_gpu = host(a)
    ref_a = O.bf16_round(O.linear_int8(qr, sr[:, 0], hw["q_o"], hw["s_o"]))
    assert rel_l2(a_gpu, ref_a) <= 2e-3, f"out-proj rel_l2 {rel_l2(a_gpu, ref_a):.2e}"

    # ---- gated residual + AdaLN-2 + quantise per token
    x_before = host(x)
    h2_bf = torch.empty_like(x)
    x_copy = x.clone()
    H.h3dit_gate_residual_adaln(shape, x_copy, a, gate1, shift2, scale2, n, h2_bf)
    h2q = torch.empty_like(x)
    h2s = torch.empty(n, device="cuda", dtype=torch.float32)
    H.h3dit_gate_residual_adaln_quant(shape, x, a, gate1, shift2, scale2, n, h2q, h2s)
    H.h3dit_check_device_error()
    x1_gpu = host(x)
    assert torch.equal(x, x_copy)
    assert np.array_equal(x1_gpu, O.bf16_round(x_before + mod[2].astype(np.float64) * a_gpu)), "x1"
    h2_gpu = host(h2_bf)
    qr, sr = O.quantize_rows(h2_gpu)
    assert np.array_equal(_codes_host(h2q), qr.astype(np.int64)), "AdaLN-2 codes"
    assert np.array_equal(h2s.cpu().numpy(), sr[:, 0]), "AdaLN-2 scales"
    ref_h2 = O.adaln(x1_gpu, mod[3], mod[4], W.eps)
    assert max_abs(h2_gpu, ref_h2) <= 2.0 ** -8 * float(np.max(np.abs(ref_h2))) + 1e-6

    # ---- FC1 (int8) + GELU
    u = torch.empty((n, F), device="cuda", dtype=torch.bfloat16)
    H.h3dit_linear_i8(h2q, h2s, d, qw["q1"], qw["s1"], n, F, d, 1, u)
    H.h3dit_check_device_error()
    u_gpu = host(u)
    ref_u = O.bf16_round(O.gelu_tanh(O.linear_int8(qr, sr[:, 0], hw["q1"], hw["s1"])))
    assert rel_l2(u_gpu, ref_u) <= 2e-3, f"FC1 rel_l2 {rel_l2(u_gpu, ref_u):.2e}"

    # ---- u quantised per (token, 1024 channels), FC2 (int8, group scales)
    uq = torch.empty_like(u)
    us = torch.empty((n, F // GROUP), device="cuda", dtype=torch.float32)
    H.h3dit_quantize_codes(u, n, F, GROUP, uq, us)
    H.h3dit_check_device_error()
    uqr, usr = O.quantize_rows(u_gpu, GROUP)
    assert np.array_equal(_codes_host(uq), uqr.astype(np.int64)), "u codes"
    assert np.array_equal(us.cpu().numpy(), usr), "u group scales"
    # a per-token scale would not do: the groups of a row do differ
    assert np.mean(usr.min(axis=1) < 0.9 * usr.max(axis=1)) > 0.5
    m = torch.empty_like(x)
    H.h3dit_linear_i8(uq, us, GROUP, qw["q2"], qw["s2"], n, d, F, 0, m)
    H.h3dit_check_device_error()
    m_gpu = host(m)
    rows = list(range(0, 8)) + [63, 64, 127, 128, 129, 199, 200, 225, 249, 250, 251, 275, 298, 299]
    ref_m = O.bf16_round(O.fc2_int8(uqr[rows], usr[rows], hw["q2"], hw["s2"], GROUP))
    assert rel_l2(m_gpu[rows], ref_m) <= 2e-3, f"FC2 rel_l2 {rel_l2(m_gpu[rows], ref_m):.2e}"

    # ---- final gated residual
    H.h3dit_gate_residual_adaln(shape, x, m, gate2, None, None, n, None)
    H.h3dit_check_device_error()
    x2_gpu = host(x)
    assert np.array_equal(x2_gpu, O.bf16_round(x1_gpu + mod[5].astype(np.float64) * m_gpu)), "x2"

    # ---- the fused block entry point gives the stepwise chain bit for bit
    bw = H.block_weights(qw["q_qkv"], qw["q_o"], qw["q1"], qw["q2"], qw["s_qkv"], qw["s_o"], qw["s1"], qw["s2"])
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_block_forward(shape, bw, dev_f32(mod), x_keep, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    assert torch.equal(x_keep, x)
