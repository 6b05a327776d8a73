"""Parity of the dynamic-int8 path on the GPU through the C ABI against the
oracle ([linlog] "int8 量化：从 36 秒到 19 秒").

* Integer work is bit-exact: the int32 accumulators of the int8 projection
  (random codes, codes at the +-127 extremes where every 1024-column chunk
  comes within 2^18 of the 2^24 fp32-exactness bound, and mixes of large and
  +-1 products whose low bits a lossy accumulator would drop), the
  quantiser's codes and scales, the widening of int8 codes, and the codes the
  fused AdaLN + quantise kernels emit for the BF16 h the plain AdaLN gives.
* Dequantised projections (per-token scales; FC2's one scale per 1024
  channels) are within relative L2 <= 2e-3 of the oracle's identical scheme
  fed the same codes and scales: the only difference is the fp32 scaling and
  one BF16 rounding of the output (<= 2^-9 relative per element).
* The whole int8 block against the oracle's int8 block (same quantisation
  scheme, BF16 storage points): the per-block acceptance bounds of the BF16
  block.  The two sides round h, o, h2 and u independently before
  quantising, so a code can differ by one where a value sits at a rounding
  boundary; the block bound covers that.
"""
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth
from tests.gpu_util import dev_bf16, dev_f32, host, max_abs, oracle_cfg, rel_l2, shape_of
from tests.test_gpu_block import assert_block

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_block"]


def codes_dev(q: np.ndarray) -> torch.Tensor:
    """int8 codes -> device operand form (BF16 values of the same integers)."""
    return torch.from_numpy(np.ascontiguousarray(q, np.float32)).to("cuda").to(torch.bfloat16)


def exact_acc(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return O.gemm_int(a, b)


def gpu_acc(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    m, k = a.shape
    n = b.shape[0]
    acc = torch.empty((m, n), device="cuda", dtype=torch.int32)
    H.h3dit_linear_i8_acc(codes_dev(a), codes_dev(b), m, n, k, acc)
    H.h3dit_check_device_error()
    return acc.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("m,n,k", [(1, 256, 64), (129, 256, 1024), (300, 512, 1088),
                                   (200, 256, 5120), (77, 256, 20480), (1000, 768, 2048)])
def test_acc_bit_exact_random(m, n, k):
    a = synth.host_int8((m, k), seed=m, stream=1)
    b = synth.host_int8((n, k), seed=n, stream=2)
    got = gpu_acc(a, b)
    assert np.array_equal(got, exact_acc(a, b))


def test_acc_bit_exact_extremes():
    """Every 1024-column chunk of row 0 sums to 127^2 * 1024 = 16516096, of
    row 1 to -16516096; rows 2-3 put +-1 products after 1000 products of
    127^2 (a partial sum of 16129000, where an accumulator keeping fewer than
    24 significant bits would drop the ones); rows 4+ are random signs of
    +-127 against +-127 and +-1."""
    k, n, m = 5120, 256, 160
    a = np.full((m, k), 127, np.int8)
    b = np.full((n, k), 127, np.int8)
    a[1] = -127
    for r in (2, 3):
        for c0 in range(0, k, 1024):
            a[r, c0 + 1000:c0 + 1024] = 1 if r == 2 else -1
    b[1::2, :] = -127
    for c0 in range(0, k, 1024):
        b[2::4, c0 + 1000:c0 + 1024] = 1
    rs = synth.host_int8((m - 4, k), seed=7, stream=3, lo=-1, hi=1)
    a[4:] = np.where(rs >= 0, 127, -127).astype(np.int8)
    a[4:, ::7] = np.where(rs[:, ::7] > 0, 1, -1).astype(np.int8)
    got = gpu_acc(a, b)
    ref = exact_acc(a, b)
    assert abs(int(ref[0, 0])) == 5 * 16516096
    assert np.array_equal(got, ref)


def _dequant_case(m, n, k, group, act, seed):
    a = synth.host_int8((m, k), seed=seed, stream=4)
    b = synth.host_int8((n, k), seed=seed, stream=5)
    ng = k // group
    sa = synth.host_uniform((m, ng), seed=seed, stream=6, lo=1e-3, hi=3e-2)
    sb = synth.host_uniform((n,), seed=seed, stream=7, lo=1e-4, hi=2e-3)
    c = torch.empty((m, n), device="cuda", dtype=torch.bfloat16)
    H.h3dit_linear_i8(codes_dev(a), dev_f32(sa), group, codes_dev(b), dev_f32(sb), m, n, k, act, c)
    H.h3dit_check_device_error()
    if group == k:
        ref = O.linear_int8(a, sa[:, 0], b, sb)
    else:
        ref = O.fc2_int8(a, sa, b, sb, group)
    if act:
        ref = O.gelu_tanh(ref)
    return host(c), O.bf16_round(ref)


@pytest.mark.parametrize("m,n,k,act", [(129, 256, 1024, 0), (300, 512, 5120, 0), (77, 256, 256, 1),
                                       (256, 768, 2048, 1)])
def test_linear_i8_per_token(m, n, k, act):
    got, ref = _dequant_case(m, n, k, k, act, seed=m + k)
    assert rel_l2(got, ref) <= 2e-3
    assert max_abs(got, ref) <= 2.0 ** -8 * float(np.max(np.abs(ref))) + 1e-6


@pytest.mark.parametrize("m,n,k,group", [(129, 256, 4096, 1024), (300, 256, 20480, 1024),
                                         (64, 512, 1024, 256)])
def test_linear_i8_grouped(m, n, k, group):
    got, ref = _dequant_case(m, n, k, group, 0, seed=m + group)
    assert rel_l2(got, ref) <= 2e-3
    assert max_abs(got, ref) <= 2.0 ** -8 * float(np.max(np.abs(ref))) + 1e-6


@pytest.mark.parametrize("rows,cols,group", [(64, 1024, 1024), (37, 4096, 1024), (5, 256, 256), (9, 5120, 5120),
                                             (7, 1536, 768)])
def test_quantize_codes_bit_exact(rows, cols, group):
    x = synth.host_activations(rows, cols, seed=rows) * np.float32(3.0)
    x = synth.to_bf16_values(x)
    x[1, :group] = 0.0                       # an all-zero group
    xd = dev_bf16(x)
    q = torch.empty_like(xd)
    s = torch.empty((rows, cols // group), device="cuda", dtype=torch.float32)
    H.h3dit_quantize_codes(xd, rows, cols, group, q, s)
    qr, sr = O.quantize_rows(x, group)
    assert np.array_equal(host(q).astype(np.int64), qr.astype(np.int64))
    assert np.array_equal(s.cpu().numpy(), sr)
    # in place gives the same codes
    s2 = torch.empty_like(s)
    H.h3dit_quantize_codes(xd, rows, cols, group, xd, s2)
    H.h3dit_check_device_error()
    assert np.array_equal(host(xd).astype(np.int64), qr.astype(np.int64))
    assert np.array_equal(s2.cpu().numpy(), sr)


def _quotient_dense_rows(amaxes, cols, seed):
    """One row per amax: amax and -amax, then BF16 values in
    (amax * 2^-9, amax] of both signs, so the quotients x / s are dense.  With
    amax = 127 * 2^e the scale is 2^e and every x = (k + 1/2) * 2^e is an
    exact tie; other amax values put many quotients next to half-integers."""
    rng = np.random.default_rng(seed)
    bits = np.arange(0x0080, 0x7F80, dtype=np.uint32)     # positive normal BF16 values
    vals = (bits << 16).view(np.float32)
    half = cols // 2 - 1
    rows = []
    for a in amaxes:
        cand = vals[(vals <= a) & (vals > a * np.float32(2.0 ** -9))]
        pick = rng.choice(cand, size=half, replace=len(cand) < half)
        rows.append(rng.permutation(np.concatenate([[a, -a], pick, -pick])))
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("cols,group", [(1024, 1024), (2048, 2048), (1024, 256)])
def test_quantize_ties_and_near_ties_bit_exact(cols, group):
    """The quantisers form x / s as x times the reciprocal of s and fall back
    to the division within 1e-4 of a half-integer; exact ties (round half to
    even) and near-ties must give the oracle's codes, through the one-warp
    (group <= 1024) and one-CTA (larger groups) kernels, int8 and BF16 codes,
    and for a scale too small for a normal reciprocal."""
    amaxes = [np.float32(v) for v in O.bf16_round(
        np.array([127.0, 15.875, 127.0 * 2 ** -20, 96.0, 100.0, 1.0, 0.3, 5e-3, 3.3e38, 1e-30]))]
    x = _quotient_dense_rows(amaxes, cols, seed=cols + group)
    rows = x.shape[0]
    qr, sr = O.quantize_rows(x, group)
    xd = dev_bf16(x)
    q8 = torch.empty((rows, cols), device="cuda", dtype=torch.int8)
    s8 = torch.empty((rows, cols // group), device="cuda", dtype=torch.float32)
    H.h3dit_quantize_act(xd, rows, cols, group, q8, s8)
    q16 = torch.empty_like(xd)
    s16 = torch.empty_like(s8)
    H.h3dit_quantize_codes(xd, rows, cols, group, q16, s16)
    H.h3dit_check_device_error()
    assert np.array_equal(q8.cpu().numpy(), qr)
    assert np.array_equal(host(q16).astype(np.int64), qr.astype(np.int64))
    assert np.array_equal(s8.cpu().numpy(), sr) and np.array_equal(s16.cpu().numpy(), sr)
    # the rows with power-of-two scales hold exact ties, so round-half-even decided some codes
    exact = (x[:3] / sr[:3].repeat(group, axis=1)) % 1.0 == 0.5
    assert exact.sum() > 100


def test_widen_codes_exact():
    q = synth.host_int8((1000, 64), seed=3, stream=9)
    qd = torch.from_numpy(q).to("cuda")
    out = torch.empty(q.shape, device="cuda", dtype=torch.bfloat16)
    H.h3dit_widen_codes(qd, q.size, out)
    H.h3dit_check_device_error()
    assert np.array_equal(host(out).astype(np.int64), q.astype(np.int64))


@pytest.mark.parametrize("n", [256, 33])
def test_adaln_quant_codes_match_quantised_adaln(n):
    w = TINY
    shape = shape_of(w, H.INT8)
    x = synth.host_activations(n, w.d, seed=4)
    mod = synth.host_mod(w.d, seed=4)
    xd = dev_bf16(x)
    h = torch.empty_like(xd)
    H.h3dit_adaln(shape, xd, dev_f32(mod[0]), dev_f32(mod[1]), n, h)
    hq = torch.empty_like(xd)
    hs = torch.empty(n, device="cuda", dtype=torch.float32)
    H.h3dit_adaln_quant(shape, xd, dev_f32(mod[0]), dev_f32(mod[1]), n, hq, hs)
    H.h3dit_check_device_error()
    qr, sr = O.quantize_rows(host(h))
    assert np.array_equal(host(hq).astype(np.int64), qr.astype(np.int64))
    assert np.array_equal(hs.cpu().numpy(), sr[:, 0])
    # and the BF16 h itself is the oracle's AdaLN to one BF16 rounding
    ref = O.adaln(x, mod[0], mod[1], w.eps)
    assert max_abs(host(h), ref) <= 2.0 ** -8 * float(np.max(np.abs(ref))) + 1e-6


def test_gate_residual_adaln_quant():
    w = TINY
    n = 200
    shape = shape_of(w, H.INT8)
    x = synth.host_activations(n, w.d, seed=5)
    br = synth.host_activations(n, w.d, seed=6)
    mod = synth.host_mod(w.d, seed=5, std=0.5)
    gate, shift, scale = (dev_f32(mod[i]) for i in (2, 3, 4))
    x_plain = dev_bf16(x)
    h = torch.empty_like(x_plain)
    H.h3dit_gate_residual_adaln(shape, x_plain, dev_bf16(br), gate, shift, scale, n, h)
    x_q = dev_bf16(x)
    hq = torch.empty_like(x_q)
    hs = torch.empty(n, device="cuda", dtype=torch.float32)
    H.h3dit_gate_residual_adaln_quant(shape, x_q, dev_bf16(br), gate, shift, scale, n, hq, hs)
    H.h3dit_check_device_error()
    assert torch.equal(x_plain, x_q)
    qr, sr = O.quantize_rows(host(h))
    assert np.array_equal(host(hq).astype(np.int64), qr.astype(np.int64))
    assert np.array_equal(hs.cpu().numpy(), sr[:, 0])


def _int8_weights(wt):
    """Per-output-channel int8 weights of the BF16 block weights (the
    oracle's quantiser), as host codes/scales and device operand form."""
    hw, dev = {}, {}
    for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"), ("w2", "q2", "s2")):
        q, s = O.quantize_weight(wt[name])
        hw[qn], hw[sn] = q, s[:, 0]
        dev[qn], dev[sn] = codes_dev(q), dev_f32(s[:, 0])
    bw = H.block_weights(dev["q_qkv"], dev["q_o"], dev["q1"], dev["q2"], dev["s_qkv"], dev["s_o"], dev["s1"], dev["s2"])
    return hw, dev, bw


def test_qkv_project_i8():
    w = TINY
    n = 256
    shape = shape_of(w, H.INT8)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    wt = synth.host_block_weights(w.d, w.ffn, seed=8)
    hw, dev, _ = _int8_weights(wt)
    h = synth.host_activations(n, w.d, seed=8)
    hq, hs = O.quantize_rows(h)
    table = torch.empty((n, w.head_dim // 2, 2), device="cuda", dtype=torch.float32)
    H.h3dit_rope_table(shape, dev_f32(pos), n, table)
    vt_ld = 256
    q = torch.empty((w.heads, n, w.head_dim), device="cuda", dtype=torch.bfloat16)
    k = torch.empty_like(q)
    vt = torch.empty((w.heads, w.head_dim, vt_ld), device="cuda", dtype=torch.bfloat16)
    H.h3dit_qkv_project_i8(shape, codes_dev(hq), dev_f32(hs[:, 0]), dev["q_qkv"], dev["s_qkv"], table, n,
                           q, k, vt, vt_ld)
    H.h3dit_check_device_error()
    cfg = oracle_cfg(w)
    qkv = O.linear_int8(hq, hs[:, 0], hw["q_qkv"], hw["s_qkv"])
    d = w.d
    tok = lambda t: t.reshape(n, w.heads, w.head_dim)     # [N, H, Dh]
    rq = O.apply_rope(tok(qkv[:, :d]), pos, cfg).transpose(1, 0, 2)
    rk = O.apply_rope(tok(qkv[:, d:2 * d]), pos, cfg).transpose(1, 0, 2)
    rv = tok(qkv[:, 2 * d:]).transpose(1, 2, 0)
    for got, ref in ((host(q), rq), (host(k), rk), (host(vt)[:, :, :n], rv)):
        assert rel_l2(got, ref) <= 2e-3
        assert max_abs(got, ref) <= 2.0 ** -8 * float(np.max(np.abs(ref))) + 1e-6


def _run_int8_block(w, x, bw, mod, pos, n):
    shape = shape_of(w, H.INT8)
    xd = dev_bf16(x)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_block_forward(shape, bw, dev_f32(mod), xd, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    return host(xd)


@pytest.mark.parametrize("n,std", [(256, 1.0), (129, 1.0), (256, 4.0)])
def test_int8_block_tiny(n, std):
    w = TINY
    pos = synth.positions(w.video, w.n_text, w.n_audio)[:n]
    x = synth.host_activations(n, w.d, seed=11)
    wt = synth.host_block_weights(w.d, w.ffn, seed=11)
    mod = synth.host_mod(w.d, seed=11, std=0.1 * std)
    hw, _, bw = _int8_weights(wt)
    got = _run_int8_block(w, x, bw, mod, pos, n)
    cfg = oracle_cfg(w)
    ref_bf = O.block_forward_int8(x, hw, mod, pos, cfg, bf16_storage=True)
    ref64 = O.block_forward_int8(x, hw, mod, pos, cfg, bf16_storage=False)
    assert_block(got, x, ref64, ref_bf)


def test_int8_block_zero_gates_identity():
    w = TINY
    n = w.n_tokens
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=12)
    wt = synth.host_block_weights(w.d, w.ffn, seed=12)
    mod = synth.host_mod(w.d, seed=12)
    mod[2] = 0.0
    mod[5] = 0.0
    _, _, bw = _int8_weights(wt)
    got = _run_int8_block(w, x, bw, mod, pos, n)
    assert np.array_equal(got, x)


def test_int8_step_of_one_block_equals_block_and_chains():
    w = TINY
    n = w.n_tokens
    shape = shape_of(w, H.INT8)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=13)
    nb = 3
    wts = [synth.host_block_weights(w.d, w.ffn, seed=13, block=b) for b in range(nb)]
    mods = np.stack([synth.host_mod(w.d, seed=13, block=b) for b in range(nb)])
    packs = [_int8_weights(wt) for wt in wts]
    # step of nb blocks vs nb block calls: bit-identical (the fused hand-over
    # of the next AdaLN codes is the same arithmetic as the separate AdaLN)
    xs = dev_bf16(x)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_step_forward(shape, [p[2] for p in packs], dev_f32(mods), xs, dev_f32(pos), n, None, ws, nbytes)
    xb = dev_bf16(x)
    for b in range(nb):
        H.h3dit_block_forward(shape, packs[b][2], dev_f32(mods[b]), xb, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    assert torch.equal(xs, xb)
    # and the chain follows the oracle's int8 step
    cfg = oracle_cfg(w)
    ref_bf = x.astype(np.float64)
    ref64 = x.astype(np.float64)
    for b in range(nb):
        ref_bf = O.block_forward_int8(ref_bf, packs[b][0], mods[b], pos, cfg, bf16_storage=True)
        ref64 = O.block_forward_int8(ref64, packs[b][0], mods[b], pos, cfg, bf16_storage=False)
    got = host(xs)
    assert rel_l2(got, ref_bf) <= 1e-2 * nb
    assert rel_l2(got - x, ref_bf - x) <= 2e-2 * nb


def _mixed_weights(wt, which):
    """Device weights for a block whose projections in ``which`` are int8
    (operand-form codes + scales) and the rest BF16; host dict with both
    forms for the oracle."""
    names = {"qkv": ("w_qkv", "q_qkv", "s_qkv"), "o": ("w_o", "q_o", "s_o"), "fc1": ("w1", "q1", "s1"),
             "fc2": ("w2", "q2", "s2")}
    hw = dict(wt)
    ptrs, scales, keep = [], [], []
    for key in ("qkv", "o", "fc1", "fc2"):
        wn, qn, sn = names[key]
        q, s = O.quantize_weight(wt[wn])
        hw[qn], hw[sn] = q, s[:, 0]
        if key in which:
            dw, ds = codes_dev(q), dev_f32(s[:, 0])
        else:
            dw, ds = dev_bf16(wt[wn]), None
        keep += [dw, ds]
        ptrs.append(dw)
        scales.append(ds)
    bw = H.block_weights(*ptrs, *scales)
    return hw, bw, keep


@pytest.mark.parametrize("prec,which", [(H.INT8_MLP, O.INT8_MLP), (H.INT8_QKV, O.INT8_QKV)])
def test_int8_variant_block_tiny(prec, which):
    """The MLP-only and QKV-only int8 blocks against the oracle's block with
    the same projections in int8."""
    w = TINY
    n = w.n_tokens
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=21)
    wt = synth.host_block_weights(w.d, w.ffn, seed=21)
    mod = synth.host_mod(w.d, seed=21)
    hw, bw, keep = _mixed_weights(wt, which)
    shape = shape_of(w, prec)
    xd = dev_bf16(x)
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    H.h3dit_block_forward(shape, bw, dev_f32(mod), xd, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(xd)
    cfg = oracle_cfg(w)
    ref_bf = O.block_forward_int8(x, hw, mod, pos, cfg, bf16_storage=True, which=which)
    ref64 = O.block_forward_int8(x, hw, mod, pos, cfg, bf16_storage=False, which=which)
    assert_block(got, x, ref64, ref_bf)
    # and it is not the full-int8 or the BF16 block
    full = O.block_forward_int8(x, hw, mod, pos, cfg, bf16_storage=True)
    bf = O.block_forward(x, wt, mod, pos, cfg, bf16_storage=True)
    assert rel_l2(got - x, ref_bf - x) < min(rel_l2(got - x, full - x), rel_l2(got - x, bf - x))


@pytest.mark.parametrize("prec", [H.INT8_MLP, H.INT8_QKV])
def test_int8_variant_step_equals_blocks(prec):
    which = O.INT8_MLP if prec == H.INT8_MLP else O.INT8_QKV
    w = TINY
    n = w.n_tokens
    shape = shape_of(w, prec)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=22)
    nb = 3
    packs = [_mixed_weights(synth.host_block_weights(w.d, w.ffn, seed=22, block=b), which) for b in range(nb)]
    mods = np.stack([synth.host_mod(w.d, seed=22, block=b) for b in range(nb)])
    nbytes = H.h3dit_workspace_size(shape, n)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    xs = dev_bf16(x)
    H.h3dit_step_forward(shape, [p[1] for p in packs], dev_f32(mods), xs, dev_f32(pos), n, None, ws, nbytes)
    xb = dev_bf16(x)
    for b in range(nb):
        H.h3dit_block_forward(shape, packs[b][1], dev_f32(mods[b]), xb, dev_f32(pos), n, ws, nbytes)
    H.h3dit_check_device_error()
    assert torch.equal(xs, xb)


def test_int8_step_with_token_reduction():
    """The int8 step through a token reduction: the reduced blocks' AdaLN
    codes come from the reduced stream, and the result follows the oracle's
    int8 step."""
    w = TINY
    n = w.n_tokens
    shape = shape_of(w, H.INT8)
    pos = synth.positions(w.video, w.n_text, w.n_audio)
    x = synth.host_activations(n, w.d, seed=71)
    nb = 3
    wts = [synth.host_block_weights(w.d, w.ffn, seed=71, block=b) for b in range(nb)]
    packs = [_int8_weights(t) for t in wts]
    mods = np.stack([synth.host_mod(w.d, seed=71, block=b) for b in range(nb)])
    T, Hh, W = w.video
    tr = H.reduction(H.video_grid(0, T, Hh, W), 0, 2)
    nbytes = H.h3dit_workspace_size(shape, n, tr)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    xd = dev_bf16(x)
    H.h3dit_step_forward(shape, [p[2] for p in packs], dev_f32(mods), xd, dev_f32(pos), n, tr, ws, nbytes)
    H.h3dit_check_device_error()
    got = host(xd)
    red = O.Reduction(O.VideoGrid(0, T, Hh, W), 0, 2)
    cfg = oracle_cfg(w)
    ref_bf = O.step_forward(x, [p[0] for p in packs], list(mods), pos, cfg, reduction=red, bf16_storage=True,
                            int8=True)
    assert rel_l2(got, ref_bf) <= 1e-2 * nb and rel_l2(got - x, ref_bf - x) <= 2e-2 * nb


def test_int8_weights_as_bytes_equal_operand_form():
    """codes_int8 = 1: the int8 projections' weights stay plain int8 bytes
    (half the resident bytes) and are widened into the workspace before each
    projection; the block and a reduced step give the operand-form results
    bit for bit, for all four projections in int8 and for the MLP alone."""
    w = TINY
    n = w.n_tokens
    pos = dev_f32(synth.positions(w.video, w.n_text, w.n_audio))
    nb = 5
    wts = [synth.host_block_weights(w.d, w.ffn, seed=40, block=b) for b in range(nb)]
    mods = dev_f32(np.stack([synth.host_mod(w.d, seed=40, block=b) for b in range(nb)]))
    x = synth.host_activations(n, w.d, seed=40)
    keep, forms = [], {False: [], True: []}
    for wt in wts:
        dev16, dev8 = {}, {}
        for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"),
                             ("w2", "q2", "s2")):
            q, s = O.quantize_weight(wt[name])
            dev16[qn], dev8[qn] = codes_dev(q), torch.from_numpy(q).to("cuda")
            dev16[sn] = dev8[sn] = dev_f32(s[:, 0])
            dev16[name] = dev8[name] = dev_bf16(wt[name])
        keep += [dev16, dev8]
        for as_bytes, dv in ((False, dev16), (True, dev8)):
            forms[as_bytes].append((dv, as_bytes))
    T, Hh, W = w.video
    tr = H.reduction(H.video_grid(0, T, Hh, W), 1, 3)
    for prec in (H.INT8, H.INT8_MLP):
        shape = shape_of(w, prec)
        outs = {}
        for as_bytes in (False, True):
            bws = []
            for dv, ab in forms[as_bytes]:
                pick = lambda name, qn: dv[qn] if (prec == H.INT8 or name in ("w1", "w2")) else dv[name]
                bws.append(H.block_weights(pick("w_qkv", "q_qkv"), pick("w_o", "q_o"), pick("w1", "q1"),
                                           pick("w2", "q2"), dv["s_qkv"], dv["s_o"], dv["s1"], dv["s2"],
                                           codes_int8=ab))
            nbytes = H.h3dit_workspace_size(shape, n, tr)
            ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
            xb = dev_bf16(x)
            H.h3dit_block_forward(shape, bws[0], mods[0], xb, pos, n, ws, nbytes)
            xs = dev_bf16(x)
            H.h3dit_step_forward(shape, bws, mods, xs, pos, n, tr, ws, nbytes)
            H.h3dit_check_device_error()
            outs[as_bytes] = (xb, xs)
        assert torch.equal(outs[False][0], outs[True][0])
        assert torch.equal(outs[False][1], outs[True][1])
        assert rel_l2(host(outs[True][0]), x) > 1e-3


def test_int8_projection_tail_halves_equal_whole_tiles(monkeypatch):
    """The int8 CTA-pair kernel also runs a short last wave (81 tiles of
    256 x 256) as 256 x 128 halves.  Per-row scales with int32 chunks, the
    raw int32 accumulators, 1024-channel groups and the QKV epilogue give
    the same bits with the split and without it (H3DIT_GEMM_TAIL=0), every
    element written; the int32 accumulators also equal the exact integer
    products."""
    m, n, k = 6900, 768, 2048
    r = np.random.default_rng(81)
    a8 = r.integers(-127, 128, (m, k)).astype(np.int8)
    b8 = r.integers(-127, 128, (n, k)).astype(np.int8)
    ad, bd = codes_dev(a8), codes_dev(b8)
    sa = dev_f32((r.random(m) * 0.01).astype(np.float32))
    sg = dev_f32((r.random((m, k // 1024)) * 0.01).astype(np.float32))
    sb = dev_f32((r.random(n) * 0.01).astype(np.float32))
    outs = {}
    for tail in ("1", "0"):
        monkeypatch.setenv("H3DIT_GEMM_TAIL", tail)
        c1 = torch.full((m, n), float("nan"), device="cuda", dtype=torch.bfloat16)
        H.h3dit_linear_i8(ad, sa, k, bd, sb, m, n, k, 1, c1)
        c2 = torch.full((m, n), float("nan"), device="cuda", dtype=torch.bfloat16)
        H.h3dit_linear_i8(ad, sg, 1024, bd, sb, m, n, k, 0, c2)
        acc = torch.full((m, n), -1, device="cuda", dtype=torch.int32)
        H.h3dit_linear_i8_acc(ad, bd, m, n, k, acc)
        H.h3dit_check_device_error()
        outs[tail] = (c1, c2, acc)
    for x, y in zip(outs["1"], outs["0"]):
        assert torch.equal(x, y)
    rows = np.array([0, 1, 255, 256, 3333, 6655, 6656, 6899])
    exact = a8[rows].astype(np.int64) @ b8.astype(np.int64).T
    assert np.array_equal(outs["1"][2].cpu().numpy()[rows], exact)
    assert not torch.isnan(outs["1"][0].float()).any() and not torch.isnan(outs["1"][1].float()).any()

    # the QKV + RoPE epilogue on half tiles: 6912 tokens, d 512 (162 tiles)
    nt, d, heads, dh = 6912, 512, 4, 128
    shape = H.BlockShape(d, heads, dh, 4 * d, precision=H.INT8)
    hq = codes_dev(r.integers(-127, 128, (nt, d)).astype(np.int8))
    hs = dev_f32((r.random(nt) * 0.01).astype(np.float32))
    wq = codes_dev(r.integers(-127, 128, (3 * d, d)).astype(np.int8))
    ws = dev_f32((r.random(3 * d) * 0.01).astype(np.float32))
    pos = dev_f32(synth.positions((6, 32, 32), 512, 256))
    table = torch.empty((nt, dh // 2, 2), device="cuda", dtype=torch.float32)
    H.h3dit_rope_table(shape, pos, nt, table)
    res = []
    for tail in ("1", "0"):
        monkeypatch.setenv("H3DIT_GEMM_TAIL", tail)
        q = torch.full((heads, nt, dh), float("nan"), device="cuda", dtype=torch.bfloat16)
        kk = torch.full_like(q, float("nan"))
        vt = torch.full((heads, dh, nt), float("nan"), device="cuda", dtype=torch.bfloat16)
        H.h3dit_qkv_project_i8(shape, hq, hs, wq, ws, table, nt, q, kk, vt, nt)
        H.h3dit_check_device_error()
        res.append((q, kk, vt))
    for x, y in zip(*res):
        assert torch.equal(x, y)
        assert not torch.isnan(x.float()).any()


@pytest.mark.parametrize("case", ["acc", "per_token", "per_token_gelu", "grouped"])
def test_int8_pair_and_single_cta_agree_bit_for_bit(monkeypatch, case):
    """The int8 projections on CTA pairs (the default) and on single CTAs
    (H3DIT_GEMM_SINGLE_CTA=1, the A/B reference) add the same exact int32
    chunk sums in the same order and scale them the same way, so every
    epilogue gives identical outputs: the raw accumulators (which also equal
    exact integer arithmetic), per-token dequantisation with and without
    GELU, and FC2's per-group scaling.  Ragged M and a short last wave are
    included."""
    m, n, k = (300, 768, 2048) if case != "grouped" else (129, 512, 4096)
    a = synth.host_int8((m, k), seed=m + 3, stream=8)
    b = synth.host_int8((n, k), seed=n + 3, stream=9)
    group = 1024 if case == "grouped" else k
    sa = synth.host_uniform((m, k // group), seed=m, stream=10, lo=1e-3, hi=3e-2)
    sb = synth.host_uniform((n,), seed=n, stream=11, lo=1e-4, hi=2e-3)
    ad, bd = codes_dev(a), codes_dev(b)
    outs = []
    for single in ("1", "0"):
        monkeypatch.setenv("H3DIT_GEMM_SINGLE_CTA", single)
        if case == "acc":
            c = torch.empty((m, n), device="cuda", dtype=torch.int32)
            H.h3dit_linear_i8_acc(ad, bd, m, n, k, c)
        else:
            c = torch.full((m, n), float("nan"), device="cuda", dtype=torch.bfloat16)
            H.h3dit_linear_i8(ad, dev_f32(sa), group, bd, dev_f32(sb), m, n, k, 1 if case == "per_token_gelu" else 0,
                              c)
        H.h3dit_check_device_error()
        outs.append(c)
    assert torch.equal(outs[0], outs[1])
    if case == "acc":
        assert np.array_equal(outs[1].cpu().numpy().astype(np.int64), exact_acc(a, b))
    else:
        assert not torch.isnan(outs[1].float()).any()
