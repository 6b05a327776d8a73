"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, the wrong variance or GELU form)
fails at least one of them: closed forms, library routines on special cases,
exact rational arithmetic and brute force loops on tiny inputs.
``test_oracle_mutations.py`` plants such slips and checks they are caught.
"""
import math
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import synth

# ------------------------------------------------------------------ bf16 rounding


def test_bf16_round_ties_and_library():
    one = 1.0
    ulp = 2.0 ** -7                        # BF16 spacing in [1, 2)
    assert O.bf16_round(one + ulp / 2) == one                    # tie -> even (1.0)
    assert O.bf16_round(one + 3 * ulp / 2) == one + 2 * ulp      # tie -> even
    assert O.bf16_round(one + ulp / 2 + 2.0 ** -20) == one + ulp  # above the tie
    r = np.random.default_rng(3).standard_normal(10000) * 37.0
    ref = torch.from_numpy(r.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_round(r.astype(np.float32)), ref)


# ------------------------------------------------------------------ LayerNorm / AdaLN


def test_layer_norm_hand_example():
    # mean 2.5, biased variance 1.25 (the unbiased one would be 5/3)
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    eps = 1e-6
    want = (x - 2.5) / math.sqrt(1.25 + eps)
    assert np.allclose(O.layer_norm(x, eps), want, rtol=0, atol=1e-15)


def test_layer_norm_matches_torch():
    x = np.random.default_rng(0).standard_normal((7, 96)) * 3 + 1.5
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (96,), eps=1e-6).numpy()
    assert np.allclose(O.layer_norm(x, 1e-6), ref, rtol=0, atol=1e-12)


def test_adaln_special_cases():
    r = np.random.default_rng(1)
    x = r.standard_normal((5, 64))
    shift = r.standard_normal(64)
    # scale = -1 cancels the normalised row: the output is the shift exactly
    assert np.allclose(O.adaln(x, shift, -np.ones(64), 1e-6), np.broadcast_to(shift, (5, 64)), atol=1e-15)
    # zero shift and zero scale: plain LayerNorm, mean 0 and variance 1 - O(eps)
    y = O.adaln(x, np.zeros(64), np.zeros(64), 1e-6)
    assert np.allclose(y.mean(axis=1), 0, atol=1e-13)
    assert np.allclose((y ** 2).mean(axis=1), 1, atol=1e-5)
    # scale = 1 doubles it
    assert np.allclose(O.adaln(x, np.zeros(64), np.ones(64), 1e-6), 2 * y, atol=1e-13)


# ------------------------------------------------------------------ RoPE

CFG_R = O.BlockConfig(d=256, heads=2, head_dim=128, ffn=64, rope_sections=(32, 48, 48))


def test_rope_identity_at_origin_and_norm():
    r = np.random.default_rng(2)
    t = r.standard_normal((9, 2, 128))
    assert np.allclose(O.apply_rope(t, np.zeros((9, 3)), CFG_R), t, atol=0)
    pos = r.uniform(-50, 300, (9, 3))
    rt = O.apply_rope(t, pos, CFG_R)
    assert np.allclose(np.linalg.norm(rt, axis=-1), np.linalg.norm(t, axis=-1), rtol=1e-13)


def test_rope_relative_position():
    r = np.random.default_rng(4)
    q = r.standard_normal((1, 1, 128))
    k = r.standard_normal((1, 1, 128))
    pm = r.uniform(0, 40, (1, 3))
    pn = r.uniform(0, 40, (1, 3))
    dots = []
    for shift in ([0, 0, 0], [3.5, -7.0, 11.25], [100.0, 2.0, -30.0]):
        a = O.apply_rope(q, pm + shift, CFG_R)
        b = O.apply_rope(k, pn + shift, CFG_R)
        dots.append(float((a * b).sum()))
    assert np.allclose(dots, dots[0], rtol=1e-12)


def test_rope_sections_axes_and_frequencies():
    # a unit vector on pair i of each section turns by exactly pos_axis * theta^(-2i/sec)
    sec = (32, 48, 48)
    starts = (0, 32, 80)
    theta = mpmath.mpf(10000)
    for axis in range(3):
        for i in (0, 1, 5, sec[axis] // 2 - 1):
            dim = starts[axis] + 2 * i
            t = np.zeros((1, 1, 128))
            t[0, 0, dim] = 1.0
            pos = np.zeros((1, 3))
            pos[0, axis] = 17.0
            out = O.apply_rope(t, pos, CFG_R)
            ang = 17 * theta ** (mpmath.mpf(-2 * i) / sec[axis])
            assert abs(out[0, 0, dim] - float(mpmath.cos(ang))) < 1e-13
            assert abs(out[0, 0, dim + 1] - float(mpmath.sin(ang))) < 1e-13
            # only that pair moves; a position on another axis leaves it alone
            rest = np.delete(out[0, 0], [dim, dim + 1])
            assert np.all(rest == 0)
            pos2 = np.zeros((1, 3))
            pos2[0, (axis + 1) % 3] = 17.0
            assert np.allclose(O.apply_rope(t, pos2, CFG_R), t, atol=0)


# ------------------------------------------------------------------ attention


def _attention_loops(q, k, v):
    h_, n, dh = q.shape
    out = np.zeros((h_, n, v.shape[2]))
    for h in range(h_):
        for i in range(n):
            s = [sum(q[h, i, c] * k[h, j, c] for c in range(dh)) / math.sqrt(dh) for j in range(n)]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            for j in range(n):
                out[h, i] += e[j] / tot * v[h, j]
    return out


def test_attention_brute_force_and_sdpa():
    r = np.random.default_rng(5)
    q, k, v = (r.standard_normal((2, 6, 4)) * 2 for _ in range(3))
    assert np.allclose(O.attention(q, k, v), _attention_loops(q, k, v), atol=1e-13)
    q, k, v = (r.standard_normal((3, 50, 16)) for _ in range(3))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v)).numpy()
    assert np.allclose(O.attention(q, k, v), ref, atol=1e-12)
    sub = O.attention(q, k, v, rows=[3, 17, 49])
    assert np.allclose(sub, O.attention(q, k, v)[:, [3, 17, 49]], atol=0)


def test_attention_identical_keys_is_mean_of_values():
    r = np.random.default_rng(6)
    q = r.standard_normal((2, 9, 8))
    k = np.broadcast_to(r.standard_normal((2, 1, 8)), (2, 9, 8))
    v = r.standard_normal((2, 9, 8))
    assert np.allclose(O.attention(q, k, v), np.broadcast_to(v.mean(axis=1, keepdims=True), v.shape), atol=1e-14)


def test_attention_one_token_returns_its_value():
    r = np.random.default_rng(7)
    q, k, v = (r.standard_normal((3, 1, 8)) for _ in range(3))
    assert np.allclose(O.attention(q, k, v), v, atol=1e-15)


# ------------------------------------------------------------------ GELU


def test_gelu_tanh_closed_form():
    x = np.array([-3.0, -1.0, -0.25, 0.0, 0.5, 1.0, 2.0, 6.0])
    got = O.gelu_tanh(x)
    c = mpmath.sqrt(2 / mpmath.pi)
    for xi, gi in zip(x, got):
        xm = mpmath.mpf(xi)
        want = xm / 2 * (1 + mpmath.tanh(c * (xm + mpmath.mpf("0.044715") * xm ** 3)))
        assert abs(gi - float(want)) < 1e-15
    # odd part: GELU(x) - GELU(-x) = x
    assert np.allclose(got - O.gelu_tanh(-x), x, atol=1e-15)
    # within the tanh form's error of the erf form
    erf_form = np.array([float(mpmath.mpf(xi) / 2 * (1 + mpmath.erf(mpmath.mpf(xi) / mpmath.sqrt(2)))) for xi in x])
    assert np.max(np.abs(got - erf_form)) < 1e-3


# ------------------------------------------------------------------ the block, brute force

TINY = O.BlockConfig(d=12, heads=2, head_dim=6, ffn=20, eps=1e-6, rope_sections=(2, 2, 2))


def _tiny_inputs(seed, n=5, gate_std=0.5):
    r = np.random.default_rng(seed)
    d, f = TINY.d, TINY.ffn
    w = {"w_qkv": r.standard_normal((3 * d, d)) * 0.3, "w_o": r.standard_normal((d, d)) * 0.3,
         "w1": r.standard_normal((f, d)) * 0.3, "w2": r.standard_normal((d, f)) * 0.3}
    mod = r.standard_normal((6, d)) * gate_std
    x = r.standard_normal((n, d))
    pos = r.uniform(0, 9, (n, 3))
    return x, w, mod, pos


def _block_loops(x, w, mod, pos, cfg):
    """The block written out element by element, independently of the numpy
    formulation: every index of every contraction is explicit."""
    n, d = x.shape
    H, Dh, F = cfg.heads, cfg.head_dim, cfg.ffn
    sh1, sc1, g1, sh2, sc2, g2 = mod

    def ln_row(row, shift, scale):
        mu = sum(row) / d
        var = sum((a - mu) ** 2 for a in row) / d
        return [(row[c] - mu) / math.sqrt(var + cfg.eps) * (1 + scale[c]) + shift[c] for c in range(d)]

    def rot(vec, p):
        out = list(vec)
        start = 0
        for axis, sec in enumerate(cfg.rope_sections):
            for i in range(sec // 2):
                ang = p[axis] * cfg.rope_theta ** (-2.0 * i / sec)
                a, b = vec[start + 2 * i], vec[start + 2 * i + 1]
                out[start + 2 * i] = a * math.cos(ang) - b * math.sin(ang)
                out[start + 2 * i + 1] = a * math.sin(ang) + b * math.cos(ang)
            start += sec
        return out

    h = [ln_row(x[t], sh1, sc1) for t in range(n)]
    qkv = [[sum(h[t][c] * w["w_qkv"][o][c] for c in range(d)) for o in range(3 * d)] for t in range(n)]
    Q = [[rot(qkv[t][hd * Dh:(hd + 1) * Dh], pos[t]) for t in range(n)] for hd in range(H)]
    K = [[rot(qkv[t][d + hd * Dh:d + (hd + 1) * Dh], pos[t]) for t in range(n)] for hd in range(H)]
    V = [[qkv[t][2 * d + hd * Dh:2 * d + (hd + 1) * Dh] for t in range(n)] for hd in range(H)]
    o = [[0.0] * d for _ in range(n)]
    for hd in range(H):
        for i in range(n):
            s = [sum(Q[hd][i][c] * K[hd][j][c] for c in range(Dh)) / math.sqrt(Dh) for j in range(n)]
            mx = max(s)
            e = [math.exp(z - mx) for z in s]
            tot = sum(e)
            for c in range(Dh):
                o[i][hd * Dh + c] = sum(e[j] / tot * V[hd][j][c] for j in range(n))
    x2 = []
    for t in range(n):
        a = [sum(o[t][c] * w["w_o"][oc][c] for c in range(d)) for oc in range(d)]
        x1 = [x[t][c] + g1[c] * a[c] for c in range(d)]
        h2 = ln_row(x1, sh2, sc2)
        pre = [sum(h2[c] * w["w1"][j][c] for c in range(d)) for j in range(F)]
        u = [0.5 * z * (1 + math.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3))) for z in pre]
        m = [sum(u[j] * w["w2"][c][j] for j in range(F)) for c in range(d)]
        x2.append([x1[c] + g2[c] * m[c] for c in range(d)])
    return np.array(x2)


@pytest.mark.parametrize("seed", [0, 1])
def test_block_brute_force_tiny(seed):
    x, w, mod, pos = _tiny_inputs(seed)
    assert np.allclose(O.block_forward(x, w, mod, pos, TINY), _block_loops(x, w, mod, pos, TINY), atol=1e-12)


def test_block_gate_zero_is_identity_and_rows():
    x, w, mod, pos = _tiny_inputs(3)
    mod0 = mod.copy()
    mod0[2] = 0
    mod0[5] = 0
    assert np.array_equal(O.block_forward(x, w, mod0, pos, TINY), x)
    full = O.block_forward(x, w, mod, pos, TINY)
    assert np.allclose(O.block_forward(x, w, mod, pos, TINY, rows=[1, 4]), full[[1, 4]], atol=1e-14)


def test_block_bf16_storage_is_close_and_rounded():
    x, w, mod, pos = _tiny_inputs(4)
    a = O.block_forward(x, w, mod, pos, TINY)
    b = O.block_forward(x, w, mod, pos, TINY, bf16_storage=True)
    assert np.array_equal(b, O.bf16_round(b))
    assert np.linalg.norm(a - b) / np.linalg.norm(a) < 2e-2


def test_block_flops_formula():
    cfg = O.BlockConfig(d=5120, heads=40, head_dim=128, ffn=20480)
    # the four projections 2*N*d*(3d + d + 2F) and attention 4*N^2*d
    assert O.block_flops(6912, cfg) == pytest.approx(5.3270e12, rel=1e-4)
    assert O.block_flops(10488, cfg) == pytest.approx(8.8512e12, rel=1e-4)


# ------------------------------------------------------------------ quantisation


def test_quantize_rows_exact_rational():
    r = np.random.default_rng(8)
    x = (r.standard_normal((6, 64)) * r.uniform(0.01, 30, (6, 1))).astype(np.float32)
    x[2] = 0.0
    q, s = O.quantize_rows(x)
    assert q.dtype == np.int8 and s.dtype == np.float32
    assert np.all(np.abs(q.astype(int)) <= 127)
    assert np.all(q[2] == 0) and s[2, 0] == 0
    for i in range(6):
        if s[i, 0] == 0:
            continue
        # s is absmax / 127 rounded to binary32
        assert abs(Fraction(float(s[i, 0])) - Fraction(float(np.abs(x[i]).max())) / 127) <= Fraction(float(s[i, 0])) * Fraction(1, 2 ** 24)
        assert abs(int(q[i, np.argmax(np.abs(x[i]))])) == 127
        for j in range(64):
            exact = Fraction(float(x[i, j])) / Fraction(float(s[i, 0]))
            nearest = round(exact)                       # Python rounds half to even
            if abs(abs(exact - math.floor(exact)) - Fraction(1, 2)) > Fraction(1, 10 ** 5):
                assert int(q[i, j]) == max(-127, min(127, nearest))
            # reconstruction error at most half a step (plus the binary32 rounding of x / s)
            assert abs(float(x[i, j]) - float(s[i, 0]) * int(q[i, j])) <= float(s[i, 0]) * (0.5 + 1e-5)


def test_quantize_ties_to_even():
    # absmax 127 gives the scale 1 exactly, so x / s = x and the halves are exact ties
    x = np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, 126.5, -126.5]], np.float32)
    q, s = O.quantize_rows(x)
    assert s[0, 0] == 1.0
    assert q.tolist() == [[127, 2, 4, -2, 0, 0, 2, 126, -126]]


def test_quantize_groups_and_idempotence():
    r = np.random.default_rng(9)
    x = r.standard_normal((4, 3 * 32)).astype(np.float32)
    q, s = O.quantize_rows(x, 32)
    assert s.shape == (4, 3)
    for g in range(3):
        qg, sg = O.quantize_rows(x[:, g * 32:(g + 1) * 32])
        assert np.array_equal(qg, q[:, g * 32:(g + 1) * 32]) and np.array_equal(sg[:, 0], s[:, g])
    deq = (q.astype(np.float32).reshape(4, 3, 32) * s[:, :, None]).reshape(4, 96)
    q2, _ = O.quantize_rows(deq, 32)
    assert np.array_equal(q2, q)


def test_gemm_int_and_fc2_groups_brute_force():
    r = np.random.default_rng(10)
    a = r.integers(-127, 128, (3, 8)).astype(np.int8)
    b = r.integers(-127, 128, (5, 8)).astype(np.int8)
    acc = O.gemm_int(a, b)
    for i in range(3):
        for j in range(5):
            assert acc[i, j] == sum(int(a[i, k]) * int(b[j, k]) for k in range(8))
    # worst case magnitudes stay exact (127*127*K)
    big = np.full((1, 4096), 127, np.int8)
    assert O.gemm_int(big, -big)[0, 0] == -127 * 127 * 4096
    us = r.uniform(0.1, 2, (3, 2))
    ws = r.uniform(0.1, 2, 5)
    m = O.fc2_int8(a, us, b, ws, group=4)
    for i in range(3):
        for j in range(5):
            want = ws[j] * sum(us[i, g] * sum(int(a[i, k]) * int(b[j, k]) for k in range(4 * g, 4 * g + 4))
                               for g in range(2))
            assert abs(m[i, j] - want) < 1e-9
    # one group spanning all channels equals the plain dequantised projection
    assert np.allclose(O.fc2_int8(a, us[:, :1], b, ws, group=8), O.linear_int8(a, us[:, 0], b, ws))


# ------------------------------------------------------------------ token reduction


def test_token_counts_of_the_workloads():
    lines = [l.split() for l in open(__file__.replace("test_oracle_pins.py", "golden/token_counts.txt"))
             if l.strip() and not l.startswith("#")]
    for name, T, Hh, W, n_text, n_audio, n, n_red in lines:
        T, Hh, W, n_text, n_audio, n, n_red = map(int, (T, Hh, W, n_text, n_audio, n, n_red))
        assert T * Hh * W + n_text + n_audio == n
        g = O.VideoGrid(0, T, Hh, W)
        assert O.reduced_token_count(n, g) == n_red
        assert synth.positions((T, Hh, W), n_text, n_audio).shape == (n, 3)


def test_reduce_restore_identity_and_pairs():
    r = np.random.default_rng(11)
    g = O.VideoGrid(offset=3, T=2, Hh=3, W=5)        # odd W: last column unpaired
    n = 3 + 30 + 4
    x = O.bf16_round(r.standard_normal((n, 8)))
    red, side = O.token_reduce(x, g, bf16_storage=True)
    assert red.shape[0] == O.reduced_token_count(n, g) == n - 2 * 3 * 2
    # text before and audio after pass through; a pair is the mean of its columns
    assert np.array_equal(red[:3], x[:3]) and np.array_equal(red[-4:], x[-4:])
    assert np.array_equal(red[3], O.bf16_round((x[3] + x[4]) / 2))
    assert np.array_equal(red[5], x[7])               # (t=0, y=0) row: column 4 unpaired
    # reduce then restore with a zero update is the identity, bit for bit
    for storage in (False, True):
        red, side = O.token_reduce(x, g, bf16_storage=storage)
        assert np.array_equal(O.token_restore(red, side, g, bf16_storage=storage), x)
    # a uniform update moves every member of every pair by that amount
    red, side = O.token_reduce(x, g)
    back = O.token_restore(red + 0.25, side, g)
    assert np.allclose(back, x + 0.25, atol=1e-15)
    # constant pairs reduce exactly
    xc = np.repeat(r.standard_normal((n // 2 + 1, 8)), 2, axis=0)[:n]
    gc = O.VideoGrid(offset=0, T=1, Hh=2, W=4)
    redc, _ = O.token_reduce(xc[:8], gc)
    assert np.array_equal(redc, xc[0:8:2])


def test_reduced_positions_pair_mean():
    g = O.VideoGrid(0, 2, 2, 4)
    pos = synth.positions((2, 2, 4), 3, 2).astype(np.float64)
    pr = O.reduced_positions(pos, g)
    assert pr.shape == (8 + 5, 3)
    assert np.array_equal(pr[0], [0, 0, 0.5]) and np.array_equal(pr[1], [0, 0, 2.5])
    assert np.array_equal(pr[7], [1, 1, 2.5])
    assert np.array_equal(pr[8:], pos[16:])


# ------------------------------------------------------------------ the step


def test_step_one_block_equals_block_and_zero_gates():
    x, w, mod, pos = _tiny_inputs(12, n=6)
    assert np.array_equal(O.step_forward(x, [w], [mod], pos, TINY), O.block_forward(x, w, mod, pos, TINY))
    mods = []
    for b in range(4):
        m = mod.copy() * (b + 1)
        m[2] = 0
        m[5] = 0
        mods.append(m)
    assert np.array_equal(O.step_forward(x, [w] * 4, mods, pos, TINY), x)


def test_step_with_reduction_boundaries():
    cfg = TINY
    r = np.random.default_rng(13)
    g = O.VideoGrid(0, 1, 2, 4)
    n = 8 + 3
    x = r.standard_normal((n, cfg.d))
    pos = synth.positions((1, 2, 4), 3, 0).astype(np.float64)
    _, w, mod, _ = _tiny_inputs(14, n=n)
    red = O.Reduction(grid=g, reduce_after_block=0, restore_before_block=2)
    # zero gates: reduce + restore around identity blocks is the identity
    m0 = mod.copy()
    m0[2] = 0
    m0[5] = 0
    assert np.allclose(O.step_forward(x, [w] * 3, [m0] * 3, pos, cfg, reduction=red), x, atol=1e-15)
    # by hand: block 0 full, block 1 reduced, restore, block 2 full
    y0 = O.block_forward(x, w, mod, pos, cfg)
    yr, side = O.token_reduce(y0, g)
    y1 = O.block_forward(yr, w, mod * 0.5, O.reduced_positions(pos, g), cfg)
    y1f = O.token_restore(y1, side, g)
    y2 = O.block_forward(y1f, w, mod * 2, pos, cfg)
    got = O.step_forward(x, [w] * 3, [mod, mod * 0.5, mod * 2], pos, cfg, reduction=red)
    assert np.allclose(got, y2, atol=1e-14)


# ------------------------------------------------------------------ int8 block


def test_int8_block_close_to_float_block():
    cfg = O.BlockConfig(d=64, heads=2, head_dim=32, ffn=128, rope_sections=(8, 12, 12))
    r = np.random.default_rng(15)
    n = 24
    w = {"w_qkv": r.standard_normal((3 * 64, 64)) * 0.1, "w_o": r.standard_normal((64, 64)) * 0.1,
         "w1": r.standard_normal((128, 64)) * 0.1, "w2": r.standard_normal((64, 128)) * 0.1}
    wq = {}
    for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"), ("w2", "q2", "s2")):
        wq[qn], s = O.quantize_weight(w[name])
        wq[sn] = s[:, 0]
    mod = r.standard_normal((6, 64)) * 0.3
    x = r.standard_normal((n, 64))
    pos = r.uniform(0, 5, (n, 3))
    ref = O.block_forward(x, w, mod, pos, cfg)
    got = O.block_forward_int8(x, wq, mod, pos, cfg, bf16_storage=False, fc2_group=64)
    # int8 error on the branch only (x itself passes through exactly)
    rel = np.linalg.norm((got - x) - (ref - x)) / np.linalg.norm(ref - x)
    assert rel < 3e-2
    # fc2 groups equal to F reduce to the per-token scheme
    a = O.block_forward_int8(x, wq, mod, pos, cfg, bf16_storage=False, fc2_group=128)
    assert np.linalg.norm((a - x) - (ref - x)) / np.linalg.norm(ref - x) < 3e-2


def test_int8_block_rows_match_full_evaluation():
    """Evaluating selected query rows gives those rows of the full block."""
    cfg = O.BlockConfig(d=64, heads=2, head_dim=32, ffn=128, rope_sections=(8, 12, 12))
    r = np.random.default_rng(16)
    n = 20
    wq = {}
    for qn, sn, shp in (("q_qkv", "s_qkv", (192, 64)), ("q_o", "s_o", (64, 64)), ("q1", "s1", (128, 64)),
                        ("q2", "s2", (64, 128))):
        wq[qn], s = O.quantize_weight(r.standard_normal(shp) * 0.1)
        wq[sn] = s[:, 0]
    mod = r.standard_normal((6, 64)) * 0.3
    x = r.standard_normal((n, 64))
    pos = r.uniform(0, 5, (n, 3))
    full = O.block_forward_int8(x, wq, mod, pos, cfg, bf16_storage=False, fc2_group=64)
    rows = [0, 7, 19]
    part = O.block_forward_int8(x, wq, mod, pos, cfg, bf16_storage=False, fc2_group=64, rows=rows)
    assert np.allclose(part, full[rows], rtol=0, atol=1e-12)


def test_int8_block_without_int8_projections_is_the_float_block():
    """With no projection in int8 the mixed-precision block is the BF16 block
    (same storage points), bit for bit; MLP-only and QKV-only sit between."""
    cfg = O.BlockConfig(d=64, heads=2, head_dim=32, ffn=128, rope_sections=(8, 12, 12))
    r = np.random.default_rng(17)
    n = 20
    w = {"w_qkv": r.standard_normal((192, 64)) * 0.1, "w_o": r.standard_normal((64, 64)) * 0.1,
         "w1": r.standard_normal((128, 64)) * 0.1, "w2": r.standard_normal((64, 128)) * 0.1}
    for name, qn, sn in (("w_qkv", "q_qkv", "s_qkv"), ("w_o", "q_o", "s_o"), ("w1", "q1", "s1"), ("w2", "q2", "s2")):
        w[qn], sc = O.quantize_weight(w[name])
        w[sn] = sc[:, 0]
    mod = r.standard_normal((6, 64)) * 0.3
    x = r.standard_normal((n, 64))
    pos = r.uniform(0, 5, (n, 3))
    for storage in (False, True):
        ref = O.block_forward(x, w, mod, pos, cfg, bf16_storage=storage)
        none = O.block_forward_int8(x, w, mod, pos, cfg, bf16_storage=storage, fc2_group=64, which=())
        assert np.array_equal(none, ref)
    ref = O.block_forward(x, w, mod, pos, cfg)
    errs = {}
    for which in (O.INT8_QKV, O.INT8_MLP, O.INT8_ALL):
        got = O.block_forward_int8(x, w, mod, pos, cfg, bf16_storage=False, fc2_group=64, which=which)
        errs[which] = np.linalg.norm((got - x) - (ref - x)) / np.linalg.norm(ref - x)
        assert 0 < errs[which] < 3e-2
    # quantising more projections adds error
    assert errs[O.INT8_ALL] > max(errs[O.INT8_QKV], errs[O.INT8_MLP])


# A block small enough for scalar loops whose widths span several FC2 groups:
# with d = 16, F = 32 and a group of 8, a per-token scale (one per row of 16
# or 32) and a per-group scale (one per 8 channels) are different things, so
# quantising a tensor at the wrong granularity changes its codes.
TINY8 = O.BlockConfig(d=16, heads=2, head_dim=8, ffn=32, eps=1e-6, rope_sections=(2, 2, 4))
TINY8_GROUP = 8


def _bf16_list(vals):
    """BF16 storage of fp64 values through torch's casts (binary64 -> binary32
    -> bfloat16, each rounding to nearest even), back as Python floats."""
    t = torch.tensor(list(vals), dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    return t.double().tolist()


def _quant_loops(vals):
    """The int8 rule written out for one group of values: s = absmax / 127
    divided in binary32, code = the binary32 quotient x / s rounded half to
    even (Python's round) and clamped to +-127; an all-zero group has s = 0
    and codes 0.  Returns (codes as Python ints, s as a Python float)."""
    amax = np.float32(max(abs(v) for v in vals))
    s = np.float32(amax / np.float32(127.0))
    if s == 0:
        return [0] * len(vals), 0.0
    codes = [max(-127, min(127, round(float(np.float32(np.float32(v) / s))))) for v in vals]
    return codes, float(s)


def _block_int8_loops(x, w, mod, pos, cfg, group):
    """The dynamic-int8 block ([linlog] "int8 量化：从 36 秒到 19 秒") written
    out element by element with every quantisation point spelled out: h, o
    and h2 are stored as BF16 and then quantised per token; FC1's GELU output
    u is stored as BF16 and quantised per token and per ``group`` channels;
    each projection is an exact integer sum (Python ints) dequantised as
    acc * s_act * s_w, FC2 as s_w * sum over groups (ascending) of
    s_u[group] * acc_group; every stored tensor is BF16.  Returns the output
    and the codes and scales of the four quantised tensors."""
    n, d = x.shape
    H, Dh, F = cfg.heads, cfg.head_dim, cfg.ffn
    sh1, sc1, g1, sh2, sc2, g2 = mod

    def ln_row(row, shift, scale):
        mu = sum(row) / d
        var = sum((a - mu) ** 2 for a in row) / d
        return [(row[c] - mu) / math.sqrt(var + cfg.eps) * (1 + scale[c]) + shift[c] for c in range(d)]

    def rot(vec, p):
        out = list(vec)
        start = 0
        for axis, sec in enumerate(cfg.rope_sections):
            for i in range(sec // 2):
                ang = p[axis] * cfg.rope_theta ** (-2.0 * i / sec)
                a, b = vec[start + 2 * i], vec[start + 2 * i + 1]
                out[start + 2 * i] = a * math.cos(ang) - b * math.sin(ang)
                out[start + 2 * i + 1] = a * math.sin(ang) + b * math.cos(ang)
            start += sec
        return out

    def qlinear(codes, s_act, wq, ws):
        acc = [sum(codes[c] * int(wq[o][c]) for c in range(len(codes))) for o in range(len(wq))]
        return [acc[o] * s_act * float(ws[o]) for o in range(len(wq))]

    h = [_bf16_list(ln_row(x[t], sh1, sc1)) for t in range(n)]
    hq = [_quant_loops(h[t]) for t in range(n)]
    qkv = [qlinear(hq[t][0], hq[t][1], w["q_qkv"], w["s_qkv"]) for t in range(n)]
    Q = [[_bf16_list(rot(qkv[t][hd * Dh:(hd + 1) * Dh], pos[t])) for t in range(n)] for hd in range(H)]
    K = [[_bf16_list(rot(qkv[t][d + hd * Dh:d + (hd + 1) * Dh], pos[t])) for t in range(n)] for hd in range(H)]
    V = [[_bf16_list(qkv[t][2 * d + hd * Dh:2 * d + (hd + 1) * Dh]) for t in range(n)] for hd in range(H)]
    o = [[0.0] * d for _ in range(n)]
    for hd in range(H):
        for i in range(n):
            s = [sum(Q[hd][i][c] * K[hd][j][c] for c in range(Dh)) / math.sqrt(Dh) for j in range(n)]
            mx = max(s)
            e = [math.exp(z - mx) for z in s]
            tot = sum(e)
            for c in range(Dh):
                o[i][hd * Dh + c] = sum(e[j] / tot * V[hd][j][c] for j in range(n))
    o = [_bf16_list(row) for row in o]
    oq, h2q, uq, out = [], [], [], []
    for t in range(n):
        oq.append(_quant_loops(o[t]))
        a = _bf16_list(qlinear(oq[t][0], oq[t][1], w["q_o"], w["s_o"]))
        x1 = _bf16_list([x[t][c] + g1[c] * a[c] for c in range(d)])
        h2 = _bf16_list(ln_row(x1, sh2, sc2))
        h2q.append(_quant_loops(h2))
        pre = qlinear(h2q[t][0], h2q[t][1], w["q1"], w["s1"])
        u = _bf16_list([0.5 * z * (1 + math.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3))) for z in pre])
        groups = [_quant_loops(u[g0:g0 + group]) for g0 in range(0, F, group)]
        uq.append(groups)
        m = []
        for c in range(d):
            tot = 0.0
            for gi, (codes, su) in enumerate(groups):
                acc = sum(codes[j] * int(w["q2"][c][gi * group + j]) for j in range(group))
                tot += su * acc
            m.append(float(w["s2"][c]) * tot)
        m = _bf16_list(m)
        out.append(_bf16_list([x1[c] + g2[c] * m[c] for c in range(d)]))
    return np.array(out), dict(hq=hq, oq=oq, h2q=h2q, uq=uq)


def _tiny8_inputs(seed, n=5):
    r = np.random.default_rng(seed)
    d, f = TINY8.d, TINY8.ffn
    w = {}
    for name, qn, sn, shp in (("w_qkv", "q_qkv", "s_qkv", (3 * d, d)), ("w_o", "q_o", "s_o", (d, d)),
                              ("w1", "q1", "s1", (f, d)), ("w2", "q2", "s2", (d, f))):
        # per-channel magnitudes that differ across each row, so group and
        # token absmax differ
        wt = r.standard_normal(shp) * 0.3 * r.uniform(0.2, 3.0, (1, shp[1]))
        w[qn], s = O.quantize_weight(wt)
        w[sn] = s[:, 0]
    mod = r.standard_normal((6, d)) * 0.5
    x = O.bf16_round(r.standard_normal((n, d)) * r.uniform(0.2, 3.0, (1, d)))
    pos = r.uniform(0, 9, (n, 3))
    return x, w, mod, pos


@pytest.mark.parametrize("seed", [0, 1])
def test_int8_block_scalar_loops(seed):
    """The oracle's int8 block against the element-by-element restatement on
    a block whose widths span several FC2 groups: every code and scale of h,
    o, h2 (per token) and u (per token and group) equal, and the outputs
    equal to rounding."""
    x, w, mod, pos = _tiny8_inputs(seed)
    got, parts = O.block_forward_int8(x, w, mod, pos, TINY8, bf16_storage=True, fc2_group=TINY8_GROUP,
                                      return_parts=True)
    want, lp = _block_int8_loops(x, w, mod, pos, TINY8, TINY8_GROUP)
    for name, qn, sn in (("h", "hq", "hs"), ("o", "oq", "os"), ("h2", "h2q", "h2s")):
        codes = np.array([c for c, _ in lp[qn]])
        scales = np.array([s for _, s in lp[qn]])
        assert np.array_equal(parts[qn].astype(np.int64), codes), f"{name} codes"
        assert np.array_equal(parts[sn][:, 0].astype(np.float64), scales), f"{name} scales"
    ucodes = np.array([[c for codes, _ in row for c in codes] for row in lp["uq"]])
    uscales = np.array([[s for _, s in row] for row in lp["uq"]])
    assert parts["us"].shape == (x.shape[0], TINY8.ffn // TINY8_GROUP)
    assert np.array_equal(parts["uq"].astype(np.int64), ucodes), "u codes"
    assert np.array_equal(parts["us"].astype(np.float64), uscales), "u scales"
    assert np.allclose(got, want, rtol=0, atol=1e-12)
    # the group and per-token scales really differ on this block
    assert not np.allclose(uscales, uscales.max(axis=1, keepdims=True))


# ------------------------------------------------------------------ per-segment modulation


def test_segment_mod_equals_per_segment_blocks():
    """Per-token modulation from segments: each output row equals the block
    run with that row's segment vectors (rows only mix through attention,
    which the modulation does not enter after AdaLN-1), and a single segment
    equals the plain [6, d] modulation bit for bit."""
    cfg = O.BlockConfig(d=64, heads=2, head_dim=32, ffn=128, rope_sections=(8, 12, 12))
    r = np.random.default_rng(18)
    n = 24
    w = {"w_qkv": r.standard_normal((192, 64)) * 0.1, "w_o": r.standard_normal((64, 64)) * 0.1,
         "w1": r.standard_normal((128, 64)) * 0.1, "w2": r.standard_normal((64, 128)) * 0.1}
    x = r.standard_normal((n, 64))
    pos = r.uniform(0, 5, (n, 3))
    seg = r.standard_normal((3, 6, 64)) * 0.3
    starts = [0, 10, 18]
    per_row = O.segment_mod(seg, starts, n)
    assert per_row.shape == (6, n, 64)
    assert np.array_equal(per_row[:, 12], seg[1]) and np.array_equal(per_row[:, 23], seg[2])
    got = O.block_forward(x, w, per_row, pos, cfg)
    one = O.block_forward(x, w, O.segment_mod(seg[:1], [0], n), pos, cfg)
    assert np.array_equal(one, O.block_forward(x, w, seg[0], pos, cfg))
    # rows of segment 1: AdaLN-1 of every row uses its own segment, so the
    # keys/values come from the per-token h; the query rows' later steps use
    # segment 1's vectors: compare against a hand-built mixture
    h_rows = per_row.copy()
    ref_rows = O.block_forward(x, w, h_rows, pos, cfg, rows=[10, 17])
    assert np.allclose(got[[10, 17]], ref_rows, atol=1e-13)
    # changing segment 2's gates leaves segments 0-1 unchanged only through
    # attention's keys (AdaLN-1 shift/scale): gates alone do not leak
    seg2 = seg.copy()
    seg2[2, 2] *= 3.0
    seg2[2, 5] *= -1.0
    moved = O.block_forward(x, w, O.segment_mod(seg2, starts, n), pos, cfg)
    assert np.array_equal(moved[:18], got[:18]) and not np.allclose(moved[18:], got[18:])


def test_step_reduction_with_segments():
    """The reduced stream's tokens keep their segment's vectors."""
    cfg = O.BlockConfig(d=64, heads=2, head_dim=32, ffn=128, rope_sections=(8, 12, 12))
    r = np.random.default_rng(19)
    grid = O.VideoGrid(0, 2, 3, 4)            # 24 video tokens, then 6 text, 2 audio
    n = 32
    w = {"w_qkv": r.standard_normal((192, 64)) * 0.1, "w_o": r.standard_normal((64, 64)) * 0.1,
         "w1": r.standard_normal((128, 64)) * 0.1, "w2": r.standard_normal((64, 128)) * 0.1}
    x = r.standard_normal((n, 64))
    pos = np.concatenate([np.stack(np.meshgrid(np.arange(2), np.arange(3), np.arange(4), indexing="ij"), -1).reshape(-1, 3),
                          np.full((8, 3), 5.0)]).astype(np.float64)
    seg = r.standard_normal((3, 6, 64)) * 0.3
    starts = [0, 24, 30]
    per_row = O.segment_mod(seg, starts, n)
    red = O.Reduction(grid, 0, 2)
    got = O.step_forward(x, [w] * 3, [per_row] * 3, pos, cfg, reduction=red)
    # by hand: block 0 full, reduce, block 1 with the reduced segment map, restore, block 2
    y = O.block_forward(x, w, per_row, pos, cfg)
    yr, side = O.token_reduce(y, grid)
    nr = O.reduced_token_count(n, grid)
    per_row_red = O.segment_mod(seg, [0, 12, 18], nr)
    yr = O.block_forward(yr, w, per_row_red, O.reduced_positions(pos, grid), cfg)
    y2 = O.token_restore(yr, side, grid)
    y2 = O.block_forward(y2, w, per_row, pos, cfg)
    assert np.allclose(got, y2, atol=1e-13)


# ------------------------------------------------------------------ final layer


def test_final_head_identity_projection_is_layer_norm():
    """With zero shift/scale and the identity as projection the head returns
    the textbook LayerNorm of its rows (torch, fp64)."""
    r = np.random.default_rng(20)
    x = r.standard_normal((30, 48)) * 3 + 1
    got = O.final_head(x, 5, 20, np.zeros(48), np.zeros(48), np.eye(48), 1e-6)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x[5:25]), (48,), eps=1e-6).numpy()
    assert np.allclose(got, ref, atol=1e-12)


def test_final_head_scalar_loops():
    r = np.random.default_rng(21)
    n, d, c = 9, 16, 5
    x = r.standard_normal((n, d))
    sh, sc, w = r.standard_normal(d) * 0.2, r.standard_normal(d) * 0.2, r.standard_normal((c, d))
    got = O.final_head(x, 2, 4, sh, sc, w, 1e-6)
    for i in range(4):
        row = x[2 + i]
        mu = sum(row) / d
        var = sum((v - mu) ** 2 for v in row) / d
        hrow = [(row[k] - mu) / math.sqrt(var + 1e-6) * (1 + sc[k]) + sh[k] for k in range(d)]
        for o in range(c):
            assert abs(got[i, o] - sum(hrow[k] * w[o, k] for k in range(d))) < 1e-12


# ------------------------------------------------------------------ core residual reuse


def test_core_reuse_replays_the_core_exactly():
    """Reusing the residual on the same input gives the core's output bit for
    bit (the residual of two BF16 streams is exact in fp64), and on another
    input adds the same update."""
    cfg = O.BlockConfig(d=64, heads=2, head_dim=32, ffn=128, rope_sections=(8, 12, 12))
    r = np.random.default_rng(22)
    n = 16
    w = {"w_qkv": r.standard_normal((192, 64)) * 0.1, "w_o": r.standard_normal((64, 64)) * 0.1,
         "w1": r.standard_normal((128, 64)) * 0.1, "w2": r.standard_normal((64, 128)) * 0.1}
    x = O.bf16_round(r.standard_normal((n, 64)))
    pos = r.uniform(0, 5, (n, 3))
    mod = r.standard_normal((6, 64)) * 0.3
    y = O.step_forward(x, [w, w], [mod, mod], pos, cfg, bf16_storage=True)
    delta = O.core_residual(x, y)
    assert np.array_equal(O.core_reuse(x, delta), y)
    x2 = O.bf16_round(x + 0.25)
    assert np.array_equal(O.core_reuse(x2, delta), O.bf16_round(x2 + (y - x)))

