"""Plant plausible slips in the oracle (on the CPU) and check that the pins
of ``test_oracle_pins.py`` catch every one of them.

Each mutation rewrites one function's source text, executes the rewritten
function in the oracle module's namespace for the duration of one test, runs
the pins that should notice, and asserts that at least one of them fails.
"""
import inspect
import textwrap

import pytest

import oracle.h3dit_oracle as M
import tests.test_oracle_pins as P

# (function, original text, replacement, pins expected to notice)
MUTATIONS = [
    ("layer_norm", ".mean(axis=-1, keepdims=True)\n    return", ".sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)\n    return",
     [P.test_layer_norm_hand_example, P.test_layer_norm_matches_torch]),
    ("layer_norm", "np.sqrt(var + eps)", "np.sqrt(var)", [P.test_layer_norm_hand_example]),
    ("adaln", "(1.0 + np.asarray(scale, np.float64))", "np.asarray(scale, np.float64)", [P.test_adaln_special_cases]),
    ("rope_angles", "-2.0 * i / sec", "-1.0 * i / sec", [P.test_rope_sections_axes_and_frequencies]),
    ("rope_angles", "pos[:, axis:axis + 1]", "pos[:, 2 - axis:3 - axis]", [P.test_rope_sections_axes_and_frequencies]),
    ("apply_rope", "a * s + b * c", "-a * s + b * c", [P.test_rope_identity_at_origin_and_norm, P.test_rope_sections_axes_and_frequencies]),
    ("apply_rope", "a = t[..., 0::2]\n    b = t[..., 1::2]", "a = t[..., :t.shape[-1] // 2]\n    b = t[..., t.shape[-1] // 2:]",
     [P.test_rope_sections_axes_and_frequencies]),
    ("attention", "/ math.sqrt(dh)", "", [P.test_attention_brute_force_and_sdpa]),
    ("attention", "p /= p.sum(axis=1, keepdims=True)", "p /= p.sum(axis=0, keepdims=True)", [P.test_attention_brute_force_and_sdpa]),
    ("gelu_tanh", "0.044715 * x ** 3", "0.0447 * x ** 3", [P.test_gelu_tanh_closed_form]),
    ("gelu_tanh", "np.tanh(", "np.tanh(0.0 * ", [P.test_gelu_tanh_closed_form]),
    ("block_forward", 'w["w_o"], np.float64).T', 'w["w_o"], np.float64)', [P.test_block_brute_force_tiny]),
    ("block_forward", 'w["w2"], np.float64).T', 'w["w2"], np.float64).T[::-1]', [P.test_block_brute_force_tiny]),
    ("block_forward", "x1 = R(x[sel] + gate1 * a)", "x1 = R(x[sel] + gate2 * a)", [P.test_block_brute_force_tiny]),
    ("block_forward", "h2 = R(adaln(x1, shift2, scale2", "h2 = R(adaln(x[sel], shift2, scale2", [P.test_block_brute_force_tiny]),
    ("block_forward", "qkv[:, d:2 * d]", "qkv[:, 2 * d:3 * d]", [P.test_block_brute_force_tiny]),
    ("block_forward", "v = R(_split_heads(qkv[:, 2 * d:3 * d], cfg))",
     "v = R(apply_rope(_split_heads(qkv[:, 2 * d:3 * d], cfg).transpose(1, 0, 2), pos, cfg)).transpose(1, 0, 2)",
     [P.test_block_brute_force_tiny]),
    ("block_forward", "adaln(x, shift1, scale1", "adaln(x, shift2, scale1", [P.test_block_brute_force_tiny]),
    ("_split_heads", "reshape(n, cfg.heads, cfg.head_dim).transpose(1, 0, 2)",
     "reshape(n, cfg.head_dim, cfg.heads).transpose(2, 0, 1)", [P.test_block_brute_force_tiny]),
    ("quantize_rows", "np.rint(y)", "np.trunc(y + np.sign(y) * 0.5)", [P.test_quantize_rows_exact_rational, P.test_quantize_ties_to_even]),
    ("quantize_rows", "np.float32(127.0)", "np.float32(128.0)", [P.test_quantize_rows_exact_rational]),
    ("fc2_int8", "us[:, g:g + 1] * acc", "us[:, 0:1] * acc", [P.test_gemm_int_and_fc2_groups_brute_force]),
    ("token_restore", "out[i] = side[i] + upd", "out[i] = side[i]", [P.test_reduce_restore_identity_and_pairs]),
    ("token_restore", "upd = x_red[p] - at_reduce", "upd = x_red[p] - side[g[0]]", [P.test_reduce_restore_identity_and_pairs]),
    ("_reduce_map", "if c0 + 1 < grid.W:", "if c0 + 1 <= grid.W:", [P.test_reduce_restore_identity_and_pairs]),
    ("reduced_token_count", "grid.T * grid.Hh *", "grid.Hh *", [P.test_token_counts_of_the_workloads, P.test_reduce_restore_identity_and_pairs]),
    ("step_forward", "b == reduction.restore_before_block", "b == reduction.restore_before_block + 1", [P.test_step_with_reduction_boundaries]),
    ("step_forward", "b == reduction.reduce_after_block", "b == reduction.reduce_after_block + 1", [P.test_step_with_reduction_boundaries]),
    # int8 projection selection
    ("block_forward_int8", 'if "qkv" in which:', 'if "o" in which:', [P.test_int8_block_without_int8_projections_is_the_float_block]),
    ("block_forward_int8", 'fc2_int8(uq, us, w["q2"], w["s2"], g2)', 'fc2_int8(uq, us, w["q2"], w["s1"][:w["q2"].shape[0]], g2)',
     [P.test_int8_block_close_to_float_block, P.test_int8_block_without_int8_projections_is_the_float_block]),
    # int8 quantisation points and granularity
    ("block_forward_int8", 'oq, os_ = quantize_rows(o)\n        a = R(linear_int8(oq, os_, w["q_o"], w["s_o"]))',
     'oq, os_ = quantize_rows(o, g2)\n        a = R(fc2_int8(oq, os_, w["q_o"], w["s_o"], g2))',
     [P.test_int8_block_scalar_loops]),
    ("block_forward_int8", "oq, os_ = quantize_rows(o)", "oq, os_ = quantize_rows(_merge_heads(attention(q, k, v, rows=rows)))",
     [P.test_int8_block_scalar_loops]),
    ("block_forward_int8", "h2q, h2s = quantize_rows(h2)", "h2q, h2s = quantize_rows(adaln(x1, shift2, scale2, cfg.eps))",
     [P.test_int8_block_scalar_loops]),
    ("block_forward_int8", "hq, hs = quantize_rows(h)", "hq, hs = quantize_rows(adaln(x, shift1, scale1, cfg.eps))",
     [P.test_int8_block_scalar_loops]),
    ("block_forward_int8", "uq, us = quantize_rows(u, g2)",
     'uq, us = quantize_rows(linear_int8(h2q, h2s, w["q1"], w["s1"]), g2)', [P.test_int8_block_scalar_loops]),
    ("fc2_int8", "out += us[:, g:g + 1] * acc", "out += us.max(axis=1, keepdims=True) * acc",
     [P.test_int8_block_scalar_loops]),
    # per-segment modulation
    ("segment_mod", "seg[starts[s_]:starts[s_ + 1]] = s_", "seg[starts[s_]:starts[s_ + 1]] = min(s_, 1)",
     [P.test_segment_mod_equals_per_segment_blocks]),
    ("_mod_parts", "(v[sel] for v in (gate1, shift2, scale2, gate2))", "(v[sel] for v in (gate1, scale2, shift2, gate2))",
     [P.test_segment_mod_equals_per_segment_blocks]),
    ("_reduce_mod_rows", "return mod[:, first, :]", "return mod[:, :len(first), :]", [P.test_step_reduction_with_segments]),
    # final layer
    ("final_head", "adaln(xs, np.asarray(shift, np.float64), np.asarray(scale, np.float64), eps)",
     "adaln(xs, np.asarray(scale, np.float64), np.asarray(shift, np.float64), eps)", [P.test_final_head_scalar_loops]),
    ("final_head", "[row_start:row_start + rows]", "[row_start + 1:row_start + rows + 1]", [P.test_final_head_scalar_loops]),
    # core residual reuse
    ("core_reuse", "np.asarray(x, np.float64) + np.asarray(delta, np.float64)",
     "np.asarray(x, np.float64) - np.asarray(delta, np.float64)", [P.test_core_reuse_replays_the_core_exactly]),
    ("core_residual", "np.asarray(x_out, np.float64) - np.asarray(x_in, np.float64)",
     "np.asarray(x_in, np.float64) - np.asarray(x_out, np.float64)", [P.test_core_reuse_replays_the_core_exactly]),
]


def _run_pin(pin):
    params = getattr(pin, "pytestmark", [])
    seeds = [0]
    for mark in params:
        if mark.name == "parametrize":
            seeds = mark.args[1]
    if "seed" in inspect.signature(pin).parameters:
        for s in seeds:
            pin(s)
    else:
        pin()


@pytest.mark.parametrize("fname,old,new,pins", MUTATIONS, ids=[f"{m[0]}-{i}" for i, m in enumerate(MUTATIONS)])
def test_planted_slip_is_caught(monkeypatch, fname, old, new, pins):
    src = textwrap.dedent(inspect.getsource(getattr(M, fname)))
    assert old in src, f"mutation anchor not found in {fname}"
    ns = dict(vars(M))
    exec(compile(src.replace(old, new, 1), f"<mutant {fname}>", "exec"), ns)
    monkeypatch.setattr(M, fname, ns[fname])
    # functions imported by name into the package namespace too
    import oracle
    if hasattr(oracle, fname):
        monkeypatch.setattr(oracle, fname, ns[fname])
    caught = False
    for pin in pins:
        try:
            _run_pin(pin)
        except AssertionError:
            caught = True
            break
    assert caught, f"planted slip in {fname} ({old!r} -> {new!r}) passed every pin"
