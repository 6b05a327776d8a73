"""Plain, slow, fp64 restatement of one MiniMax-H3 DiT block and the step.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
CUDA library or its Python binding.

Sources.  The method is described by five web pages about h3.c ("h3-metal"),
an Apple-Silicon inference engine for MiniMax-H3.  Citations below name the
page and the section on it:

* [alphalab] "h3-metal 把 MiniMax-H3 搬上 Apple Silicon：突破與代價（2026）",
  section "h3-metal 發布的是推論引擎，不是 MiniMax-H3 模型" (model facts:
  33B dense single-stream Omni Transformer, 50 layers, full attention).
* [linlog] linlog.top article 1265 on h3.c, sections
  "MiniMax H3：原生音频视频一体化生成" (AdaLN branch precomputed at inference),
  "h3.c 的核心设计" (QKV routed head-major), "int8 量化：从 36 秒到 19 秒"
  (dynamic activations, per-output-channel weights, one scale per 1024 FC2
  input channels), "DiT 融合内核：减少全局内存往返" (gated AdaLN fusion, BF16
  residual rounding), "Token 缩减：28% 的去噪时间消减" (horizontal pairing
  after block 3, restore before block 40), "音频处理" (audio on the rotary
  timeline as width-32 rows).
* [steinslab] "零 Python 依赖：Redis 作者的 3.5 秒端侧实验", section
  "极简主控逻辑" (spatial RoPE).

The pages give neither the block's sizes nor its norm type, RoPE split or
GELU form.  Readings adopted where they are silent (each also stated at the
function that uses it):

* LayerNorm with biased variance, eps 1e-6, no elementwise affine.
* AdaLN modulation x_hat * (1 + scale) + shift; gates broadcast per channel.
* Per-block modulation layout [6][d]: shift1, scale1, gate1, shift2, scale2,
  gate2.
* No biases, no QK-norm.
* GELU, tanh form.
* 3D RoPE: theta 10000, head-dim sections (t, h, w) = (32, 48, 48) for
  Dh = 128 and (16, 24, 24) for Dh = 64, frequencies theta^(-2i/section),
  pairs interleaved (2i, 2i+1), float positions, applied to Q and K only.
* Attention scale 1/sqrt(Dh), non-causal, no mask.
* Quantisation: symmetric absmax / 127 in fp32, round half to even,
  clamp to [-127, 127], zero rows give scale 0 and codes 0.
* Token reduction: pair columns (2j, 2j+1) of every (t, y) video row, fp32/
  fp64 mean; an odd last column passes through; restore adds the pair's
  update (current reduced value minus the value the pair had when reduced).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library routines on special cases, brute force on tiny
inputs).  None is "parity unpinned" except where a function docstring says
so.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

__all__ = [
    "BlockConfig", "VideoGrid", "Reduction",
    "bf16_round", "layer_norm", "adaln", "rope_angles", "apply_rope",
    "attention", "gelu_tanh", "block_forward", "step_forward", "segment_mod", "final_head", "core_residual", "core_reuse",
    "quantize_rows", "quantize_weight", "gemm_int", "linear_int8", "INT8_ALL", "INT8_MLP", "INT8_QKV",
    "fc2_int8", "block_forward_int8",
    "reduced_token_count", "token_reduce", "token_restore",
    "reduced_positions", "block_flops",
]


# --------------------------------------------------------------------------
# configuration
# --------------------------------------------------------------------------
@dataclass
class BlockConfig:
    """Shape of one DiT block.  The pages give none of these numbers; the
    synthetic workloads fix d, heads, Dh, F and eps, the rest are readings."""
    d: int
    heads: int
    head_dim: int
    ffn: int
    eps: float = 1e-6
    rope_sections: Sequence[int] = field(default_factory=lambda: (32, 48, 48))
    rope_theta: float = 10000.0

    def __post_init__(self):
        assert self.d == self.heads * self.head_dim
        assert sum(self.rope_sections) == self.head_dim
        assert all(s % 2 == 0 for s in self.rope_sections)


@dataclass
class VideoGrid:
    """Target-video tokens: ``T*Hh*W`` rows starting at row ``offset``,
    ordered t-major, then y, then x."""
    offset: int
    T: int
    Hh: int
    W: int

    @property
    def n_video(self) -> int:
        return self.T * self.Hh * self.W

    @property
    def w_reduced(self) -> int:
        return (self.W + 1) // 2


@dataclass
class Reduction:
    """Token-reduction schedule ([linlog] "Token 缩减"): blocks
    0..reduce_after_block run at full resolution, blocks up to
    restore_before_block-1 run on the reduced sequence, the rest at full
    resolution again.  Block indices are 0-based."""
    grid: VideoGrid
    reduce_after_block: int = 3
    restore_before_block: int = 40
    pos_reduced: Optional[np.ndarray] = None


# --------------------------------------------------------------------------
# storage rounding (only used to mirror stored BF16 tensors on request)
# --------------------------------------------------------------------------
def bf16_round(a) -> np.ndarray:
    """Round to the nearest BF16 value, ties to even, returned as fp64.

    BF16 is the top 16 bits of an IEEE binary32; the value is first rounded
    to binary32 (numpy casts round to nearest even) and then its low 16 bits
    are rounded away, ties to even."""
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) & 0xFFFF0000
    out = r.astype(np.uint32).view(np.float32)
    # NaN stays NaN, infinities stay infinite
    out = np.where(np.isnan(f), f, out)
    return out.astype(np.float64)


def _maybe_round(a, on: bool):
    return bf16_round(a) if on else np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# AdaLN ([linlog] "MiniMax H3" section: AdaLN branch precomputed and cached;
# "DiT 融合内核": gated AdaLN)
# --------------------------------------------------------------------------
def layer_norm(x, eps: float) -> np.ndarray:
    """LayerNorm over the last axis with the biased (population) variance and
    no elementwise affine: (x - mean) / sqrt(var + eps)."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps)


def adaln(x, shift, scale, eps: float) -> np.ndarray:
    """AdaLN modulation of a normalised row: LN(x) * (1 + scale) + shift, with
    per-channel shift/scale vectors from the precomputed timestep branch."""
    return layer_norm(x, eps) * (1.0 + np.asarray(scale, np.float64)) + np.asarray(shift, np.float64)


# --------------------------------------------------------------------------
# 3D RoPE ([steinslab] "极简主控逻辑": spatial RoPE over (t, h, w);
# [linlog] "音频处理": audio rows share the rotary timeline)
# --------------------------------------------------------------------------
def rope_angles(pos, cfg: BlockConfig) -> np.ndarray:
    """Rotation angle of every interleaved pair of a head: [N, Dh/2].

    The head dimension is split into three sections, one per position axis
    (t, y, x); pair i of a section of width s turns by pos_axis *
    theta^(-2i/s)."""
    pos = np.asarray(pos, dtype=np.float64)
    cols = []
    for axis, sec in enumerate(cfg.rope_sections):
        i = np.arange(sec // 2, dtype=np.float64)
        omega = cfg.rope_theta ** (-2.0 * i / sec)
        cols.append(pos[:, axis:axis + 1] * omega[None, :])
    return np.concatenate(cols, axis=1)


def apply_rope(t, pos, cfg: BlockConfig) -> np.ndarray:
    """Rotate pairs (2i, 2i+1) of every head of t [N, H, Dh] by the angles
    of ``rope_angles``: (a, b) -> (a cos - b sin, a sin + b cos)."""
    t = np.asarray(t, dtype=np.float64)
    ang = rope_angles(pos, cfg)                       # [N, Dh/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a = t[..., 0::2]
    b = t[..., 1::2]
    out = np.empty_like(t)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


# --------------------------------------------------------------------------
# full attention ([alphalab] model facts: full attention, single stream)
# --------------------------------------------------------------------------
def attention(q, k, v, rows=None) -> np.ndarray:
    """Non-causal softmax attention per head, no mask.

    q, k, v: [H, N, Dh].  Returns [H, len(rows) or N, Dh] with
    o = softmax(q k^T / sqrt(Dh)) v over all N keys."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if rows is not None:
        q = q[:, rows, :]
    dh = q.shape[-1]
    out = np.empty((q.shape[0], q.shape[1], v.shape[-1]))
    for h in range(q.shape[0]):
        s = (q[h] @ k[h].T) / math.sqrt(dh)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[h] = p @ v[h]
    return out


# --------------------------------------------------------------------------
# MLP ([linlog] "int8 量化": FC1 / FC2 of the block MLP)
# --------------------------------------------------------------------------
def gelu_tanh(x) -> np.ndarray:
    """GELU, tanh form: x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


# --------------------------------------------------------------------------
# one block
# --------------------------------------------------------------------------
def _split_heads(t, cfg: BlockConfig) -> np.ndarray:
    """[N, d] -> [H, N, Dh]: channel c belongs to head c // Dh."""
    n = t.shape[0]
    return t.reshape(n, cfg.heads, cfg.head_dim).transpose(1, 0, 2)


def _merge_heads(t) -> np.ndarray:
    """[H, N, Dh] -> [N, H*Dh]."""
    h, n, dh = t.shape
    return t.transpose(1, 0, 2).reshape(n, h * dh)


def segment_mod(mod_seg, starts, n_tokens: int) -> np.ndarray:
    """Per-token modulation [6, N, d] from per-segment vectors.

    [linlog] "音频处理": the reference audio is conditioned at its own timestep
    (1.0), so its precomputed AdaLN vectors differ from the video's; each
    segment of consecutive tokens has its own [6, d] set.  mod_seg [S, 6, d];
    segment s covers tokens starts[s] .. starts[s+1]-1 (starts[0] = 0, the
    last segment runs to the end)."""
    mod_seg = np.asarray(mod_seg, dtype=np.float64)
    starts = list(starts) + [n_tokens]
    assert starts[0] == 0 and len(starts) == mod_seg.shape[0] + 1
    seg = np.zeros(n_tokens, dtype=np.int64)
    for s_ in range(mod_seg.shape[0]):
        seg[starts[s_]:starts[s_ + 1]] = s_
    return mod_seg[seg].transpose(1, 0, 2)


def _mod_parts(mod, sel):
    """(shift1, scale1, gate1, shift2, scale2, gate2) of a [6, d] or per-token
    [6, N, d] modulation; the last four restricted to the rows ``sel``."""
    mod = np.asarray(mod, dtype=np.float64)
    shift1, scale1, gate1, shift2, scale2, gate2 = mod
    if mod.ndim == 3:
        gate1, shift2, scale2, gate2 = (v[sel] for v in (gate1, shift2, scale2, gate2))
    return shift1, scale1, gate1, shift2, scale2, gate2


def block_forward(x, w: Dict[str, np.ndarray], mod, pos, cfg: BlockConfig,
                  bf16_storage: bool = False, rows=None, return_parts: bool = False):
    """One dense single-stream DiT block, fp64.

    x [N, d]; w: w_qkv [3d, d], w_o [d, d], w1 [F, d], w2 [d, F] (rows are
    output channels); mod [6, d] = shift1, scale1, gate1, shift2, scale2,
    gate2, or per token [6, N, d] (``segment_mod``); pos [N, 3].

    Steps ([linlog] "DiT 融合内核" names the gated-AdaLN pairs; [alphalab]
    the full attention):
      h  = AdaLN(x; shift1, scale1)
      q, k, v = split(h W_qkv^T); q, k rotated by 3D RoPE
      o  = softmax(q k^T / sqrt(Dh)) v, heads concatenated
      x1 = x + gate1 * (o W_o^T)
      h2 = AdaLN(x1; shift2, scale2)
      x2 = x1 + gate2 * (GELU(h2 W1^T) W2^T)

    ``bf16_storage`` rounds every tensor a BF16 pipeline stores (h, q, k, v,
    o, a, x1, h2, u, m, x2) to BF16.  ``rows`` evaluates the output only for
    those query rows (keys and values still come from every token)."""
    R = lambda a: _maybe_round(a, bf16_storage)
    x = np.asarray(x, dtype=np.float64)
    sel = slice(None) if rows is None else np.asarray(rows)
    shift1, scale1, gate1, shift2, scale2, gate2 = _mod_parts(mod, sel)
    d = cfg.d
    h = R(adaln(x, shift1, scale1, cfg.eps))
    qkv = h @ np.asarray(w["w_qkv"], np.float64).T
    q = R(apply_rope(_split_heads(qkv[:, 0:d], cfg).transpose(1, 0, 2), pos, cfg)).transpose(1, 0, 2)
    k = R(apply_rope(_split_heads(qkv[:, d:2 * d], cfg).transpose(1, 0, 2), pos, cfg)).transpose(1, 0, 2)
    v = R(_split_heads(qkv[:, 2 * d:3 * d], cfg))
    o = R(_merge_heads(attention(q, k, v, rows=rows)))
    a = R(o @ np.asarray(w["w_o"], np.float64).T)
    x1 = R(x[sel] + gate1 * a)
    h2 = R(adaln(x1, shift2, scale2, cfg.eps))
    u = R(gelu_tanh(h2 @ np.asarray(w["w1"], np.float64).T))
    m = R(u @ np.asarray(w["w2"], np.float64).T)
    x2 = R(x1 + gate2 * m)
    if return_parts:
        return x2, dict(h=h, q=q, k=k, v=v, o=o, a=a, x1=x1, h2=h2, u=u, m=m)
    return x2


def block_flops(n: int, cfg: BlockConfig) -> float:
    """Multiply-add count x2 of one block: four projections plus the two
    attention contractions (q k^T and p v)."""
    d, f = cfg.d, cfg.ffn
    gemm = 2.0 * n * d * (3 * d) + 2.0 * n * d * d + 2.0 * n * d * f * 2
    attn = 4.0 * n * n * d
    return gemm + attn


# --------------------------------------------------------------------------
# final layer ([linlog] "DiT 融合内核": final-layer binding)
# --------------------------------------------------------------------------
def final_head(x, row_start: int, rows: int, shift, scale, w, eps: float, bf16_storage: bool = False):
    """One output head of the final layer: the rows row_start .. row_start +
    rows - 1 of the residual stream, normalised with the head's own AdaLN
    vectors (the audio and video heads read their rows in place), projected
    by w [c_out, d]: out = AdaLN(x[rows]) w^T.  ``bf16_storage`` rounds the
    normalised operand and the output to BF16, as a BF16 head does."""
    R = lambda a: _maybe_round(a, bf16_storage)
    xs = np.asarray(x, dtype=np.float64)[row_start:row_start + rows]
    h = R(adaln(xs, np.asarray(shift, np.float64), np.asarray(scale, np.float64), eps))
    return R(h @ np.asarray(w, np.float64).T)


# --------------------------------------------------------------------------
# core residual reuse ([linlog] speed/quality preset table, "--core-reuse":
# every step refreshes the patch and head, the block core runs less often)
# --------------------------------------------------------------------------
def core_residual(x_in, x_out) -> np.ndarray:
    """The core's residual, x_out - x_in, kept at full precision."""
    return np.asarray(x_out, np.float64) - np.asarray(x_in, np.float64)


def core_reuse(x, delta, bf16_storage: bool = True) -> np.ndarray:
    """A reuse step: the core's cached residual added to this step's core
    input in place of running the blocks; the stream stays BF16."""
    return _maybe_round(np.asarray(x, np.float64) + np.asarray(delta, np.float64), bf16_storage)


# --------------------------------------------------------------------------
# token reduction ([linlog] "Token 缩减：28% 的去噪时间消减")
# --------------------------------------------------------------------------
def reduced_token_count(n_tokens: int, grid: VideoGrid) -> int:
    """Tokens left after pairing: every (t, y) video row keeps ceil(W/2)."""
    return n_tokens - grid.T * grid.Hh * (grid.W - grid.w_reduced)


def _reduce_map(n_tokens: int, grid: VideoGrid):
    """For each reduced row, the list of full rows it stands for."""
    groups = []
    for i in range(grid.offset):
        groups.append([i])
    for t in range(grid.T):
        for y in range(grid.Hh):
            base = grid.offset + (t * grid.Hh + y) * grid.W
            for j in range(grid.w_reduced):
                c0 = 2 * j
                if c0 + 1 < grid.W:
                    groups.append([base + c0, base + c0 + 1])
                else:
                    groups.append([base + c0])
    for i in range(grid.offset + grid.n_video, n_tokens):
        groups.append([i])
    return groups


def token_reduce(x_full, grid: VideoGrid, bf16_storage: bool = False):
    """Pair horizontally adjacent target-video tokens (columns 2j, 2j+1 of
    every (t, y) row) into their mean; all other tokens are copied.  Returns
    (x_reduced, side) with side the untouched full-resolution state."""
    x_full = np.asarray(x_full, dtype=np.float64)
    groups = _reduce_map(x_full.shape[0], grid)
    red = np.stack([x_full[g].mean(axis=0) for g in groups])
    return _maybe_round(red, bf16_storage), x_full.copy()


def token_restore(x_red, side, grid: VideoGrid, bf16_storage: bool = False):
    """Back to full resolution.  A paired video token returns its own side
    value plus its pair's update, update = (current reduced value) - (the
    value the pair held when it was reduced, i.e. the pair mean of side).
    An unpaired token (text, audio, an odd last column) takes its current
    reduced value."""
    x_red = np.asarray(x_red, dtype=np.float64)
    side = np.asarray(side, dtype=np.float64)
    groups = _reduce_map(side.shape[0], grid)
    out = np.empty_like(side)
    for p, g in enumerate(groups):
        if len(g) == 2:
            at_reduce = _maybe_round(side[g].mean(axis=0), bf16_storage)
            upd = x_red[p] - at_reduce
            for i in g:
                out[i] = side[i] + upd
        else:
            out[g[0]] = x_red[p]
    return _maybe_round(out, bf16_storage)


def reduced_positions(pos, grid: VideoGrid) -> np.ndarray:
    """Position of a reduced token: the mean of its members' positions
    (a pair (t, y, 2j), (t, y, 2j+1) sits at (t, y, 2j + 0.5))."""
    pos = np.asarray(pos, dtype=np.float64)
    groups = _reduce_map(pos.shape[0], grid)
    return np.stack([pos[g].mean(axis=0) for g in groups])


# --------------------------------------------------------------------------
# the denoiser step ([alphalab] 50 layers; [linlog] AdaLN precomputed per
# block, token reduction boundaries)
# --------------------------------------------------------------------------
def _reduce_mod_rows(mod, grid: VideoGrid, n_tokens: int):
    """A per-token modulation [6, N, d] for the reduced sequence: each
    reduced token takes its first member's vectors (members of a pair are
    adjacent video tokens of one segment).  [6, d] passes through."""
    mod = np.asarray(mod, dtype=np.float64)
    if mod.ndim == 2:
        return mod
    first = [g[0] for g in _reduce_map(n_tokens, grid)]
    return mod[:, first, :]


def step_forward(x, weights: List[Dict[str, np.ndarray]], mods, pos, cfg: BlockConfig,
                 reduction: Optional[Reduction] = None, bf16_storage: bool = False,
                 int8: bool = False, which=None):
    """Run the blocks in order with their own weights and modulation (each
    [6, d] or per token [6, N, d] at full resolution).  With a reduction, the
    sequence is reduced after block ``reduce_after_block`` and restored
    before block ``restore_before_block``."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.float64)
    n_full = x.shape[0]
    cur, cur_pos, side = x, pos, None
    for b, (w, mod) in enumerate(zip(weights, mods)):
        if reduction is not None and side is not None and b == reduction.restore_before_block:
            cur = token_restore(cur, side, reduction.grid, bf16_storage)
            cur_pos, side = pos, None
        if side is not None:
            mod = _reduce_mod_rows(mod, reduction.grid, n_full)
        if int8:
            cur = block_forward_int8(cur, w, mod, cur_pos, cfg, bf16_storage=bf16_storage,
                                     which=INT8_ALL if which is None else which)
        else:
            cur = block_forward(cur, w, mod, cur_pos, cfg, bf16_storage=bf16_storage)
        if (reduction is not None and b == reduction.reduce_after_block
                and b + 1 < reduction.restore_before_block and b + 1 < len(weights)):
            cur, side = token_reduce(cur, reduction.grid, bf16_storage)
            cur_pos = (reduced_positions(pos, reduction.grid) if reduction.pos_reduced is None
                       else np.asarray(reduction.pos_reduced, np.float64))
    if side is not None:
        cur = token_restore(cur, side, reduction.grid, bf16_storage)
    return cur


# --------------------------------------------------------------------------
# dynamic int8 ([linlog] "int8 量化：从 36 秒到 19 秒")
# --------------------------------------------------------------------------
def quantize_rows(x, group: Optional[int] = None):
    """Symmetric absmax quantisation of each row (or each ``group`` of
    consecutive columns of a row).

    The decision is taken in IEEE binary32, the precision the kernels use:
    s = absmax / 127 (correctly rounded), q = clamp(rne(x / s), -127, 127)
    with x / s correctly rounded; a group of zeros gives s = 0 and q = 0.
    Returns (q int8 [R, C], s float32 [R, C/group])."""
    x = np.asarray(x, dtype=np.float32)
    r, c = x.shape
    g = c if group is None else group
    assert c % g == 0
    xg = x.reshape(r, c // g, g)
    amax = np.abs(xg).max(axis=2)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s)
    y = (xg / safe[:, :, None]).astype(np.float32)
    q = np.clip(np.rint(y), -127, 127)              # rint rounds half to even
    q = np.where(s[:, :, None] == 0, 0, q)
    return q.reshape(r, c).astype(np.int8), s


def quantize_weight(w):
    """Per-output-channel (per row of W [out, in]) int8 weights: the same rule
    as ``quantize_rows`` with one scale per row."""
    return quantize_rows(w, None)


def gemm_int(aq, bq) -> np.ndarray:
    """Exact integer product acc[t, n] = sum_k a[t, k] * b[n, k], as int64.

    Computed with a float64 matmul: the operands are integers of magnitude
    <= 127, so every product and every partial sum is an integer of
    magnitude <= 127^2 * K, far below 2^53 for any K here; float64 holds all
    of them exactly and the result is the exact integer sum in any summation
    order (the same value an int64 matmul gives, at BLAS speed)."""
    a = np.asarray(aq, np.float64)
    b = np.asarray(bq, np.float64)
    assert a.shape[1] == b.shape[1] and 127 * 127 * a.shape[1] < 2 ** 53
    return (a @ b.T).astype(np.int64)


def linear_int8(xq, xs, wq, ws) -> np.ndarray:
    """Dequantised int8 projection: acc[t, n] * s_x[t] * s_w[n]."""
    acc = gemm_int(xq, wq).astype(np.float64)
    return acc * np.asarray(xs, np.float64).reshape(-1, 1) * np.asarray(ws, np.float64).reshape(1, -1)


def fc2_int8(uq, us, wq, ws, group: int = 1024) -> np.ndarray:
    """FC2 with one activation scale per ``group`` input channels:
    m[t, n] = s_w[n] * sum_g s_u[t, g] * acc_g[t, n], acc_g the exact integer
    sum over channels g*group .. g*group+group-1."""
    uq = np.asarray(uq, np.int64)
    wq = np.asarray(wq, np.int64)
    us = np.asarray(us, np.float64)
    f = uq.shape[1]
    out = np.zeros((uq.shape[0], wq.shape[0]))
    for g in range(f // group):
        sl = slice(g * group, (g + 1) * group)
        acc = (uq[:, sl] @ wq[:, sl].T).astype(np.float64)
        out += us[:, g:g + 1] * acc
    return out * np.asarray(ws, np.float64).reshape(1, -1)


INT8_ALL = ("qkv", "o", "fc1", "fc2")
INT8_MLP = ("fc1", "fc2")
INT8_QKV = ("qkv",)


def block_forward_int8(x, w: Dict[str, np.ndarray], mod, pos, cfg: BlockConfig,
                       bf16_storage: bool = True, fc2_group: int = 1024, return_parts: bool = False,
                       rows=None, which=INT8_ALL):
    """The block of ``block_forward`` on the dynamic-int8 path.

    ``which`` names the projections that run in int8 ([linlog] "int8 量化":
    the MLP alone, QKV alone, or all four); the others use the BF16 weights
    ``w_qkv, w_o, w1, w2`` exactly as ``block_forward``.  For an int8
    projection w holds int8 codes (``q_qkv, q_o, q1, q2``) and fp32
    per-output-channel scales (``s_qkv, s_o, s1, s2``).  QKV, out-projection
    and FC1 quantise their input per token; FC2 quantises per token and per
    ``fc2_group`` input channels.  Attention itself stays in floating point.
    ``rows`` evaluates the output only for those query rows (every
    quantisation after QKV is per token, so the rows are independent once keys
    and values exist)."""
    R = lambda a: _maybe_round(a, bf16_storage)
    x = np.asarray(x, dtype=np.float64)
    sel = slice(None) if rows is None else np.asarray(rows)
    shift1, scale1, gate1, shift2, scale2, gate2 = _mod_parts(mod, sel)
    d = cfg.d
    f = cfg.ffn
    g2 = min(fc2_group, f)
    h = R(adaln(x, shift1, scale1, cfg.eps))
    if "qkv" in which:
        hq, hs = quantize_rows(h)
        qkv = linear_int8(hq, hs, w["q_qkv"], w["s_qkv"])
    else:
        hq = hs = None
        qkv = h @ np.asarray(w["w_qkv"], np.float64).T
    q = R(apply_rope(_split_heads(qkv[:, 0:d], cfg).transpose(1, 0, 2), pos, cfg)).transpose(1, 0, 2)
    k = R(apply_rope(_split_heads(qkv[:, d:2 * d], cfg).transpose(1, 0, 2), pos, cfg)).transpose(1, 0, 2)
    v = R(_split_heads(qkv[:, 2 * d:3 * d], cfg))
    o = R(_merge_heads(attention(q, k, v, rows=rows)))
    if "o" in which:
        oq, os_ = quantize_rows(o)
        a = R(linear_int8(oq, os_, w["q_o"], w["s_o"]))
    else:
        oq = os_ = None
        a = R(o @ np.asarray(w["w_o"], np.float64).T)
    x1 = R(x[sel] + gate1 * a)
    h2 = R(adaln(x1, shift2, scale2, cfg.eps))
    if "fc1" in which:
        h2q, h2s = quantize_rows(h2)
        u = R(gelu_tanh(linear_int8(h2q, h2s, w["q1"], w["s1"])))
    else:
        h2q = h2s = None
        u = R(gelu_tanh(h2 @ np.asarray(w["w1"], np.float64).T))
    if "fc2" in which:
        uq, us = quantize_rows(u, g2)
        m = R(fc2_int8(uq, us, w["q2"], w["s2"], g2))
    else:
        uq = us = None
        m = R(u @ np.asarray(w["w2"], np.float64).T)
    x2 = R(x1 + gate2 * m)
    if return_parts:
        return x2, dict(h=h, hq=hq, hs=hs, qkv=qkv, q=q, k=k, v=v, o=o, oq=oq, os=os_, a=a,
                        x1=x1, h2=h2, h2q=h2q, h2s=h2s, u=u, uq=uq, us=us, m=m)
    return x2
