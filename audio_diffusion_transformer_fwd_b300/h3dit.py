"""ctypes binding of libh3dit.so: the C ABI of ``include/h3dit.h`` under the
same names.  Argument marshalling only: every step of the path runs in the
library's CUDA kernels.  Tensors may be passed as torch tensors (their
``data_ptr()`` is used) or as raw integer addresses; streams as
``torch.cuda.Stream`` objects, raw handles or None (the current torch
stream).

The library is loaded on first use.  If it is missing or fails to load the
call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libh3dit.so")

OK, E_INVAL, E_UNSUPPORTED, E_NOMEM, E_CUDA, E_TIMEOUT = range(6)
BF16, INT8, INT8_MLP, INT8_QKV = 0, 1, 2, 3
# kernel classes of h3dit_timing_read
KC_ROWS, KC_QKV, KC_ATTN, KC_OPROJ, KC_FC1, KC_FC2, KC_REDUCE, KC_QUANT = range(8)

_EXPORTS = [
    "h3dit_last_error", "h3dit_version", "h3dit_check_device_error",
    "h3dit_timing_enable", "h3dit_timing_reset", "h3dit_timing_read",
    "h3dit_workspace_size", "h3dit_block_forward", "h3dit_block_forward_noalloc", "h3dit_step_forward",
    "h3dit_block_forward_seg", "h3dit_step_forward_seg", "h3dit_final_layer", "h3dit_core_residual",
    "h3dit_core_reuse",
    "h3dit_quantize_act", "h3dit_quantize_weight",
    "h3dit_reduced_tokens", "h3dit_token_reduce", "h3dit_token_restore", "h3dit_reduced_positions",
    "h3dit_adaln", "h3dit_gate_residual_adaln", "h3dit_rope_table", "h3dit_qkv_project",
    "h3dit_attention", "h3dit_linear",
    "h3dit_quantize_codes", "h3dit_widen_codes", "h3dit_linear_i8", "h3dit_linear_i8_acc",
    "h3dit_adaln_quant", "h3dit_gate_residual_adaln_quant", "h3dit_qkv_project_i8",
    "h3dit_test_set_wait_limit", "h3dit_test_stall_next_gemm",
]


class H3DitError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"h3dit status {status}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("ffn", ctypes.c_int), ("eps", ctypes.c_float), ("rope_sections", ctypes.c_int * 3),
                ("rope_theta", ctypes.c_float), ("precision", ctypes.c_int)]


class BlockWeights(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("w1", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("s_qkv", ctypes.c_void_p), ("s_o", ctypes.c_void_p),
                ("s1", ctypes.c_void_p), ("s2", ctypes.c_void_p), ("codes_int8", ctypes.c_int)]


class VideoGrid(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int), ("T", ctypes.c_int), ("Hh", ctypes.c_int), ("W", ctypes.c_int)]


class Segments(ctypes.Structure):
    _fields_ = [("count", ctypes.c_int), ("start", ctypes.c_int * 4)]


class FinalHead(ctypes.Structure):
    _fields_ = [("row_start", ctypes.c_int), ("rows", ctypes.c_int), ("shift", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("w", ctypes.c_void_p), ("c_out", ctypes.c_int), ("out", ctypes.c_void_p)]


class Reduction(ctypes.Structure):
    _fields_ = [("grid", VideoGrid), ("reduce_after_block", ctypes.c_int),
                ("restore_before_block", ctypes.c_int), ("pos_reduced", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded library (raises if it is absent)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise H3DitError(E_CUDA, f"{LIB_PATH} is not built; run "
                             "`python -m audio_diffusion_transformer_fwd_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        P = ctypes.POINTER
        sig = {
            "h3dit_last_error": (ctypes.c_char_p, []),
            "h3dit_version": (i, []),
            "h3dit_check_device_error": (i, [vp]),
            "h3dit_test_set_wait_limit": (i, [ctypes.c_ulonglong]),
            "h3dit_test_stall_next_gemm": (i, [i]),
            "h3dit_timing_enable": (i, [i]),
            "h3dit_timing_reset": (i, []),
            "h3dit_timing_read": (i, [i, P(ctypes.c_double), P(ctypes.c_longlong)]),
            "h3dit_workspace_size": (i, [P(Config), i, P(Reduction), P(sz)]),
            "h3dit_block_forward": (i, [P(Config), P(BlockWeights), vp, vp, vp, i, vp, sz, vp]),
            "h3dit_block_forward_noalloc": (i, [P(Config), P(BlockWeights), vp, vp, vp, i, vp]),
            "h3dit_step_forward": (i, [P(Config), P(BlockWeights), i, vp, vp, vp, i, P(Reduction), vp, sz, vp]),
            "h3dit_final_layer": (i, [P(Config), vp, i, P(FinalHead), i, vp]),
            "h3dit_core_residual": (i, [vp, vp, sz, vp, vp]),
            "h3dit_core_reuse": (i, [vp, vp, sz, vp]),
            "h3dit_block_forward_seg": (i, [P(Config), P(BlockWeights), vp, P(Segments), vp, vp, i, vp, sz, vp]),
            "h3dit_step_forward_seg": (i, [P(Config), P(BlockWeights), i, vp, P(Segments), vp, vp, i, P(Reduction),
                                           vp, sz, vp]),
            "h3dit_quantize_act": (i, [vp, i, i, i, vp, vp, vp]),
            "h3dit_quantize_weight": (i, [vp, i, i, vp, vp, vp]),
            "h3dit_reduced_tokens": (i, [i, P(VideoGrid)]),
            "h3dit_token_reduce": (i, [vp, i, i, P(VideoGrid), vp, vp, vp]),
            "h3dit_token_restore": (i, [vp, vp, i, i, P(VideoGrid), vp, vp]),
            "h3dit_reduced_positions": (i, [vp, i, P(VideoGrid), vp, vp]),
            "h3dit_adaln": (i, [P(Config), vp, vp, vp, i, vp, vp]),
            "h3dit_gate_residual_adaln": (i, [P(Config), vp, vp, vp, vp, vp, i, vp, vp]),
            "h3dit_rope_table": (i, [P(Config), vp, i, vp, vp]),
            "h3dit_qkv_project": (i, [P(Config), vp, vp, vp, i, vp, vp, vp, i, vp]),
            "h3dit_attention": (i, [P(Config), vp, vp, vp, i, i, vp, vp]),
            "h3dit_linear": (i, [vp, vp, i, i, i, i, vp, vp]),
            "h3dit_quantize_codes": (i, [vp, i, i, i, vp, vp, vp]),
            "h3dit_widen_codes": (i, [vp, sz, vp, vp]),
            "h3dit_linear_i8": (i, [vp, vp, i, vp, vp, i, i, i, i, vp, vp]),
            "h3dit_linear_i8_acc": (i, [vp, vp, i, i, i, vp, vp]),
            "h3dit_adaln_quant": (i, [P(Config), vp, vp, vp, i, vp, vp, vp]),
            "h3dit_gate_residual_adaln_quant": (i, [P(Config), vp, vp, vp, vp, vp, i, vp, vp, vp]),
            "h3dit_qkv_project_i8": (i, [P(Config), vp, vp, vp, vp, vp, i, vp, vp, vp, i, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int):
    if st != OK:
        raise H3DitError(st, lib().h3dit_last_error().decode())


@dataclass
class BlockShape:
    d: int
    heads: int
    head_dim: int
    ffn: int
    eps: float = 1e-6
    rope_sections: Sequence[int] = (32, 48, 48)
    rope_theta: float = 10000.0
    precision: int = BF16

    def c(self) -> Config:
        c = Config()
        c.d, c.heads, c.head_dim, c.ffn = self.d, self.heads, self.head_dim, self.ffn
        c.eps = self.eps
        for k in range(3):
            c.rope_sections[k] = int(self.rope_sections[k])
        c.rope_theta = self.rope_theta
        c.precision = self.precision
        return c


def block_weights(w_qkv, w_o, w1, w2, s_qkv=None, s_o=None, s1=None, s2=None, codes_int8=False) -> BlockWeights:
    bw = BlockWeights()
    bw.w_qkv, bw.w_o, bw.w1, bw.w2 = _ptr(w_qkv), _ptr(w_o), _ptr(w1), _ptr(w2)
    bw.s_qkv, bw.s_o, bw.s1, bw.s2 = _ptr(s_qkv), _ptr(s_o), _ptr(s1), _ptr(s2)
    bw.codes_int8 = 1 if codes_int8 else 0
    return bw


def video_grid(offset: int, T: int, Hh: int, W: int) -> VideoGrid:
    g = VideoGrid()
    g.offset, g.T, g.Hh, g.W = offset, T, Hh, W
    return g


def reduction(grid: VideoGrid, reduce_after_block: int = 3, restore_before_block: int = 40,
              pos_reduced=None) -> Reduction:
    r = Reduction()
    r.grid = grid
    r.reduce_after_block = reduce_after_block
    r.restore_before_block = restore_before_block
    r.pos_reduced = _ptr(pos_reduced)
    return r


# ---------------------------------------------------------------- entry points
def h3dit_version() -> int:
    return lib().h3dit_version()


def h3dit_check_device_error(stream=None):
    _check(lib().h3dit_check_device_error(_stream(stream)))


def h3dit_test_set_wait_limit(ns: int):
    """Device-side limit of every pipeline wait, in ns (0 = the default 2 s)."""
    _check(lib().h3dit_test_set_wait_limit(ns))


def h3dit_test_stall_next_gemm(kblock: int):
    """Make the next BF16 projection's first CTA stop loading at ``kblock``
    (its wait then runs out; -1 cancels)."""
    _check(lib().h3dit_test_stall_next_gemm(kblock))


def h3dit_timing_enable(on: bool):
    _check(lib().h3dit_timing_enable(1 if on else 0))


def h3dit_timing_reset():
    _check(lib().h3dit_timing_reset())


def h3dit_timing_read(kernel_class: int):
    ms = ctypes.c_double()
    n = ctypes.c_longlong()
    _check(lib().h3dit_timing_read(kernel_class, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def h3dit_workspace_size(shape: BlockShape, n_tokens: int, tr: Optional[Reduction] = None) -> int:
    out = ctypes.c_size_t()
    _check(lib().h3dit_workspace_size(ctypes.byref(shape.c()), n_tokens,
                                      ctypes.byref(tr) if tr is not None else None, ctypes.byref(out)))
    return out.value


def h3dit_block_forward(shape: BlockShape, w: BlockWeights, mod, x, pos, n_tokens: int, ws, ws_bytes: int,
                        stream=None):
    _check(lib().h3dit_block_forward(ctypes.byref(shape.c()), ctypes.byref(w), _ptr(mod), _ptr(x), _ptr(pos),
                                     n_tokens, _ptr(ws), ws_bytes, _stream(stream)))


def h3dit_block_forward_noalloc(shape: BlockShape, w: BlockWeights, mod, x, pos, n_tokens: int, stream=None):
    """h3dit_block_forward with the library's built-in 64 MiB scratch instead of
    a caller workspace (for callers that cannot allocate device memory)."""
    _check(lib().h3dit_block_forward_noalloc(ctypes.byref(shape.c()), ctypes.byref(w), _ptr(mod), _ptr(x),
                                             _ptr(pos), n_tokens, _stream(stream)))


def h3dit_step_forward(shape: BlockShape, ws_list: Sequence[BlockWeights], mods, x, pos, n_tokens: int,
                       tr: Optional[Reduction], ws, ws_bytes: int, stream=None):
    arr = (BlockWeights * len(ws_list))(*ws_list)
    _check(lib().h3dit_step_forward(ctypes.byref(shape.c()), arr, len(ws_list), _ptr(mods), _ptr(x), _ptr(pos),
                                    n_tokens, ctypes.byref(tr) if tr is not None else None, _ptr(ws),
                                    ws_bytes, _stream(stream)))


def segments(starts: Sequence[int]) -> Segments:
    """Segment table from the first row of each segment (starts[0] = 0)."""
    sg = Segments()
    sg.count = len(starts)
    for k, v in enumerate(starts):
        sg.start[k] = int(v)
    return sg


def h3dit_block_forward_seg(shape: BlockShape, w: BlockWeights, mods, seg: Segments, x, pos, n_tokens: int, ws,
                            ws_bytes: int, stream=None):
    _check(lib().h3dit_block_forward_seg(ctypes.byref(shape.c()), ctypes.byref(w), _ptr(mods), ctypes.byref(seg),
                                         _ptr(x), _ptr(pos), n_tokens, _ptr(ws), ws_bytes, _stream(stream)))


def h3dit_step_forward_seg(shape: BlockShape, ws_list: Sequence[BlockWeights], mods, seg: Segments, x, pos,
                           n_tokens: int, tr: Optional[Reduction], ws, ws_bytes: int, stream=None):
    arr = (BlockWeights * len(ws_list))(*ws_list)
    _check(lib().h3dit_step_forward_seg(ctypes.byref(shape.c()), arr, len(ws_list), _ptr(mods), ctypes.byref(seg),
                                        _ptr(x), _ptr(pos), n_tokens, ctypes.byref(tr) if tr is not None else None,
                                        _ptr(ws), ws_bytes, _stream(stream)))


def final_head(row_start: int, rows: int, shift, scale, w, c_out: int, out) -> FinalHead:
    h = FinalHead()
    h.row_start, h.rows, h.c_out = row_start, rows, c_out
    h.shift, h.scale, h.w, h.out = _ptr(shift), _ptr(scale), _ptr(w), _ptr(out)
    return h


def h3dit_final_layer(shape: BlockShape, x, n_tokens: int, heads: Sequence[FinalHead], stream=None):
    arr = (FinalHead * len(heads))(*heads)
    _check(lib().h3dit_final_layer(ctypes.byref(shape.c()), _ptr(x), n_tokens, arr, len(heads), _stream(stream)))


def h3dit_core_residual(x_in, x_out, count: int, delta, stream=None):
    _check(lib().h3dit_core_residual(_ptr(x_in), _ptr(x_out), count, _ptr(delta), _stream(stream)))


def h3dit_core_reuse(x, delta, count: int, stream=None):
    _check(lib().h3dit_core_reuse(_ptr(x), _ptr(delta), count, _stream(stream)))


def h3dit_quantize_act(x, rows: int, cols: int, group: int, q, scales, stream=None):
    _check(lib().h3dit_quantize_act(_ptr(x), rows, cols, group, _ptr(q), _ptr(scales), _stream(stream)))


def h3dit_quantize_weight(w, out: int, inp: int, q, scales, stream=None):
    _check(lib().h3dit_quantize_weight(_ptr(w), out, inp, _ptr(q), _ptr(scales), _stream(stream)))


def h3dit_reduced_tokens(n_tokens: int, grid: VideoGrid) -> int:
    n = lib().h3dit_reduced_tokens(n_tokens, ctypes.byref(grid))
    if n < 0:
        raise H3DitError(E_INVAL, "video grid outside the token rows")
    return n


def h3dit_token_reduce(x_full, n_tokens: int, d: int, grid: VideoGrid, x_red, side=None, stream=None):
    _check(lib().h3dit_token_reduce(_ptr(x_full), n_tokens, d, ctypes.byref(grid), _ptr(x_red), _ptr(side),
                                    _stream(stream)))


def h3dit_token_restore(x_red, side, n_tokens: int, d: int, grid: VideoGrid, x_full, stream=None):
    _check(lib().h3dit_token_restore(_ptr(x_red), _ptr(side), n_tokens, d, ctypes.byref(grid), _ptr(x_full),
                                     _stream(stream)))


def h3dit_reduced_positions(pos, n_tokens: int, grid: VideoGrid, pos_red, stream=None):
    _check(lib().h3dit_reduced_positions(_ptr(pos), n_tokens, ctypes.byref(grid), _ptr(pos_red),
                                         _stream(stream)))


def h3dit_adaln(shape: BlockShape, x, shift, scale, n_tokens: int, h, stream=None):
    _check(lib().h3dit_adaln(ctypes.byref(shape.c()), _ptr(x), _ptr(shift), _ptr(scale), n_tokens, _ptr(h),
                             _stream(stream)))


def h3dit_gate_residual_adaln(shape: BlockShape, x, branch, gate, shift, scale, n_tokens: int, h, stream=None):
    _check(lib().h3dit_gate_residual_adaln(ctypes.byref(shape.c()), _ptr(x), _ptr(branch), _ptr(gate),
                                           _ptr(shift), _ptr(scale), n_tokens, _ptr(h), _stream(stream)))


def h3dit_rope_table(shape: BlockShape, pos, n_tokens: int, table, stream=None):
    _check(lib().h3dit_rope_table(ctypes.byref(shape.c()), _ptr(pos), n_tokens, _ptr(table), _stream(stream)))


def h3dit_qkv_project(shape: BlockShape, h, w_qkv, table, n_tokens: int, q, k, vt, vt_ld: int, stream=None):
    _check(lib().h3dit_qkv_project(ctypes.byref(shape.c()), _ptr(h), _ptr(w_qkv), _ptr(table), n_tokens,
                                   _ptr(q), _ptr(k), _ptr(vt), vt_ld, _stream(stream)))


def h3dit_attention(shape: BlockShape, q, k, vt, vt_ld: int, n_tokens: int, o, stream=None):
    _check(lib().h3dit_attention(ctypes.byref(shape.c()), _ptr(q), _ptr(k), _ptr(vt), vt_ld, n_tokens, _ptr(o),
                                 _stream(stream)))


def h3dit_linear(a, b, m: int, n: int, k: int, act: int, c, stream=None):
    _check(lib().h3dit_linear(_ptr(a), _ptr(b), m, n, k, act, _ptr(c), _stream(stream)))


def h3dit_quantize_codes(x, rows: int, cols: int, group: int, q, scales, stream=None):
    _check(lib().h3dit_quantize_codes(_ptr(x), rows, cols, group, _ptr(q), _ptr(scales), _stream(stream)))


def h3dit_widen_codes(q, count: int, out, stream=None):
    _check(lib().h3dit_widen_codes(_ptr(q), count, _ptr(out), _stream(stream)))


def h3dit_linear_i8(a_codes, sa, group: int, b_codes, sb, m: int, n: int, k: int, act: int, c, stream=None):
    _check(lib().h3dit_linear_i8(_ptr(a_codes), _ptr(sa), group, _ptr(b_codes), _ptr(sb), m, n, k, act, _ptr(c),
                                 _stream(stream)))


def h3dit_linear_i8_acc(a_codes, b_codes, m: int, n: int, k: int, acc, stream=None):
    _check(lib().h3dit_linear_i8_acc(_ptr(a_codes), _ptr(b_codes), m, n, k, _ptr(acc), _stream(stream)))


def h3dit_adaln_quant(shape: BlockShape, x, shift, scale, n_tokens: int, hq, hs, stream=None):
    c = shape.c()
    _check(lib().h3dit_adaln_quant(ctypes.byref(c), _ptr(x), _ptr(shift), _ptr(scale), n_tokens, _ptr(hq), _ptr(hs),
                                   _stream(stream)))


def h3dit_gate_residual_adaln_quant(shape: BlockShape, x, branch, gate, shift, scale, n_tokens: int, hq, hs,
                                    stream=None):
    c = shape.c()
    _check(lib().h3dit_gate_residual_adaln_quant(ctypes.byref(c), _ptr(x), _ptr(branch), _ptr(gate), _ptr(shift),
                                                 _ptr(scale), n_tokens, _ptr(hq), _ptr(hs), _stream(stream)))


def h3dit_qkv_project_i8(shape: BlockShape, hq, hs, w_qkv, s_qkv, table, n_tokens: int, q, k, vt, vt_ld: int,
                         stream=None):
    c = shape.c()
    _check(lib().h3dit_qkv_project_i8(ctypes.byref(c), _ptr(hq), _ptr(hs), _ptr(w_qkv), _ptr(s_qkv), _ptr(table),
                                      n_tokens, _ptr(q), _ptr(k), _ptr(vt), vt_ld, _stream(stream)))
