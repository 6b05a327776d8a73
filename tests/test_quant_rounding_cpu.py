"""The quantisers' rounding shortcut, checked in IEEE binary32 on the CPU.

The int8 code of x at scale s is rne(fl(x / s)) clamped to +-127 ([linlog]
"int8 量化：从 36 秒到 19 秒": dynamic per-token activation scales).  The
kernels form t = fl(x * fl(1 / s)) instead of the division and use rne(t)
unless |t - rne(t)| >= 0.4999 (t within 1e-4 of a half-integer), where they
divide.  Since
|x / s| <= 127.x, t is within 128 * 2^-23 of x / s and fl(x / s) within
128 * 2^-24 of it, so outside that band both round to the same integer.
This test replays the shortcut with numpy float32 arithmetic (correctly
rounded like the kernels' fp32 multiply and reciprocal) over every positive
normal BF16 value up to amax, for random BF16 amax values."""
import numpy as np


def test_reciprocal_shortcut_matches_division():
    rng = np.random.default_rng(11)
    bits = np.arange(0x0080, 0x7F80, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    amaxes = list(vals[rng.integers(0, len(vals), 500)]) + [np.float32(127.0), np.float32(96.0)]
    checked = 0
    for a in amaxes:
        s = np.float32(np.float32(a) / np.float32(127.0))
        if not s >= np.float32(2.0 ** -100):
            continue                      # the kernels divide for such scales
        r = np.float32(np.float32(1.0) / s)
        xs = vals[vals <= a]
        xs = np.concatenate([xs, -xs])
        t = (xs * r).astype(np.float32)
        f = (xs / s).astype(np.float32)
        c = np.rint(t)
        fast = np.abs((t - c).astype(np.float32)) < np.float32(0.4999)
        assert np.array_equal(c[fast], np.rint(f[fast]))
        checked += int(fast.sum())
    assert checked > 10_000_000
