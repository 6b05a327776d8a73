"""Seeded synthetic inputs shaped like the MiniMax-H3 DiT workloads.

This module only draws random numbers and lays out token positions; it holds
none of the block's arithmetic.  The tests feed the same draws to the fp64
oracle and to the CUDA library, and ``bench.py`` uses it for its workloads.

Recipe (the pages publish no dataset; their workloads are prompts run through
trained weights, so seeded stand-ins with the same shapes are used):

* weights ~ N(0, 0.02^2), rounded to BF16, independent per block;
* AdaLN shift/scale/gate vectors ~ N(0, 0.1^2), fp32;
* activations x ~ N(0, 1), rounded to BF16;
* token order: target video (t-major, then y, then x), then text, then
  audio; positions video (t, y, x), text token j at (T + j) on all three
  axes, audio token k at (k // 32, 0, k % 32) (width-32 rows on the shared
  rotary timeline).

Small cases draw with numpy PCG64 on the host; the large bench workloads
draw with torch's Philox generator directly on the device.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    d: int
    heads: int
    head_dim: int
    ffn: int
    video: Tuple[int, int, int]     # T, Hh, W
    n_text: int
    n_audio: int
    n_blocks: int = 1
    eps: float = 1e-6
    sections: Tuple[int, int, int] = (32, 48, 48)
    theta: float = 10000.0
    int8: bool = False
    reduction: Optional[Tuple[int, int]] = None  # (reduce_after_block, restore_before_block)
    seed: int = 0

    @property
    def n_video(self) -> int:
        return self.video[0] * self.video[1] * self.video[2]

    @property
    def n_tokens(self) -> int:
        return self.n_video + self.n_text + self.n_audio


# The five workloads: a tiny block, one 512x512x22-frame-class block (BF16
# and dynamic int8), and the 864x480-class 50-block step without and with
# token reduction.
WORKLOADS: Dict[str, Workload] = {
    "tiny_block": Workload("tiny_block", 256, 4, 64, 1024, (2, 8, 12), 48, 16,
                           sections=(16, 24, 24)),
    "block_512": Workload("block_512", 5120, 40, 128, 20480, (6, 32, 32), 512, 256),
    "block_512_int8": Workload("block_512_int8", 5120, 40, 128, 20480, (6, 32, 32), 512, 256,
                               int8=True),
    "step_864": Workload("step_864", 5120, 40, 128, 20480, (6, 30, 54), 512, 256, n_blocks=50),
    "step_864_tr": Workload("step_864_tr", 5120, 40, 128, 20480, (6, 30, 54), 512, 256,
                            n_blocks=50, reduction=(3, 40), seed=1),
}


def positions(video: Tuple[int, int, int], n_text: int, n_audio: int) -> np.ndarray:
    """Float positions [N, 3] in token order video, text, audio."""
    T, Hh, W = video
    t, y, x = np.meshgrid(np.arange(T), np.arange(Hh), np.arange(W), indexing="ij")
    vid = np.stack([t.ravel(), y.ravel(), x.ravel()], axis=1)
    j = np.arange(n_text)
    txt = np.stack([T + j, T + j, T + j], axis=1)
    k = np.arange(n_audio)
    aud = np.stack([k // 32, np.zeros_like(k), k % 32], axis=1)
    return np.concatenate([vid, txt, aud], axis=0).astype(np.float32)


def to_bf16_values(a: np.ndarray) -> np.ndarray:
    """float32 array of the nearest BF16 values (torch's round-to-nearest-even
    cast), so that the host copy and the device BF16 tensor hold the same
    numbers."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def host_block_weights(d: int, ffn: int, seed: int, block: int = 0, std: float = 0.02) -> Dict[str, np.ndarray]:
    """One block's BF16 weights as float32 arrays (rows = output channels)."""
    r = _rng(seed, 1000 + block)
    def draw(shape):
        return to_bf16_values(r.standard_normal(shape, dtype=np.float32) * np.float32(std))
    return {
        "w_qkv": draw((3 * d, d)),
        "w_o": draw((d, d)),
        "w1": draw((ffn, d)),
        "w2": draw((d, ffn)),
    }


def host_mod(d: int, seed: int, block: int = 0, std: float = 0.1) -> np.ndarray:
    """Precomputed AdaLN vectors [6, d] (shift1, scale1, gate1, shift2,
    scale2, gate2), fp32."""
    r = _rng(seed, 2000 + block)
    return (r.standard_normal((6, d), dtype=np.float32) * np.float32(std)).astype(np.float32)


def host_activations(n: int, d: int, seed: int, std: float = 1.0) -> np.ndarray:
    r = _rng(seed, 1)
    return to_bf16_values(r.standard_normal((n, d), dtype=np.float32) * np.float32(std))


def host_int8(shape, seed: int, stream: int, lo: int = -127, hi: int = 127) -> np.ndarray:
    """Uniform int8 codes in [lo, hi]."""
    r = _rng(seed, stream)
    return r.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int8)


def host_uniform(shape, seed: int, stream: int, lo: float, hi: float) -> np.ndarray:
    r = _rng(seed, stream)
    return r.uniform(lo, hi, size=shape).astype(np.float32)


# ---- device-side draws for the large workloads -------------------------------------------
def device_block_weights(d: int, ffn: int, seed: int, block: int, device="cuda", std: float = 0.02):
    """One block's BF16 weights drawn on the device with a seeded Philox
    generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 100003 + block)
    def draw(shape):
        return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return {
        "w_qkv": draw((3 * d, d)),
        "w_o": draw((d, d)),
        "w1": draw((ffn, d)),
        "w2": draw((d, ffn)),
    }


def device_mods(n_blocks: int, d: int, seed: int, device="cuda", std: float = 0.1):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 100003 + 77777)
    return torch.randn((n_blocks, 6, d), generator=g, device=device, dtype=torch.float32) * std


def device_activations(n: int, d: int, seed: int, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 100003 + 55555)
    return torch.randn((n, d), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
