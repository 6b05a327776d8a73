"""Helpers shared by the GPU parity tests: device copies of the seeded host
inputs and error norms.  No arithmetic of the method lives here."""
import numpy as np
import torch

import oracle as O
from audio_diffusion_transformer_fwd_b300 import h3dit as H
from audio_diffusion_transformer_fwd_b300 import synth


def dev_bf16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to("cuda").to(torch.bfloat16)


def dev_f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to("cuda")


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))


def shape_of(w: synth.Workload, precision=H.BF16) -> H.BlockShape:
    return H.BlockShape(w.d, w.heads, w.head_dim, w.ffn, w.eps, w.sections, w.theta, precision)


def oracle_cfg(w: synth.Workload) -> O.BlockConfig:
    return O.BlockConfig(d=w.d, heads=w.heads, head_dim=w.head_dim, ffn=w.ffn, eps=w.eps,
                         rope_sections=w.sections, rope_theta=w.theta)
