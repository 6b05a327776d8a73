"""B300-native forward pass of the MiniMax-H3 DiT block and denoiser step.

The compute lives in ``libh3dit.so`` (hand-written sm_103a CUDA behind a C
ABI declared in ``include/h3dit.h``); ``audio_diffusion_transformer_fwd_b300.h3dit``
is a thin ctypes binding with the same entry-point names.  The library is
loaded on first use and its absence is an error: there is no fallback.
"""
__version__ = "0.1.0"
