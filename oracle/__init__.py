"""fp64 CPU oracle of the MiniMax-H3 DiT block and 50-block denoiser step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, header, helper, table or constant generator with the CUDA library;
the only thing both sides consume is the seeded input generator, which holds
none of the method's arithmetic.

Parity status per function is listed in the module docstring of
``oracle.h3dit_oracle``.
"""
from .h3dit_oracle import *  # noqa: F401,F403
