"""CPU oracle for the DFlash speculative round at batch 1.

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, fp64 statement of
what the GPU library computes. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the
CUDA library and its Python binding never do, and the two share no code.
"""

from .dflash_oracle import *  # noqa: F401,F403
