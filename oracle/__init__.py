"""Plain CPU oracle of the WhiteMatter cross-layer KV pool forward pass.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it, to check and to time the CUDA implementation.
"""

from .whitematter import *  # noqa: F401,F403
