"""B300-native WhiteMatter cross-layer KV pool.

The compute path is the C-ABI library ``libwm.so`` (hand-written sm_103a CUDA
kernels) built from ``csrc/``; ``wm`` is its thin ctypes binding and ``synth``
draws seeded synthetic inputs. Importing the package loads nothing native;
``wm.lib()`` loads the library and raises if it is missing.
"""

__all__ = ["synth", "wm"]
