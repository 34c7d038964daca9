"""Exact tiled attention (forward + backward) for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libattn.so`` built from ``csrc/``
(hand-written tcgen05 / TMA kernels).  ``attn`` is its thin ctypes binding;
``inputs`` draws the seeded synthetic workloads.  Importing the package does
not load the library; the first use of ``attn`` does, and fails loudly if the
library has not been built.
"""
import importlib

__all__ = ["attn", "inputs", "build"]


def __getattr__(name):
    if name in ("attn", "inputs", "build"):
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
