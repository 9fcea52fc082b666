"""GB300-native MSA (MiniMax Sparse Attention) training hot path.

libmsa.so (csrc/, C ABI in include/msa.h) holds every kernel; this package is the
thin Python binding (`ops`, `_lib`) plus the seeded synthetic inputs (`synth`).
"""
from . import synth  # noqa: F401

__all__ = ["synth", "ops", "_lib"]


def __getattr__(name):
    # the binding imports torch and loads the CUDA library: only on first use
    if name in ("ops", "_lib"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
