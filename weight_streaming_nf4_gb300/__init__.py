"""GB300-native streamed NF4-LoRA linear (frozen NF4 base + rank-16 LoRA).

The compute path lives in ``libwsnf4.so`` (hand-written CUDA for sm_103a
behind a C ABI, declared in ``include/wsnf4.h``).  ``ops`` is the thin ctypes
binding with the same names as the C entry points; importing it loads the
library and raises if it is missing -- there is no fallback path.
``synth`` holds the seeded synthetic input generators.
"""
import importlib

__all__ = ["ops", "synth", "build", "stack"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
