"""GB300-native K-tiled, operand-staged GEMM: C = A.B, f16 in, f32 accumulate.

The compute path is the CUDA library ``libtsm_gemm.so`` (sm_103a: TMA into a
shared-memory ring, tcgen05 MMA into TMEM, split-K with a fixed-order
reduction).  ``binding`` is a thin ctypes layer over its C ABI
(``include/tsm_gemm.h``); importing it loads the library and raises if it is
missing -- there is no CPU fallback.  ``synthetic`` draws seeded operands.
"""
import importlib

__all__ = ["binding", "synthetic"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
