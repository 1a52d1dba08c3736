"""q4lin: weight-only 4-bit (Q4_G64_FP16) linear layer for GB300 (sm_103a).

The compute path is the C-ABI library ``libq4lin.so`` (hand-written CUDA);
``weight_only_bit_q4_gb300.q4lin`` is its thin ctypes binding.  Importing the
package itself loads nothing; ``synth`` and ``metrics`` are pure Python.
"""
__all__ = ["q4lin", "synth", "metrics"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
