"""GB300 (sm_103a) four-layer bidirectional LSTM stack.

The compute runs in ``liblstmstack.so`` (hand-written CUDA kernels behind a C
ABI declared in ``include/lstm_stack.h``); ``binding`` marshals arguments to
it through ctypes.  The library is loaded on first use: importing this package
never needs a GPU, and every call fails loudly when the library is missing.
"""
from .synthetic import FEATURES, HIDDEN, LAYERS, GATES  # noqa: F401

__all__ = ["FEATURES", "HIDDEN", "LAYERS", "GATES"]
