"""ctypes binding of liblstmstack.so (declared in include/lstm_stack.h).

Argument marshalling only: every function here checks nothing the library
does not check again, computes nothing, and forwards to the C entry point of
the same name.  Device buffers are torch CUDA tensors (their ``data_ptr``),
streams are torch streams (their ``cuda_stream`` handle; default: the current
stream of the tensor's device).  If the library is missing, every call raises
``LibraryMissing``: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from .synthetic import FEATURES, HIDDEN, LAYERS

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblstmstack.so")
GATE_COLUMNS = 8 * HIDDEN
OUTPUT = 2 * HIDDEN

LSTM_OK = 0
LSTM_E_INVALID = 1
LSTM_E_LENGTH = 2
LSTM_E_OVERFLOW = 3
LSTM_E_DEVICE = 4
LSTM_E_CUDA = 5
LSTM_E_ALLOC = 6
LSTM_E_FAULT = 7
LSTM_MATH_3XTF32 = 0
LSTM_MATH_TF32 = 1
LSTM_GATES_IFGO = 0
LSTM_GATES_IOFC = 1
LSTM_BOTH_DIRECTIONS = 2

_c_float_p = ctypes.POINTER(ctypes.c_float)
_vp = ctypes.c_void_p


class LibraryMissing(RuntimeError):
    """liblstmstack.so has not been built (run __graft_entry__.build())."""


class LSTMError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"liblstmstack error {code}: {message}")
        self.code = code


class _Weights(ctypes.Structure):
    _fields_ = [("w", _vp * LAYERS), ("r", _vp * LAYERS), ("b", _vp * LAYERS)]


_lock = threading.Lock()
_lib = None


def load():
    """Loads liblstmstack.so (once) and declares its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise LibraryMissing(f"{LIB_PATH} not found; build it with __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        i, sz = ctypes.c_int, ctypes.c_size_t
        sig = {
            "lstm_stack_create": (i, [ctypes.POINTER(_Weights), i, i, i, ctypes.POINTER(_vp)]),
            "lstm_stack_create_ordered": (i, [ctypes.POINTER(_Weights), i, i, i, i,
                                              ctypes.POINTER(_vp)]),
            "lstm_stack_forward": (i, [_vp, _vp, sz, _vp, sz, i, i, _vp]),
            "lstm_stack_forward_host": (i, [_vp, _vp, sz, _vp, sz, i, i, _vp]),
            "lstm_stack_forward_host_async": (i, [_vp, _vp, sz, _vp, sz, i, i, _vp]),
            "lstm_stack_host_sync": (i, [_vp]),
            "lstm_stack_enable_phase_timing": (i, [_vp, i]),
            "lstm_stack_set_graphs": (i, [_vp, i]),
            "lstm_stack_set_math": (i, [_vp, i]),
            "lstm_stack_phase_times": (i, [_vp, _c_float_p]),
            "lstm_stack_destroy": (None, [_vp]),
            "lstm_stack_last_error": (ctypes.c_char_p, []),
            "lstm_pack_layer": (i, [_vp, _vp, _vp, i, i, _vp, _vp, _vp, _vp]),
            "lstm_pack_layer_ordered": (i, [_vp, _vp, _vp, i, i, i, _vp, _vp, _vp, _vp]),
            "lstm_projection": (i, [_vp, i, i, _vp, _vp, i, _vp, _vp]),
            "lstm_projection_math": (i, [_vp, i, i, _vp, _vp, i, _vp, i, _vp]),
            "lstm_recurrence": (i, [_vp, _vp, _vp, _vp, i, i, i, _vp]),
            "lstm_recurrence_variant": (i, [_vp, _vp, _vp, _vp, i, i, i, i, i, i, i, _vp]),
            "lstm_recurrence_max_clusters": (i, [i, i, i, i, i, ctypes.POINTER(i)]),
            "lstm_fault_status": (i, [ctypes.POINTER(ctypes.c_uint)]),
            "lstm_layer_forward_static": (i, [_vp, i, i, i, _vp, _vp, i, _vp, _vp, _vp, _vp]),
            "lstm_heads_create": (i, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, i, i,
                                      ctypes.POINTER(_vp)]),
            "lstm_heads_forward": (i, [_vp, _vp, sz, _vp, sz, i, _vp]),
            "lstm_heads_destroy": (None, [_vp]),
            "lstm_test_fail_allocations": (i, [i, i]),
            "lstm_test_fail_launches": (i, [i, i]),
            "lstm_test_recurrence_timeout": (i, [i, ctypes.c_uint, i]),
            "lstm_test_projection_timeout": (i, [i, ctypes.c_uint, i]),
            "lstm_test_heads_timeout": (i, [i, ctypes.c_uint, i]),
            "lstm_recurrence_floor": (i, [_vp, _vp, _vp, _vp, i, i, i, _vp]),
            "lstm_tf32_rate": (i, [i, i, ctypes.POINTER(ctypes.c_double)]),
            "lstm_recurrence_fused": (i, [_vp, i, _vp, _vp, i, _vp, _vp, _vp, i, i, i, _vp]),
            "lstm_stack_set_fused_batches": (i, [_vp, i]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def lstm_stack_last_error() -> str:
    return load().lstm_stack_last_error().decode()


def _check(code: int) -> None:
    if code != LSTM_OK:
        raise LSTMError(code, lstm_stack_last_error())


def _ptr(t) -> int:
    """Address of a torch tensor's data (None for None)."""
    return None if t is None else t.data_ptr()


def _stream(stream, device=None):
    if stream is None:
        import torch
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host(a, dtype=np.float32) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def lstm_pack_layer(w, r, b, in_width: int, kp: int, gate_order: int = LSTM_GATES_IFGO):
    """Host packer; returns (wp_hi, wp_lo, rp, bias) numpy arrays."""
    w, r, b = _host(w), _host(r), _host(b)
    wp_hi = np.empty((GATE_COLUMNS, kp), np.float32)
    wp_lo = np.empty((GATE_COLUMNS, kp), np.float32)
    rp = np.empty((2, 4 * HIDDEN, HIDDEN), np.float32)
    bias = np.empty((2, 4 * HIDDEN), np.float32)
    _check(load().lstm_pack_layer_ordered(w.ctypes.data, r.ctypes.data, b.ctypes.data, in_width,
                                          kp, gate_order, wp_hi.ctypes.data, wp_lo.ctypes.data,
                                          rp.ctypes.data, bias.ctypes.data))
    return wp_hi, wp_lo, rp, bias


def lstm_projection(x, rows: int, in_width: int, wp_hi, wp_lo, kp: int, g, stream=None):
    """G = X . Wp^T on the device (torch CUDA tensors)."""
    _check(load().lstm_projection(_ptr(x), rows, in_width, _ptr(wp_hi), _ptr(wp_lo), kp, _ptr(g),
                                  _stream(stream, x.device)))


def lstm_projection_math(x, rows: int, in_width: int, wp_hi, wp_lo, kp: int, g, math: int,
                         stream=None):
    """G = X . Wp^T with the chosen products (LSTM_MATH_*); wp_lo may be None
    for LSTM_MATH_TF32."""
    _check(load().lstm_projection_math(_ptr(x), rows, in_width, _ptr(wp_hi),
                                       _ptr(wp_lo), kp, _ptr(g), math,
                                       _stream(stream, x.device)))


def lstm_recurrence(g, rp, bias, y, batch: int, steps: int, direction: int, stream=None):
    _check(load().lstm_recurrence(_ptr(g), _ptr(rp), _ptr(bias), _ptr(y), batch, steps,
                                  direction, _stream(stream, g.device)))


def lstm_recurrence_floor(g, rp, bias, y, batch: int, steps: int, direction: int, stream=None):
    _check(load().lstm_recurrence_floor(_ptr(g), _ptr(rp), _ptr(bias), _ptr(y), batch, steps,
                                        direction, _stream(stream, g.device)))


def lstm_recurrence_fused(x, in_width: int, wp_hi, wp_lo, kp: int, rp, bias, y, batch: int,
                          steps: int, direction: int, stream=None):
    _check(load().lstm_recurrence_fused(_ptr(x), in_width, _ptr(wp_hi), _ptr(wp_lo), kp,
                                        _ptr(rp), _ptr(bias), _ptr(y), batch, steps, direction,
                                        _stream(stream, x.device)))


def lstm_stack_set_fused_batches(handle, max_batch: int) -> None:
    _check(load().lstm_stack_set_fused_batches(handle, max_batch))


def lstm_tf32_rate(device: int = 0, iterations: int = 20000) -> float:
    v = ctypes.c_double(0.0)
    _check(load().lstm_tf32_rate(device, iterations, ctypes.byref(v)))
    return float(v.value)


def lstm_recurrence_variant(g, rp, bias, y, batch: int, steps: int, direction: int,
                            cluster_size: int, windows_per_chunk: int, chunks: int = 1,
                            threads_per_block: int = 0, stream=None):
    _check(load().lstm_recurrence_variant(_ptr(g), _ptr(rp), _ptr(bias), _ptr(y), batch, steps,
                                          direction, cluster_size, windows_per_chunk, chunks,
                                          threads_per_block, _stream(stream, g.device)))


def lstm_recurrence_max_clusters(cluster_size: int, windows_per_chunk: int, chunks: int = 1,
                                 threads_per_block: int = 0, device: int = 0) -> int:
    v = ctypes.c_int(0)
    _check(load().lstm_recurrence_max_clusters(cluster_size, windows_per_chunk, chunks,
                                               threads_per_block, device, ctypes.byref(v)))
    return int(v.value)


def lstm_layer_forward_static(x, batch: int, steps: int, in_width: int, wp_hi, wp_lo, kp: int,
                              rp, bias, y, stream=None):
    """One bidirectional layer through the entry point that allocates no
    device memory (its gate buffer is a fixed array inside the library)."""
    _check(load().lstm_layer_forward_static(_ptr(x), batch, steps, in_width, _ptr(wp_hi),
                                            _ptr(wp_lo), kp, _ptr(rp), _ptr(bias), _ptr(y),
                                            _stream(stream, x.device)))


def lstm_fault_status() -> int:
    v = ctypes.c_uint(0)
    _check(load().lstm_fault_status(ctypes.byref(v)))
    return int(v.value)


def lstm_stack_create(layers, max_batch: int, max_steps: int, device: int = 0,
                      gate_order: int = LSTM_GATES_IFGO):
    """Creates a stack from source weights (list of dicts w, r, b; numpy) whose
    gate row blocks are in ``gate_order`` (LSTM_GATES_IFGO or _IOFC).

    Returns the opaque handle (an int).  The host arrays are only read during
    the call.
    """
    arrs = [{k: _host(l[k]) for k in ("w", "r", "b")} for l in layers]
    ws = _Weights()
    for l, a in enumerate(arrs):
        ws.w[l] = a["w"].ctypes.data
        ws.r[l] = a["r"].ctypes.data
        ws.b[l] = a["b"].ctypes.data
    h = _vp()
    _check(load().lstm_stack_create_ordered(ctypes.byref(ws), gate_order, max_batch, max_steps,
                                            device, ctypes.byref(h)))
    return h.value


def lstm_stack_forward(handle, x, y, batch: int, steps: int, stream=None):
    _check(load().lstm_stack_forward(handle, _ptr(x), x.numel(), _ptr(y), y.numel(), batch,
                                     steps, _stream(stream, x.device)))


def lstm_stack_forward_host(handle, x: np.ndarray, y: np.ndarray, batch: int, steps: int,
                            stream=None):
    """x, y: C-contiguous float32 host arrays (pinned memory recommended)."""
    assert x.dtype == np.float32 and y.dtype == np.float32
    assert x.flags.c_contiguous and y.flags.c_contiguous
    _check(load().lstm_stack_forward_host(handle, x.ctypes.data, x.size, y.ctypes.data, y.size,
                                          batch, steps, _stream(stream)))


def lstm_stack_forward_host_async(handle, x: np.ndarray, y: np.ndarray, batch: int, steps: int,
                                  stream=None):
    """Enqueue without waiting; x must stay unchanged and y is valid only after
    lstm_stack_host_sync.  x, y: C-contiguous float32 host arrays, pinned for
    the copies to overlap the forward."""
    assert x.dtype == np.float32 and y.dtype == np.float32
    assert x.flags.c_contiguous and y.flags.c_contiguous
    _check(load().lstm_stack_forward_host_async(handle, x.ctypes.data, x.size, y.ctypes.data,
                                                y.size, batch, steps, _stream(stream)))


def lstm_stack_host_sync(handle):
    _check(load().lstm_stack_host_sync(handle))


def lstm_stack_set_graphs(handle, enable: bool = True):
    _check(load().lstm_stack_set_graphs(handle, int(bool(enable))))


def lstm_stack_set_math(handle, math: int):
    _check(load().lstm_stack_set_math(handle, math))


def lstm_stack_enable_phase_timing(handle, enable: bool = True):
    _check(load().lstm_stack_enable_phase_timing(handle, int(bool(enable))))


def lstm_stack_phase_times(handle) -> np.ndarray:
    ms = (ctypes.c_float * (3 * LAYERS))()
    _check(load().lstm_stack_phase_times(handle, ms))
    return np.array(ms[:], dtype=np.float64).reshape(LAYERS, 3)


def lstm_stack_destroy(handle) -> None:
    if handle:
        load().lstm_stack_destroy(handle)


class LSTMStack:
    """Owns a stack handle; ``forward`` takes and returns torch CUDA tensors."""

    def __init__(self, layers, max_batch: int, max_steps: int, device: int = 0,
                 gate_order: int = LSTM_GATES_IFGO):
        self.device = device
        self.max_batch = max_batch
        self.max_steps = max_steps
        self.handle = lstm_stack_create(layers, max_batch, max_steps, device, gate_order)

    def forward(self, x, y=None, stream=None):
        """x: [B, T, 60] float32 CUDA tensor -> y [B, T, 256] (new unless given)."""
        import torch
        B, T, F = x.shape
        if F != FEATURES:
            raise ValueError(f"input width {F}, expected {FEATURES}")
        if y is None:
            y = torch.empty((B, T, OUTPUT), dtype=torch.float32, device=x.device)
        lstm_stack_forward(self.handle, x, y, B, T, stream)
        return y

    __call__ = forward

    def close(self):
        if self.handle:
            lstm_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


HEADS_CLASSES = 7


class LSTMHeads:
    """The segmentation model's dense heads (linear0, linear1, classifier) on
    stack output rows; ``forward`` takes and returns torch CUDA tensors."""

    def __init__(self, weights, max_rows: int, negative_slope: float = 0.01, device: int = 0):
        arrs = {k: _host(weights[k]) for k in ("w0", "b0", "w1", "b1", "w2", "b2")}
        h = _vp()
        _check(load().lstm_heads_create(*(arrs[k].ctypes.data for k in
                                          ("w0", "b0", "w1", "b1", "w2", "b2")),
                                        float(negative_slope), max_rows, device, ctypes.byref(h)))
        self.handle = h.value
        self.max_rows = max_rows
        self.device = device

    def forward(self, y, out=None, stream=None):
        """y: [..., 256] float32 CUDA tensor -> log-probabilities [..., 7]."""
        import torch
        if y.shape[-1] != OUTPUT:
            raise ValueError(f"input width {y.shape[-1]}, expected {OUTPUT}")
        rows = y.numel() // OUTPUT
        if out is None:
            out = torch.empty((*y.shape[:-1], HEADS_CLASSES), dtype=torch.float32,
                              device=y.device)
        _check(load().lstm_heads_forward(self.handle, _ptr(y), y.numel(), _ptr(out), out.numel(),
                                         rows, _stream(stream, y.device)))
        return out

    __call__ = forward

    def close(self):
        if self.handle:
            load().lstm_heads_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass
