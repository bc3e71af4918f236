"""Float64 CPU oracle of the four-layer bidirectional LSTM stack.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never loads it, and it imports nothing from the
product package: it shares no code, header, table or constant with the CUDA
path.  Inputs reach it as plain numpy arrays.

It wraps ``lstm_oracle.c`` (plain C, float64, libm) through ctypes.  Every
function follows the definition of the method on the speakrs 0.6.0 pages
(``lstmproj.rs``: module docs, ``PackedLayer``, ``Oxide::with_recurrence``,
``recur``); the C file's header lists the passages and the readings taken where
the pages are silent.

Pins (the checks that tie the oracle to something other than itself) live in
``tests/test_oracle_pins.py``: zero weights, the R = 0 closed form, reverse
equals forward on time-reversed input, brute force on H = 2, T = 3 (every gate
written out as scalar arithmetic), a saturated-gate counter whose outputs
are tanh of integers (``tests/golden/saturated_counter.json``), a one-hot
projection, and agreement with ``torch.nn.LSTM`` in float64; for the TF32
projection mode, the rounding against a bit-level definition and the TF32
stack against the float64 stack on pre-rounded operands.  No oracle function
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lstm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblstm_oracle.so")
_lock = threading.Lock()
_lib = None

_dptr = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``lstm_oracle.c`` into ``liblstm_oracle.so`` beside it."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_lstm_direction.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _dptr, ctypes.c_long, _dptr, _dptr, _dptr, _dptr,
                ctypes.c_int, _dptr, ctypes.c_long]
            for f in (lib.oracle_lstm_stack, lib.oracle_lstm_stack_tf32):
                f.argtypes = [
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                    ctypes.c_int, _dptr, ctypes.POINTER(_dptr),
                    ctypes.POINTER(_dptr), ctypes.POINTER(_dptr), _dptr]
            for f in (lib.oracle_projection, lib.oracle_projection_tf32):
                f.argtypes = [
                    ctypes.c_long, ctypes.c_int, ctypes.c_int, _dptr, _dptr, _dptr]
            lib.oracle_tf32_array.argtypes = [ctypes.c_long, _dptr, _dptr]
            lib.oracle_heads.argtypes = [
                ctypes.c_long, _dptr, _dptr, _dptr, _dptr, _dptr, _dptr, _dptr,
                ctypes.c_double, _dptr]
            lib.oracle_recurrence.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, _dptr, _dptr, _dptr,
                _dptr]
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dptr)


def threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_threads())


def lstm_direction(x, W, R, Wb, Rb, reverse: bool) -> np.ndarray:
    """One direction of one layer over one window.

    x ``[T, in]``, W ``[4H, in]``, R ``[4H, H]``, Wb/Rb ``[4H]`` (gate row
    blocks i, f, g, o).  Returns h ``[T, H]``; the reverse direction visits
    t = T-1 .. 0 and still writes row t.
    """
    x, W, R, Wb, Rb = map(_f64, (x, W, R, Wb, Rb))
    T, inw = x.shape
    H = R.shape[1]
    assert W.shape == (4 * H, inw) and R.shape == (4 * H, H)
    assert Wb.shape == (4 * H,) and Rb.shape == (4 * H,)
    h = np.zeros((T, H), dtype=np.float64)
    _load().oracle_lstm_direction(T, inw, H, _p(x), inw, _p(W), _p(R),
                                  _p(Wb), _p(Rb), int(bool(reverse)), _p(h), H)
    return h


def tf32(v) -> np.ndarray:
    """``v`` rounded to TF32 (10 stored mantissa bits, to nearest, ties away
    from zero), as float64."""
    v = _f64(v)
    out = np.empty_like(v)
    _load().oracle_tf32_array(v.size, _p(v), _p(out))
    return out


def lstm_stack(x, layers, projection: str = "f64") -> np.ndarray:
    """The bidirectional stack.

    x ``[B, T, in0]``; ``layers`` is a sequence of dicts with ``w``
    ``[2, 4H, in_l]``, ``r`` ``[2, 4H, H]`` and ``b`` ``[2, 8H]`` (per
    direction Wb then Rb).  Returns y ``[B, T, 2H]`` =
    concat(forward h, reverse h) of the last layer.  ``projection="tf32"``
    rounds both factors of every input-projection product to TF32 (the
    method's TF32 projection mode); everything else stays float64.
    """
    assert projection in ("f64", "tf32"), projection
    x = _f64(x)
    B, T, in0 = x.shape
    L = len(layers)
    ws = [_f64(l["w"]) for l in layers]
    rs = [_f64(l["r"]) for l in layers]
    bs = [_f64(l["b"]) for l in layers]
    H = rs[0].shape[2]
    for i, (w, r, b) in enumerate(zip(ws, rs, bs)):
        inw = in0 if i == 0 else 2 * H
        assert w.shape == (2, 4 * H, inw), (i, w.shape)
        assert r.shape == (2, 4 * H, H), (i, r.shape)
        assert b.shape == (2, 8 * H), (i, b.shape)
    y = np.zeros((B, T, 2 * H), dtype=np.float64)
    arr = _dptr * L
    fn = _load().oracle_lstm_stack if projection == "f64" else _load().oracle_lstm_stack_tf32
    fn(B, T, in0, H, L, _p(x), arr(*[_p(w) for w in ws]), arr(*[_p(r) for r in rs]),
       arr(*[_p(b) for b in bs]), _p(y))
    return y


def projection(X, W, tf32: bool = False) -> np.ndarray:
    """Packed-column input projection of one layer, both directions.

    X ``[M, in]``, W ``[2, 4H, in]``.  Returns G ``[M, 8H]`` with
    ``G[m, d*4H + 4u + k] = sum_j X[m, j] * W[d, k*H + u, j]`` (no bias);
    with ``tf32`` both factors of each product are rounded to TF32 first.
    """
    X, W = _f64(X), _f64(W)
    M, inw = X.shape
    H = W.shape[1] // 4
    assert W.shape == (2, 4 * H, inw)
    G = np.zeros((M, 8 * H), dtype=np.float64)
    fn = _load().oracle_projection_tf32 if tf32 else _load().oracle_projection
    fn(M, inw, H, _p(X), _p(W), _p(G))
    return G


def recurrence(G, R, bias, batch: int, steps: int) -> np.ndarray:
    """One layer's recurrence for both directions from a packed projection.

    G ``[B*T, 8H]`` (packed columns, no bias), R ``[2, 4H, H]``, bias
    ``[2, 8H]`` (Wb then Rb).  Returns y ``[B, T, 2H]``.
    """
    G, R, bias = _f64(G), _f64(R), _f64(bias)
    H = R.shape[2]
    assert G.shape == (batch * steps, 8 * H)
    assert R.shape == (2, 4 * H, H) and bias.shape == (2, 8 * H)
    y = np.zeros((batch, steps, 2 * H), dtype=np.float64)
    _load().oracle_recurrence(batch, steps, H, _p(G), _p(R), _p(bias), _p(y))
    return y


def heads(y, W0, b0, W1, b1, W2, b2, slope: float = 0.01) -> np.ndarray:
    """The segmentation model's dense heads on stack output rows.

    y ``[M, 256]``; W0 ``[256, 128]``, W1 ``[128, 128]``, W2 ``[128, 7]``
    (row-major ``[k, n]``, as the pages store them), biases ``[n]``.  Returns
    the log-probabilities ``[M, 7]`` of
    ``log_softmax(leaky(leaky(y W0 + b0) W1 + b1) W2 + b2)``.
    """
    y, W0, b0, W1, b1, W2, b2 = map(_f64, (y, W0, b0, W1, b1, W2, b2))
    M = y.shape[0]
    assert y.shape == (M, 256) and W0.shape == (256, 128) and b0.shape == (128,)
    assert W1.shape == (128, 128) and b1.shape == (128,)
    assert W2.shape == (128, 7) and b2.shape == (7,)
    out = np.zeros((M, 7), dtype=np.float64)
    _load().oracle_heads(M, _p(y), _p(W0), _p(b0), _p(W1), _p(b1), _p(W2), _p(b2),
                         float(slope), _p(out))
    return out
