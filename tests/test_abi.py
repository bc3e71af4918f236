"""The C ABI without a GPU: the library builds and loads, exports every
symbol include/lstm_stack.h declares, rejects bad arguments before touching
CUDA, and its host-side packer lays the weights out as documented."""
import ctypes
import os
import re

import numpy as np
import pytest

from bidirectional_lstm_stack_gb300 import binding, synthetic
from bidirectional_lstm_stack_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lstm_stack.h")
H = synthetic.HIDDEN


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lstm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_stack_api():
    names = _declared_functions()
    for must in ["lstm_stack_create", "lstm_stack_forward", "lstm_stack_destroy",
                 "lstm_stack_last_error", "lstm_pack_layer", "lstm_projection",
                 "lstm_recurrence"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_forward_rejects_null_stack(lib):
    assert lib.lstm_stack_forward(None, None, 0, None, 0, 1, 1, None) == binding.LSTM_E_INVALID
    assert "null" in binding.lstm_stack_last_error()


def test_host_entry_points_reject_null_stack(lib):
    for fn in (lib.lstm_stack_forward_host, lib.lstm_stack_forward_host_async):
        assert fn(None, None, 0, None, 0, 1, 1, None) == binding.LSTM_E_INVALID
        assert "null" in binding.lstm_stack_last_error()
    assert lib.lstm_stack_host_sync(None) == binding.LSTM_E_INVALID


def test_create_rejects_null_weights(lib):
    h = ctypes.c_void_p()
    assert lib.lstm_stack_create(None, 1, 1, 0, ctypes.byref(h)) == binding.LSTM_E_INVALID
    assert h.value is None


def test_create_rejects_bad_sizes(lib):
    layers = synthetic.stack_weights()
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_stack_create(layers, 0, 10)
    assert e.value.code == binding.LSTM_E_INVALID
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_stack_create(layers, 100000, 100000)
    assert e.value.code == binding.LSTM_E_OVERFLOW


def test_step_entry_points_reject_bad_arguments(lib):
    assert lib.lstm_projection(None, 1, 60, None, None, 64, None, None) == binding.LSTM_E_INVALID
    assert lib.lstm_recurrence(None, None, None, None, 1, 1, 0, None) == binding.LSTM_E_INVALID
    assert lib.lstm_fault_status(None) == binding.LSTM_E_INVALID


def test_recurrence_rejects_unaligned_buffers(lib):
    # checked on the host before any device call: g and y (h goes out four
    # units at a time) must be 16-byte aligned, like rp
    assert lib.lstm_recurrence(4, 16, 16, 16, 1, 1, 0, None) == binding.LSTM_E_INVALID
    assert "g (" in binding.lstm_stack_last_error()
    assert lib.lstm_recurrence(16, 16, 16, 20, 1, 1, 0, None) == binding.LSTM_E_INVALID
    assert "y (" in binding.lstm_stack_last_error()


def test_destroy_null_is_a_noop(lib):
    lib.lstm_stack_destroy(None)


def _tf32_exact(a):
    bits = np.asarray(a, np.float32).view(np.uint32)
    return np.all((bits & 0x1FFF) == 0)


@pytest.mark.parametrize("in_width,kp", [(60, 64), (256, 256)])
def test_packer_layout(lib, in_width, kp):
    rng = np.random.default_rng(3)
    w = rng.uniform(-1, 1, (2, 4 * H, in_width)).astype(np.float32)
    r = rng.uniform(-1, 1, (2, 4 * H, H)).astype(np.float32)
    b = rng.uniform(-1, 1, (2, 8 * H)).astype(np.float32)
    wp_hi, wp_lo, rp, bias = binding.lstm_pack_layer(w, r, b, in_width, kp)
    assert _tf32_exact(wp_hi) and _tf32_exact(wp_lo)
    for d in range(2):
        for u in (0, 1, 77, H - 1):
            for k in range(4):
                src = k * H + u
                dst = 4 * u + k
                n = d * 4 * H + dst
                full = wp_hi[n].astype(np.float64) + wp_lo[n]
                np.testing.assert_allclose(full[:in_width], w[d, src], rtol=2e-7, atol=1e-12)
                assert np.all(wp_hi[n, in_width:] == 0) and np.all(wp_lo[n, in_width:] == 0)
                np.testing.assert_array_equal(rp[d, dst], r[d, src])
                assert bias[d, dst] == np.float32(b[d, src] + b[d, 4 * H + src])


def test_packer_hi_is_nearest_tf32(lib):
    # hi is w rounded to 10 mantissa bits (nearest, ties away from zero)
    w = np.zeros((2, 4 * H, 32), np.float32)
    vals = np.array([1.0 + 2.0 ** -11, 1.0 + 2.0 ** -12, -(1.0 + 2.0 ** -11),
                     1.0 + 3 * 2.0 ** -12, 3.0e-39], np.float32)
    w[0, 0, :len(vals)] = vals
    z = np.zeros((2, 4 * H, H), np.float32)
    bb = np.zeros((2, 8 * H), np.float32)
    wp_hi, wp_lo, _, _ = binding.lstm_pack_layer(w, z, bb, 32, 32)
    got = wp_hi[0, :len(vals)]
    expect = np.array([1.0 + 2.0 ** -10, 1.0, -(1.0 + 2.0 ** -10), 1.0 + 2.0 ** -10,
                       got[4]], np.float32)
    np.testing.assert_array_equal(got, expect)
    np.testing.assert_allclose(wp_hi[0, :4].astype(np.float64) + wp_lo[0, :4], vals[:4],
                               rtol=0, atol=0)


def test_packer_rejects_bad_kp(lib):
    w = np.zeros((2, 4 * H, 60), np.float32)
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_pack_layer(w, np.zeros((2, 4 * H, H)), np.zeros((2, 8 * H)), 60, 60)
    assert e.value.code == binding.LSTM_E_INVALID


def _to_iofc(a, H, axis):
    """Reorders i, f, g, o row blocks (length H each) into ONNX's i, o, f, c."""
    i, f, g, o = np.split(a, 4, axis=axis)
    return np.concatenate([i, o, f, g], axis=axis)


def test_packer_onnx_gate_order_matches_default(lib):
    rng = np.random.default_rng(5)
    w = rng.uniform(-1, 1, (2, 4 * H, 60)).astype(np.float32)
    r = rng.uniform(-1, 1, (2, 4 * H, H)).astype(np.float32)
    b = rng.uniform(-1, 1, (2, 8 * H)).astype(np.float32)
    b_onnx = np.concatenate([_to_iofc(b[:, :4 * H], H, 1), _to_iofc(b[:, 4 * H:], H, 1)], axis=1)
    ref = binding.lstm_pack_layer(w, r, b, 60, 64)
    got = binding.lstm_pack_layer(_to_iofc(w, H, 1), _to_iofc(r, H, 1), b_onnx, 60, 64,
                                  binding.LSTM_GATES_IOFC)
    for a, c in zip(ref, got):
        np.testing.assert_array_equal(a, c)
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_pack_layer(w, r, b, 60, 64, 2)
    assert e.value.code == binding.LSTM_E_INVALID


def test_heads_create_rejects_null_weights(lib):
    import ctypes
    out = ctypes.c_void_p()
    w = np.zeros(256 * 128, np.float32)
    ptrs = [w.ctypes.data] * 5 + [None]
    assert lib.lstm_heads_create(*ptrs, 0.01, 10, 0, ctypes.byref(out)) == binding.LSTM_E_INVALID
    assert not out.value
    assert lib.lstm_heads_create(*([w.ctypes.data] * 6), 0.01, 0, 0,
                                 ctypes.byref(out)) == binding.LSTM_E_INVALID
    lib.lstm_heads_destroy(None)


def test_measurement_entry_points_reject_bad_arguments(lib):
    import ctypes
    v = ctypes.c_double(0.0)
    assert lib.lstm_tf32_rate(0, 0, ctypes.byref(v)) == 1  # iterations outside 1..10^7
    assert lib.lstm_tf32_rate(0, 100, None) == 1
    assert lib.lstm_recurrence_floor(None, None, None, None, 1, 1, 0, None) == 1


def test_timeout_hooks_reject_limits_above_two_seconds(lib):
    for hook in (lib.lstm_test_recurrence_timeout, lib.lstm_test_projection_timeout,
                 lib.lstm_test_heads_timeout):
        assert hook(1, 2000001, 0) == 1
