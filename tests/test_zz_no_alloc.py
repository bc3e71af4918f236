"""The layer entry point that allocates no device memory.

Callers that cannot call cudaMalloc (graph capture, frameworks that own all
device memory, allocation-free hot loops) use lstm_layer_forward_static,
whose gate buffer is a fixed array inside the library.  Its output must match
the allocating step entry points (lstm_projection + lstm_recurrence with a
caller-owned gate buffer) on two calls in a row that share that array: within
the stack's tolerance, and in fact bit for bit, since both run the same
kernels on the same inputs.  Both are also checked against the float64
oracle's layer.  This file is collected last so that a failure here leaves
every other test run.
"""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu


def _reference_layer(x, lay, in_width, kp, batch, steps):
    import torch
    wp_hi, wp_lo, rp, bias = binding.lstm_pack_layer(lay["w"], lay["r"], lay["b"], in_width, kp)
    d = {k: cuda(v) for k, v in (("wp_hi", wp_hi), ("wp_lo", wp_lo), ("rp", rp), ("bias", bias))}
    rows = batch * steps
    g = torch.empty((rows, 1024), device="cuda")
    binding.lstm_projection(x, rows, in_width, d["wp_hi"], d["wp_lo"], kp, g)
    y = torch.full((batch, steps, 256), float("nan"), device="cuda")
    for k in range(2):
        binding.lstm_recurrence(g, d["rp"][k], d["bias"][k], y, batch, steps, k)
    torch.cuda.synchronize()
    return d, y.cpu().numpy()


def test_static_layer_matches_allocating_entry_points_twice():
    import torch
    layers = synthetic.stack_weights()
    # two calls in a row sharing the static buffer: a 60-wide first layer,
    # then a 256-wide later layer of another shape
    cases = [(layers[0], 60, 64, 3, 100, 31), (layers[1], 256, 256, 5, 61, 32)]
    for lay, in_width, kp, batch, steps, seed in cases:
        x = cuda(synthetic.random_matrix(seed, (batch, steps, in_width)))
        d, ref = _reference_layer(x, lay, in_width, kp, batch, steps)
        y = torch.full((batch, steps, 256), float("nan"), device="cuda")
        binding.lstm_layer_forward_static(x, batch, steps, in_width, d["wp_hi"], d["wp_lo"], kp,
                                          d["rp"], d["bias"], y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        what = f"static layer b{batch} t{steps} k{in_width}"
        assert_within(got, ref, what=what)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), what
        x64 = x.cpu().numpy().astype(np.float64)
        assert_within(got, oracle.lstm_stack(x64, [lay]), what=what + " vs oracle")
    assert binding.lstm_fault_status() == 0


def test_static_layer_rejects_rows_beyond_its_buffer():
    import torch
    x = torch.zeros((2, 2049, 60), device="cuda")
    z = torch.zeros(16, device="cuda")
    y = torch.zeros((2, 2049, 256), device="cuda")
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_layer_forward_static(x, 2, 2049, 60, z, z, 64, z, z, y)
    assert e.value.code == binding.LSTM_E_INVALID
    assert "exceed" in str(e.value)
