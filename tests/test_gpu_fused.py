"""The recurrence with the input projection fused in (small batches), through
the C ABI: one layer against the float64 oracle's layer for both input
widths, ragged steps and several windows; the two directions launched apart
against the one launch (bitwise); the whole stack in fused mode against the
oracle; a timed-out wait reported and recovered from."""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layers():
    return synthetic.stack_weights()


def _packed(lay, in_width):
    kp = 64 if in_width == 60 else 256
    wp_hi, wp_lo, rp, bias = binding.lstm_pack_layer(lay["w"], lay["r"], lay["b"], in_width, kp)
    return kp, cuda(wp_hi), cuda(wp_lo), cuda(rp), cuda(bias)


def _fused_layer(lay, x, direction=binding.LSTM_BOTH_DIRECTIONS):
    import torch
    batch, steps, in_width = x.shape
    kp, whi, wlo, rp, bias = _packed(lay, in_width)
    y = torch.full((batch, steps, 256), float("nan"), device="cuda")
    if direction == binding.LSTM_BOTH_DIRECTIONS:
        binding.lstm_recurrence_fused(cuda(x), in_width, whi, wlo, kp, rp, bias, y, batch, steps,
                                      direction)
    else:
        for d in (0, 1):
            binding.lstm_recurrence_fused(cuda(x), in_width, whi, wlo, kp, rp[d], bias[d], y,
                                          batch, steps, d)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("layer_index", [0, 1])
@pytest.mark.parametrize("batch,steps", [(1, 1), (1, 2), (1, 37), (2, 64), (5, 100), (6, 33)])
def test_fused_layer_matches_oracle(layers, layer_index, batch, steps):
    lay = layers[layer_index]
    in_width = lay["w"].shape[2]
    x = synthetic.random_matrix(batch * 100 + steps + layer_index, (batch, steps, in_width))
    y = _fused_layer(lay, x)
    assert_within(y, oracle.lstm_stack(x, [lay]), what=f"fused layer {layer_index} b{batch} t{steps}")
    assert binding.lstm_fault_status() == 0


def test_fused_directions_apart_equal_one_launch(layers):
    lay = layers[1]
    x = synthetic.random_matrix(77, (3, 45, 256))
    both = _fused_layer(lay, x)
    apart = _fused_layer(lay, x, direction=0)
    assert np.array_equal(both.view(np.uint32), apart.view(np.uint32))


@pytest.mark.parametrize("name", ["b1_t64", "b1_t589", "b8_t589_x3"])
def test_fused_stack_matches_oracle(layers, name):
    import torch
    wl = synthetic.WORKLOADS[name]
    x = synthetic.stack_input(wl)
    s = binding.LSTMStack(layers, wl.batch, wl.steps)
    try:
        binding.lstm_stack_set_fused_batches(s.handle, 8)
        y = s(cuda(x))
        torch.cuda.synchronize()
        assert_within(y.cpu().numpy(), oracle.lstm_stack(x, layers), what=f"fused stack {name}")
        assert binding.lstm_fault_status() == 0
    finally:
        s.close()


def test_fused_stack_timeout_is_reported_and_recovered(layers):
    lib = binding.load()
    x = synthetic.stack_input(synthetic.WORKLOADS["b1_t64"])
    s = binding.LSTMStack(layers, 1, 64)
    try:
        binding.lstm_stack_set_fused_batches(s.handle, 1)
        y = np.empty((1, 64, 256), np.float32)
        lib.lstm_test_recurrence_timeout(1, 20000, 0)  # CTA 0 of every cluster pushes nothing
        try:
            with pytest.raises(binding.LSTMError) as e:
                binding.lstm_stack_forward_host(s.handle, x, y, 1, 64)
            assert e.value.code == binding.LSTM_E_FAULT
        finally:
            lib.lstm_test_recurrence_timeout(0, 0, 0)
        binding.lstm_stack_forward_host(s.handle, x, y, 1, 64)
        assert_within(y, oracle.lstm_stack(x, layers), what="fused stack after timeout")
    finally:
        s.close()
        binding.lstm_fault_status()


def test_fused_setting_above_the_device_falls_back(layers):
    # a batch whose fused clusters would not all run at once takes the
    # projection kernel and the recurrence instead, with the same result bound
    import torch
    batch, steps = 40, 20
    x = synthetic.random_matrix(5, (batch, steps, 60))
    s = binding.LSTMStack(layers, batch, steps)
    try:
        binding.lstm_stack_set_fused_batches(s.handle, 100000)
        y = s(cuda(x))
        torch.cuda.synchronize()
        assert_within(y.cpu().numpy(), oracle.lstm_stack(x, layers), what="fused fallback")
        with pytest.raises(binding.LSTMError) as e:
            binding.lstm_stack_set_fused_batches(s.handle, -1)
        assert e.value.code == binding.LSTM_E_INVALID
    finally:
        s.close()
