"""Failure detection without a GPU fault: injected allocation and launch
failures on the host, and bounded waits made to run out on the GPU (the
recurrence: CTA 0 of every cluster withholds its hidden state, so its peers'
waits expire; the projection and the dense heads: the TMA producer loads
nothing, so the waits of the warps that consume its stages expire).  In every
case the call reports the failure and the next call on the same objects works
again."""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu

FAULT_RECURRENCE = 1 << 5
# the roles of the projection and heads kernels whose waits can run out:
# producer, converters, MMA issuer, epilogue (not the drain at teardown)
FAULT_TILED_ROLES = (1 << 0) | (1 << 1) | (1 << 2) | (1 << 3)


@pytest.fixture(scope="module")
def layers():
    return synthetic.stack_weights()


@pytest.fixture(autouse=True)
def _clean():
    lib = binding.load()
    yield
    lib.lstm_test_fail_allocations(0, 0)
    lib.lstm_test_fail_launches(0, 0)
    lib.lstm_test_recurrence_timeout(0, 0, 0)
    lib.lstm_test_projection_timeout(0, 0, 0)
    lib.lstm_test_heads_timeout(0, 0, 0)
    binding.lstm_fault_status()


def _free():
    import torch
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def test_allocation_failures_are_reported_and_leak_nothing(layers):
    lib = binding.load()
    s = binding.LSTMStack(layers, 4, 64)  # warm the context, then measure
    s.close()
    free0 = _free()
    for skip in range(6):  # the stack makes six device allocations
        lib.lstm_test_fail_allocations(skip, 1)
        with pytest.raises(binding.LSTMError) as e:
            binding.LSTMStack(layers, 4, 64)
        assert e.value.code == binding.LSTM_E_ALLOC
    lib.lstm_test_fail_allocations(0, 0)
    assert abs(_free() - free0) < (4 << 20)
    lib.lstm_test_fail_allocations(0, 1)  # the heads' one device allocation
    with pytest.raises(binding.LSTMError) as e:
        binding.LSTMHeads(synthetic.heads_weights(), 100)
    assert e.value.code == binding.LSTM_E_ALLOC
    lib.lstm_test_fail_allocations(0, 0)
    s = binding.LSTMStack(layers, 4, 64)
    s.close()


@pytest.mark.parametrize("graphs", [False, True])
def test_launch_failure_mid_forward_then_recovery(layers, graphs):
    import torch
    lib = binding.load()
    x_np = synthetic.stack_input(synthetic.WORKLOADS["b1_t64"])
    x = cuda(x_np)
    s = binding.LSTMStack(layers, 1, 64)
    try:
        binding.lstm_stack_set_graphs(s.handle, graphs)
        for skip in (0, 3, 7):  # the first, a middle and the last of the 8 launches of a pass
            lib.lstm_test_fail_launches(skip, 1)
            with pytest.raises(binding.LSTMError) as e:
                s(x)
            assert e.value.code == binding.LSTM_E_CUDA
            assert "injected" in binding.lstm_stack_last_error()
            torch.cuda.synchronize()
        lib.lstm_test_fail_launches(0, 0)
        y = s(x)
        torch.cuda.synchronize()
        assert_within(y.cpu().numpy(), oracle.lstm_stack(x_np, layers), what="after failures")
    finally:
        s.close()


def test_recurrence_wait_timeout_sets_fault_and_recovers(layers):
    import torch
    lib = binding.load()
    rng = np.random.default_rng(9)
    wp_hi, wp_lo, rp, bias = binding.lstm_pack_layer(layers[1]["w"], layers[1]["r"],
                                                     layers[1]["b"], 256, 256)
    steps = 40
    g = cuda(rng.standard_normal((steps, 1024)).astype(np.float32))
    y = torch.zeros((1, steps, 256), device="cuda")
    assert binding.lstm_fault_status() == 0
    lib.lstm_test_recurrence_timeout(1, 20000, 0)  # withhold, 20 ms per wait
    binding.lstm_recurrence(g, cuda(rp[0]), cuda(bias[0]), y, 1, steps, 0)
    torch.cuda.synchronize()
    assert binding.lstm_fault_status() == FAULT_RECURRENCE
    assert binding.lstm_fault_status() == 0  # read and cleared
    lib.lstm_test_recurrence_timeout(0, 0, 0)
    binding.lstm_recurrence(g, cuda(rp[0]), cuda(bias[0]), y, 1, steps, 0)
    torch.cuda.synchronize()
    assert binding.lstm_fault_status() == 0
    ref = oracle.recurrence(g.cpu().numpy().astype(np.float64), layers[1]["r"], layers[1]["b"],
                            1, steps)
    assert_within(y.cpu().numpy()[..., :128], ref[..., :128], what="recurrence after timeout")


def test_tensor_core_recurrence_wait_timeout_sets_fault_and_recovers(layers):
    # CTA 0 of every cluster withholds its h slices; the peers' bounded waits
    # run out, the kernel frees its tensor memory and ends, and the next
    # launch is correct
    import torch
    lib = binding.load()
    rng = np.random.default_rng(10)
    _, _, rp, bias = binding.lstm_pack_layer(layers[1]["w"], layers[1]["r"], layers[1]["b"],
                                             256, 256)
    batch, steps = 20, 24
    g = cuda(rng.standard_normal((batch * steps, 1024)).astype(np.float32))
    y = torch.zeros((batch, steps, 256), device="cuda")
    rpt, bt = cuda(rp), cuda(bias)
    assert binding.lstm_fault_status() == 0
    lib.lstm_test_recurrence_timeout(1, 20000, 0)
    try:
        binding.lstm_recurrence_variant(g, rpt, bt, y, batch, steps,
                                        binding.LSTM_BOTH_DIRECTIONS, 4, 16, 1, 128)
        torch.cuda.synchronize()
        assert binding.lstm_fault_status() == FAULT_RECURRENCE
    finally:
        lib.lstm_test_recurrence_timeout(0, 0, 0)
    binding.lstm_recurrence_variant(g, rpt, bt, y, batch, steps, binding.LSTM_BOTH_DIRECTIONS,
                                    4, 16, 1, 128)
    torch.cuda.synchronize()
    assert binding.lstm_fault_status() == 0
    ref = oracle.recurrence(g.cpu().numpy().astype(np.float64), layers[1]["r"], layers[1]["b"],
                            batch, steps)
    assert_within(y.cpu().numpy(), ref, what="tensor-core recurrence after timeout")


def test_forward_host_reports_a_timed_out_wait(layers):
    lib = binding.load()
    x = synthetic.stack_input(synthetic.WORKLOADS["b1_t64"])
    s = binding.LSTMStack(layers, 1, 64)
    try:
        y = np.empty((1, 64, 256), np.float32)
        lib.lstm_test_recurrence_timeout(1, 20000, 0)
        with pytest.raises(binding.LSTMError) as e:
            binding.lstm_stack_forward_host(s.handle, x, y, 1, 64)
        assert e.value.code == binding.LSTM_E_FAULT
        lib.lstm_test_recurrence_timeout(0, 0, 0)
        binding.lstm_stack_forward_host(s.handle, x, y, 1, 64)
        assert_within(y, oracle.lstm_stack(x, layers), what="forward_host after timeout")
    finally:
        s.close()


def test_projection_wait_timeout_sets_fault_and_recovers(layers):
    import torch
    lib = binding.load()
    rows = 700  # several 128-row tiles and a ragged tail
    x_np = synthetic.random_matrix(21, (rows, 256))
    x = cuda(x_np)
    wp_hi, wp_lo, _, _ = binding.lstm_pack_layer(layers[1]["w"], layers[1]["r"], layers[1]["b"],
                                                 256, 256)
    whi, wlo = cuda(wp_hi), cuda(wp_lo)
    g = torch.zeros((rows, 1024), device="cuda")
    assert binding.lstm_fault_status() == 0
    lib.lstm_test_projection_timeout(1, 20000, 0)  # producer loads nothing, 20 ms per wait
    binding.lstm_projection(x, rows, 256, whi, wlo, 256, g)
    torch.cuda.synchronize()
    bits = binding.lstm_fault_status()
    assert bits != 0 and (bits & ~FAULT_TILED_ROLES) == 0, hex(bits)
    lib.lstm_test_projection_timeout(0, 0, 0)
    binding.lstm_projection(x, rows, 256, whi, wlo, 256, g)
    torch.cuda.synchronize()
    assert binding.lstm_fault_status() == 0
    ref = oracle.projection(x_np, layers[1]["w"])
    assert_within(g.cpu().numpy(), ref, what="projection after timeout")


def test_forward_host_reports_a_timed_out_projection_wait(layers):
    lib = binding.load()
    x = synthetic.stack_input(synthetic.WORKLOADS["b1_t64"])
    s = binding.LSTMStack(layers, 1, 64)
    try:
        y = np.empty((1, 64, 256), np.float32)
        lib.lstm_test_projection_timeout(1, 20000, 0)
        with pytest.raises(binding.LSTMError) as e:
            binding.lstm_stack_forward_host(s.handle, x, y, 1, 64)
        assert e.value.code == binding.LSTM_E_FAULT
        lib.lstm_test_projection_timeout(0, 0, 0)
        binding.lstm_stack_forward_host(s.handle, x, y, 1, 64)
        assert_within(y, oracle.lstm_stack(x, layers), what="forward_host after timeout")
    finally:
        s.close()


def test_heads_wait_timeout_sets_fault_and_recovers():
    import torch
    lib = binding.load()
    hw = synthetic.heads_weights()
    rows = 300
    y_np = synthetic.random_matrix(22, (rows, 256))
    y = cuda(y_np)
    heads = binding.LSTMHeads(hw, rows)
    try:
        assert binding.lstm_fault_status() == 0
        lib.lstm_test_heads_timeout(1, 20000, 0)
        heads(y)
        torch.cuda.synchronize()
        bits = binding.lstm_fault_status()
        assert bits != 0 and (bits & ~FAULT_TILED_ROLES) == 0, hex(bits)
        lib.lstm_test_heads_timeout(0, 0, 0)
        logp = heads(y)
        torch.cuda.synchronize()
        assert binding.lstm_fault_status() == 0
        ref = oracle.heads(y_np, hw["w0"], hw["b0"], hw["w1"], hw["b1"], hw["w2"], hw["b2"])
        assert_within(logp.cpu().numpy(), ref, what="heads after timeout")
    finally:
        heads.close()
