"""The single-product TF32 projection mode (the pages' `CudaMath::Tf32`)
against the oracle's TF32 mode: both factors of every projection product
rounded to TF32, everything else fp32 on the GPU and float64 in the oracle.
Its error against the exact float64 stack is printed: that is the accuracy
question the pages' `tf32_projection_accurate` answers per device."""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu

TF32 = binding.LSTM_MATH_TF32


@pytest.fixture(scope="module")
def layers():
    return synthetic.stack_weights()


@pytest.fixture(scope="module")
def stack(layers):
    s = binding.LSTMStack(layers, 32, 589)
    yield s
    s.close()


@pytest.mark.parametrize("in_width,rows", [(60, 1), (60, 300), (256, 129), (256, 4712)])
def test_tf32_projection_matches_oracle(layers, in_width, rows):
    import torch
    layer = layers[0] if in_width == 60 else layers[1]
    kp = 64 if in_width == 60 else 256
    wp_hi, _, _, _ = binding.lstm_pack_layer(layer["w"], layer["r"], layer["b"], in_width, kp)
    x = synthetic.random_matrix(200 + rows + in_width, (rows, in_width))
    g = torch.full((rows, 1024), float("nan"), device="cuda")
    binding.lstm_projection_math(cuda(x), rows, in_width, cuda(wp_hi), None, kp, g, TF32)
    torch.cuda.synchronize()
    got = g.cpu().numpy()
    # identical fp32 operands round identically on both sides; what is left is
    # the fp32 accumulation order
    assert_within(got, oracle.projection(x, layer["w"], tf32=True), atol=1e-5, rtol=1e-5,
                  what=f"tf32 projection {in_width}x{rows}")
    if rows > 1:
        # and it is the single product: the exact projection is measurably off
        assert np.abs(got - oracle.projection(x, layer["w"])).max() > 1e-5
    assert binding.lstm_fault_status() == 0


@pytest.mark.parametrize("name,idx", [("b1_t64", None), ("b8_t589_x3", None),
                                      ("b32_t589", [0, 13, 31])])
def test_tf32_stack_matches_oracle(stack, layers, name, idx):
    import torch
    wl = synthetic.WORKLOADS[name]
    x = synthetic.stack_input(wl)
    binding.lstm_stack_set_math(stack.handle, TF32)
    try:
        y = stack(cuda(x))
        torch.cuda.synchronize()
    finally:
        binding.lstm_stack_set_math(stack.handle, binding.LSTM_MATH_3XTF32)
    y = y.cpu().numpy()
    idx = list(range(wl.batch)) if idx is None else idx
    ref = oracle.lstm_stack(x[idx], layers, projection="tf32")
    err = assert_within(y[idx], ref, what=f"tf32 stack {name}")
    exact = np.abs(y[idx] - oracle.lstm_stack(x[idx], layers)).max()
    print(f"{name}: TF32 mode vs its oracle {err:.2e}; vs the exact float64 stack {exact:.2e}")
    assert binding.lstm_fault_status() == 0


def test_math_mode_switch_replays_the_right_graph(stack):
    import torch
    x = cuda(synthetic.stack_input(synthetic.WORKLOADS["b1_t64"]))
    outs = {}
    for graphs in (False, True):
        binding.lstm_stack_set_graphs(stack.handle, graphs)
        for math in (TF32, binding.LSTM_MATH_3XTF32, TF32, binding.LSTM_MATH_3XTF32):
            binding.lstm_stack_set_math(stack.handle, math)
            y = torch.full((1, 64, 256), float("nan"), device="cuda")
            stack(x, y)
            torch.cuda.synchronize()
            outs.setdefault(math, []).append(y.cpu().numpy())
    binding.lstm_stack_set_graphs(stack.handle, True)
    for math, ys in outs.items():
        for other in ys[1:]:
            assert np.array_equal(ys[0].view(np.uint32), other.view(np.uint32)), math
    assert not np.array_equal(outs[TF32][0], outs[binding.LSTM_MATH_3XTF32][0])
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_stack_set_math(stack.handle, 7)
    assert e.value.code == binding.LSTM_E_INVALID
