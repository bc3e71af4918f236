"""The segmentation model's dense heads (linear0 + LeakyReLU, linear1 +
LeakyReLU, classifier + log-softmax) through the C ABI against the float64
oracle: on their own over ragged row counts, and behind the stack."""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hw():
    return synthetic.heads_weights()


@pytest.fixture(scope="module")
def heads(hw):
    h = binding.LSTMHeads(hw, 32 * 589)
    yield h
    h.close()


def _oracle(y, hw, slope=0.01):
    return oracle.heads(y, hw["w0"], hw["b0"], hw["w1"], hw["b1"], hw["w2"], hw["b2"], slope)


@pytest.mark.parametrize("rows", [1, 64, 129, 300, 589, 4712])
def test_heads_match_oracle(heads, hw, rows):
    import torch
    # stack outputs are hidden states in (-1, 1)
    y = synthetic.random_matrix(300 + rows, (rows, 256)) * 0.5
    guard = 9
    out_all = torch.full((rows + guard, 7), float("nan"), device="cuda")
    out = out_all[:rows]
    heads(cuda(y), out)
    torch.cuda.synchronize()
    assert torch.isnan(out_all[rows:]).all()
    got = out.cpu().numpy()
    assert_within(got, _oracle(y, hw), atol=1e-5, rtol=1e-5, what=f"heads {rows} rows")
    np.testing.assert_allclose(np.exp(got.astype(np.float64)).sum(axis=1), 1.0, atol=1e-5)
    assert binding.lstm_fault_status() == 0


def test_heads_negative_slope(hw):
    import torch
    h = binding.LSTMHeads(hw, 256, negative_slope=0.2)
    try:
        y = synthetic.random_matrix(77, (200, 256))
        got = h(cuda(y))
        torch.cuda.synchronize()
    finally:
        h.close()
    assert_within(got.cpu().numpy(), _oracle(y, hw, 0.2), atol=1e-5, rtol=1e-5,
                  what="heads slope 0.2")
    assert np.abs(got.cpu().numpy() - _oracle(y, hw, 0.01)).max() > 1e-4


def test_stack_then_heads_match_oracle(heads, hw):
    import torch
    layers = synthetic.stack_weights()
    wl = synthetic.WORKLOADS["b8_t589_x3"]
    x = synthetic.stack_input(wl)
    s = binding.LSTMStack(layers, 8, 589)
    try:
        y = s(cuda(x))
        logp = heads(y)
        torch.cuda.synchronize()
    finally:
        s.close()
    ref = _oracle(oracle.lstm_stack(x, layers).reshape(-1, 256), hw).reshape(8, 589, 7)
    assert_within(logp.cpu().numpy(), ref, what="stack + heads")


def test_heads_argument_errors(heads):
    import torch
    lib = binding.load()
    y = torch.zeros((10, 256), device="cuda")
    out = torch.zeros((10, 7), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    h = heads.handle
    assert lib.lstm_heads_forward(h, y.data_ptr(), 2559, out.data_ptr(), 70, 10,
                                  s) == binding.LSTM_E_LENGTH
    assert lib.lstm_heads_forward(h, y.data_ptr(), 2560, out.data_ptr(), 71, 10,
                                  s) == binding.LSTM_E_LENGTH
    big = heads.max_rows + 1
    assert lib.lstm_heads_forward(h, y.data_ptr(), big * 256, out.data_ptr(), big * 7, big,
                                  s) == binding.LSTM_E_INVALID
    ym = torch.zeros(10 * 256 + 1, device="cuda")[1:]
    assert lib.lstm_heads_forward(h, ym.data_ptr(), 2560, out.data_ptr(), 70, 10,
                                  s) == binding.LSTM_E_INVALID
