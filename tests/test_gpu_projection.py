"""Parity of the tcgen05 3xTF32 projection (through the C ABI) with the
float64 oracle's packed-column projection, over ragged row counts and both
layer widths."""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def weights():
    return synthetic.stack_weights()


# rows: one row; a full tile; a tile plus one; several tiles with a ragged
# tail; the small workload's 64 rows; up to 2304 rows the kernel runs
# 128-column tiles, above that (the batch-8 workload's 4712 rows) 256-column
# tiles
CASES = [(60, 1), (60, 64), (256, 128), (256, 129), (60, 300), (256, 300), (256, 1024),
         (60, 1025), (256, 1500), (256, 2304), (60, 4712), (256, 4712)]


@pytest.mark.parametrize("in_width,rows", CASES)
def test_projection_matches_oracle(weights, in_width, rows):
    import torch
    layer = weights[0] if in_width == 60 else weights[1]
    kp = 64 if in_width == 60 else 256
    wp_hi, wp_lo, _, _ = binding.lstm_pack_layer(layer["w"], layer["r"], layer["b"], in_width, kp)
    x = synthetic.random_matrix(100 + rows + in_width, (rows, in_width))
    # guard rows past the end must stay untouched (the ragged last tile)
    guard = 37
    g_all = torch.full((rows + guard, 1024), float("nan"), device="cuda")
    g = g_all[:rows]
    binding.lstm_projection(cuda(x), rows, in_width, cuda(wp_hi), cuda(wp_lo), kp, g)
    torch.cuda.synchronize()
    assert torch.isnan(g_all[rows:]).all()
    ref = oracle.projection(x, layer["w"])
    # 3xTF32 keeps fp32-level accuracy: a single TF32 product would miss this
    # bound by ~100x
    assert_within(g.cpu().numpy(), ref, atol=1e-5, rtol=1e-5, what=f"projection {in_width}x{rows}")
    assert binding.lstm_fault_status() == 0


@pytest.mark.parametrize("in_width,kp,rows", [(60, 64, 20011), (20, 32, 20011), (60, 64, 150)])
def test_projection_resident_w_tiles(weights, in_width, kp, rows):
    # K <= 64 keeps each CTA's W tile resident in shared memory across all of
    # its row tiles: rows enough for several tiles per CTA (and a ragged
    # last tile), one or two K blocks of 16 per 32 columns, and a grid
    # smaller than the device
    import torch
    rng = np.random.default_rng(rows + in_width)
    if in_width == 60:
        w = weights[0]["w"]
    else:
        w = rng.uniform(-0.1, 0.1, (2, 512, in_width)).astype(np.float32)
    r = np.zeros((2, 512, 128), np.float32)
    b = np.zeros((2, 1024), np.float32)
    wp_hi, wp_lo, _, _ = binding.lstm_pack_layer(w, r, b, in_width, kp)
    x = synthetic.random_matrix(rows + 5, (rows, in_width))
    g_all = torch.full((rows + 3, 1024), float("nan"), device="cuda")
    g = g_all[:rows]
    binding.lstm_projection(cuda(x), rows, in_width, cuda(wp_hi), cuda(wp_lo), kp, g)
    torch.cuda.synchronize()
    assert torch.isnan(g_all[rows:]).all()
    assert_within(g.cpu().numpy(), oracle.projection(x, w), atol=1e-5, rtol=1e-5,
                  what=f"resident-W projection {in_width}x{rows}")
    assert binding.lstm_fault_status() == 0


def test_projection_large_inputs_exercise_the_lo_plane(weights):
    # inputs of magnitude ~100 make the dropped lo terms visible if any product
    # of the split were missing
    import torch
    layer = weights[1]
    wp_hi, wp_lo, _, _ = binding.lstm_pack_layer(layer["w"], layer["r"], layer["b"], 256, 256)
    rows = 257
    x = synthetic.random_matrix(7, (rows, 256), scale=100.0)
    g = torch.empty((rows, 1024), device="cuda")
    binding.lstm_projection(cuda(x), rows, 256, cuda(wp_hi), cuda(wp_lo), 256, g)
    torch.cuda.synchronize()
    ref = oracle.projection(x, layer["w"])
    assert_within(g.cpu().numpy(), ref, atol=5e-4, rtol=1e-5, what="projection x100")


def test_projection_rejects_misaligned_input(weights):
    import torch
    layer = weights[0]
    wp_hi, wp_lo, _, _ = binding.lstm_pack_layer(layer["w"], layer["r"], layer["b"], 60, 64)
    x = torch.zeros(2 * 60 + 1, device="cuda")[1:]  # 4-byte offset
    g = torch.empty((2, 1024), device="cuda")
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_projection(x, 2, 60, cuda(wp_hi), cuda(wp_lo), 64, g)
    assert e.value.code == binding.LSTM_E_INVALID
