"""The measurement entry points the benchmark reports against: the
recurrence's latency floor (the same launch with the step's arithmetic
removed) runs cleanly and faster than the real recurrence, and the tensor
cores' kind::tf32 rate is a plausible dense rate for this GPU."""
import numpy as np
import pytest

from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import cuda

pytestmark = pytest.mark.gpu


def _pair_ms(fn, g, rp, bias, y, batch, steps):
    import torch
    s0 = torch.cuda.current_stream()
    s1 = torch.cuda.Stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s0)
    s1.wait_event(e0)
    fn(g, rp[0], bias[0], y, batch, steps, 0, s0)
    fn(g, rp[1], bias[1], y, batch, steps, 1, s1)
    j = torch.cuda.Event()
    j.record(s1)
    s0.wait_event(j)
    e1.record(s0)
    e1.synchronize()
    return e0.elapsed_time(e1)


@pytest.mark.parametrize("batch", [1, 32, 256])
def test_recurrence_floor_is_below_the_recurrence(batch):
    import torch
    lay = synthetic.stack_weights()[1]
    wp_hi, wp_lo, rp, bias = binding.lstm_pack_layer(lay["w"], lay["r"], lay["b"], 256, 256)
    steps = 200
    g = cuda(synthetic.random_matrix(5, (batch * steps, 1024)))
    y = torch.zeros((batch, steps, 256), device="cuda")
    rp_d, bias_d = cuda(rp), cuda(bias)
    assert binding.lstm_fault_status() == 0
    full, floor = [], []
    for _ in range(3):
        full.append(_pair_ms(binding.lstm_recurrence, g, rp_d, bias_d, y, batch, steps))
        floor.append(_pair_ms(binding.lstm_recurrence_floor, g, rp_d, bias_d, y, batch, steps))
    assert binding.lstm_fault_status() == 0  # no wait of either kernel ran out
    assert np.all(np.isfinite(y.cpu().numpy()))
    assert min(floor) < min(full), (floor, full)


def test_tf32_rate_is_a_plausible_dense_rate():
    rate = binding.lstm_tf32_rate(0, 20000)
    # GB300: 1.1 PFLOP/s nominal dense TF32; anything far outside means the
    # kernel did not run the MMAs it counts
    assert 300.0 < rate < 2000.0, rate
    assert binding.lstm_fault_status() == 0
