"""The whole stack through the C ABI against the float64 oracle on the five
synthetic workloads (the large ones on sampled windows, which are
independent), plus determinism, the host-buffer entry point and argument
errors with a live device."""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu

MAX_BATCH, MAX_STEPS = 256, 589


@pytest.fixture(scope="module")
def layers():
    return synthetic.stack_weights()


@pytest.fixture(scope="module")
def stack(layers):
    s = binding.LSTMStack(layers, MAX_BATCH, MAX_STEPS)
    yield s
    s.close()


def _forward(stack, x):
    import torch
    y = stack(cuda(x))
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("name", list(synthetic.WORKLOADS))
def test_stack_matches_oracle(stack, layers, name):
    # every window of every workload (the oracle runs the 256 windows of the
    # largest in about 8 s on 16 cores)
    wl = synthetic.WORKLOADS[name]
    x = synthetic.stack_input(wl)
    y = _forward(stack, x)
    ref = oracle.lstm_stack(x, layers)
    assert_within(y, ref, what=name)
    assert binding.lstm_fault_status() == 0


def test_stack_ragged_small_shapes(stack, layers):
    for batch, steps in [(1, 1), (2, 3), (7, 129), (19, 40), (41, 30), (83, 12), (130, 9),
                         (192, 5)]:
        x = synthetic.random_matrix(batch * 1000 + steps, (batch, steps, 60))
        y = _forward(stack, x)
        assert_within(y, oracle.lstm_stack(x, layers), what=f"stack b{batch} t{steps}")


def test_stack_is_deterministic_and_host_path_matches(stack):
    x = synthetic.stack_input(synthetic.WORKLOADS["b8_t589_x3"])
    y1 = _forward(stack, x)
    y2 = _forward(stack, x)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    yh = np.empty_like(y1)
    binding.lstm_stack_forward_host(stack.handle, np.ascontiguousarray(x), yh, 8, 589)
    assert np.array_equal(y1.view(np.uint32), yh.view(np.uint32))


def test_async_host_calls_in_flight(stack, layers):
    # five calls in a row, different shapes and inputs, results collected at
    # the end: the staging slots are reused (calls 3-5) while earlier output
    # copies may still be in flight; every output equals the device path
    import torch
    shapes = [(3, 40), (5, 17), (2, 64), (4, 33), (1, 9)]
    xs = [synthetic.random_matrix(300 + i, (b, t, 60)) for i, (b, t) in enumerate(shapes)]
    xp = [torch.from_numpy(x).pin_memory() for x in xs]
    yp = [torch.full((b, t, 256), float("nan")).pin_memory() for b, t in shapes]
    for (b, t), xi, yi in zip(shapes, xp, yp):
        binding.lstm_stack_forward_host_async(stack.handle, xi.numpy(), yi.numpy(), b, t)
    binding.lstm_stack_host_sync(stack.handle)
    for x, yi in zip(xs, yp):
        ref = _forward(stack, x)
        assert np.array_equal(ref.view(np.uint32), yi.numpy().view(np.uint32))
    assert_within(yp[0].numpy(), oracle.lstm_stack(xs[0], layers), what="async host call")


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_async_host_call_rejects_a_capturing_stream(stack):
    import torch
    x = np.zeros((1, 4, 60), np.float32)
    y = np.zeros((1, 4, 256), np.float32)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(binding.LSTMError) as e:
        with torch.cuda.graph(g, stream=s):
            binding.lstm_stack_forward_host_async(stack.handle, x, y, 1, 4, s)
    assert e.value.code == binding.LSTM_E_INVALID
    torch.cuda.synchronize()
    # the stack still works afterwards
    binding.lstm_stack_forward_host(stack.handle, x, y, 1, 4)


def test_stack_phase_timing(stack):
    import torch
    x = cuda(synthetic.stack_input(synthetic.WORKLOADS["b1_t64"]))
    binding.lstm_stack_enable_phase_timing(stack.handle, True)
    stack(x)
    ms = binding.lstm_stack_phase_times(stack.handle)
    binding.lstm_stack_enable_phase_timing(stack.handle, False)
    torch.cuda.synchronize()
    assert ms.shape == (4, 3) and np.all(ms > 0)


def test_stack_argument_errors(stack):
    import torch
    x = torch.zeros((2, 10, 60), device="cuda")
    y = torch.zeros((2, 10, 256), device="cuda")
    h = stack.handle
    lib = binding.load()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.lstm_stack_forward(h, x.data_ptr(), x.numel() - 1, y.data_ptr(), y.numel(), 2, 10,
                                  s) == binding.LSTM_E_LENGTH
    assert "expected" in binding.lstm_stack_last_error()
    assert lib.lstm_stack_forward(h, x.data_ptr(), x.numel(), y.data_ptr(), y.numel() + 1, 2, 10,
                                  s) == binding.LSTM_E_LENGTH
    big = MAX_BATCH + 1
    assert lib.lstm_stack_forward(h, x.data_ptr(), big * 10 * 60, y.data_ptr(), big * 10 * 256,
                                  big, 10, s) == binding.LSTM_E_INVALID
    assert lib.lstm_stack_forward(h, x.data_ptr(), 0, y.data_ptr(), 0, 0, 10,
                                  s) == binding.LSTM_E_INVALID
    xm = torch.zeros(2 * 10 * 60 + 1, device="cuda")[1:]
    assert lib.lstm_stack_forward(h, xm.data_ptr(), 1200, y.data_ptr(), y.numel(), 2, 10,
                                  s) == binding.LSTM_E_INVALID
    xh = np.zeros(1200, np.float32)
    assert lib.lstm_stack_forward(h, xh.ctypes.data, 1200, y.data_ptr(), y.numel(), 2, 10,
                                  s) == binding.LSTM_E_INVALID


def test_graph_replay_matches_direct_launches(stack):
    import torch
    x = cuda(synthetic.stack_input(synthetic.WORKLOADS["b8_t589_x3"]))
    outs = []
    for graphs in (False, True, True):
        binding.lstm_stack_set_graphs(stack.handle, graphs)
        y = torch.full((8, 589, 256), float("nan"), device="cuda")
        stack(x, y)
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy())
    binding.lstm_stack_set_graphs(stack.handle, True)
    for o in outs[1:]:
        assert np.array_equal(outs[0].view(np.uint32), o.view(np.uint32))


def test_small_batch_early_recurrence_start_changes_no_bit(stack):
    # at one window the recurrence is launched as a programmatic dependent of
    # the projection (its set-up overlaps the projection); with phase timing
    # on an event sits between them and it starts after: the same bits, with
    # and without graph replay
    import torch
    x = cuda(synthetic.stack_input(synthetic.WORKLOADS["b1_t589"]))
    outs = []
    try:
        for timing, graphs in ((True, False), (False, False), (False, True), (False, True)):
            binding.lstm_stack_enable_phase_timing(stack.handle, timing)
            binding.lstm_stack_set_graphs(stack.handle, graphs)
            y = torch.full((1, 589, 256), float("nan"), device="cuda")
            stack(x, y)
            torch.cuda.synchronize()
            outs.append(y.cpu().numpy())
    finally:
        binding.lstm_stack_enable_phase_timing(stack.handle, False)
        binding.lstm_stack_set_graphs(stack.handle, True)
    for o in outs[1:]:
        assert np.array_equal(outs[0].view(np.uint32), o.view(np.uint32))
    assert binding.lstm_fault_status() == 0


@pytest.mark.parametrize("timing", [False, True])
@pytest.mark.parametrize("graphs", [False, True])
@pytest.mark.parametrize("math", ["3xtf32", "tf32"])
@pytest.mark.parametrize("fused", [0, 1])
def test_setting_combinations(stack, layers, timing, graphs, math, fused):
    # every combination of phase timing, graph replay, projection math and
    # the fused small-batch mode runs and stays within the stack's tolerance
    # of the exact float64 stack (the TF32 mode's own error is ~3e-5)
    import torch
    x = synthetic.stack_input(synthetic.WORKLOADS["b1_t64"])
    h = stack.handle
    try:
        binding.lstm_stack_enable_phase_timing(h, timing)
        binding.lstm_stack_set_graphs(h, graphs)
        binding.lstm_stack_set_math(h, binding.LSTM_MATH_TF32 if math == "tf32"
                                    else binding.LSTM_MATH_3XTF32)
        binding.lstm_stack_set_fused_batches(h, fused)
        y = stack(cuda(x))
        torch.cuda.synchronize()
        if timing:
            assert np.all(binding.lstm_stack_phase_times(h) >= 0)
        # the host-memory entry point runs the same kernels: the same bits
        yh = np.empty((1, 64, 256), np.float32)
        binding.lstm_stack_forward_host(h, np.ascontiguousarray(x), yh, 1, 64)
        assert np.array_equal(yh.view(np.uint32), y.cpu().numpy().view(np.uint32))
    finally:
        binding.lstm_stack_enable_phase_timing(h, False)
        binding.lstm_stack_set_graphs(h, True)
        binding.lstm_stack_set_math(h, binding.LSTM_MATH_3XTF32)
        binding.lstm_stack_set_fused_batches(h, 0)
    what = f"timing {timing} graphs {graphs} math {math} fused {fused}"
    assert_within(y.cpu().numpy(), oracle.lstm_stack(x, layers), what=what)
    assert binding.lstm_fault_status() == 0


def test_forward_inside_a_caller_graph_capture(stack, layers):
    # the forward is capturable: a caller's CUDA graph records its launches
    import torch
    x_np = synthetic.random_matrix(77, (3, 50, 60))
    x = cuda(x_np)
    y = torch.full((3, 50, 256), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        stack(x, y, s)  # warm-up outside capture (variant tables, tensor maps)
    torch.cuda.synchronize()
    y.fill_(float("nan"))
    with torch.cuda.graph(g, stream=s):
        stack(x, y, s)
    g.replay()
    torch.cuda.synchronize()
    assert_within(y.cpu().numpy(), oracle.lstm_stack(x_np, layers), what="captured forward")


def _to_iofc(a, axis):
    """Reorders i, f, g, o row blocks into ONNX's i, o, f, c."""
    i, f, g, o = np.split(a, 4, axis=axis)
    return np.concatenate([i, o, f, g], axis=axis)


def test_onnx_gate_order_stack(stack, layers):
    # the same stack from ONNX-ordered weights gives the same bits
    onnx = [{"w": _to_iofc(l["w"], 1), "r": _to_iofc(l["r"], 1),
             "b": np.concatenate([_to_iofc(l["b"][:, :512], 1), _to_iofc(l["b"][:, 512:], 1)],
                                 axis=1)} for l in layers]
    x = synthetic.stack_input(synthetic.WORKLOADS["b8_t589_x3"])
    s2 = binding.LSTMStack(onnx, 8, 589, gate_order=binding.LSTM_GATES_IOFC)
    try:
        import torch
        y2 = s2(cuda(x))
        torch.cuda.synchronize()
        y2 = y2.cpu().numpy()
    finally:
        s2.close()
    y1 = _forward(stack, x)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert_within(y2, oracle.lstm_stack(x, layers), what="onnx gate order")


def test_two_host_threads_with_their_own_stacks(layers):
    # per-thread error state, per-stack scratch and thread-local graph capture:
    # two threads forwarding concurrently on their own streams agree with the
    # oracle (and with each other on the same input)
    import threading

    import torch
    wl = synthetic.WORKLOADS["b8_t589_x3"]
    x_np = synthetic.stack_input(wl)
    results, errors = {}, []

    def worker(k):
        try:
            torch.cuda.set_device(0)
            s = binding.LSTMStack(layers, 8, 589)
            stream = torch.cuda.Stream()
            x = cuda(x_np)
            with torch.cuda.stream(stream):
                outs = [s(x, None, stream) for _ in range(3)]
            stream.synchronize()
            results[k] = [o.cpu().numpy() for o in outs]
            s.close()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    ref = oracle.lstm_stack(x_np, layers)
    first = results[0][0]
    for k in range(2):
        for y in results[k]:
            assert np.array_equal(y.view(np.uint32), first.view(np.uint32))
    assert_within(first, ref, what="threads")


def test_per_layer_error_localises_drift(layers):
    # the stack layer by layer through the step entry points: each layer's
    # error on its own (GPU) input, and the error accumulated from x
    import torch
    wl = synthetic.WORKLOADS["b8_t589_x3"]
    x = synthetic.stack_input(wl)
    B, T = wl.batch, wl.steps
    cur = cuda(x.reshape(B * T, 60))
    ref_chain = x
    for l, lay in enumerate(layers):
        inw, kp = (60, 64) if l == 0 else (256, 256)
        wp_hi, wp_lo, rp, bias = binding.lstm_pack_layer(lay["w"], lay["r"], lay["b"], inw, kp)
        g = torch.empty((B * T, 1024), device="cuda")
        y = torch.empty((B, T, 256), device="cuda")
        binding.lstm_projection(cur, B * T, inw, cuda(wp_hi), cuda(wp_lo), kp, g)
        rpt, bt = cuda(rp), cuda(bias)
        for d in range(2):
            binding.lstm_recurrence(g, rpt[d], bt[d], y, B, T, d)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        local = oracle.lstm_stack(cur.cpu().numpy().reshape(B, T, inw), [lay])
        ref_chain = oracle.lstm_stack(ref_chain, [lay])
        e_local = assert_within(got, local, what=f"layer {l} on its own input")
        e_chain = assert_within(got, ref_chain, what=f"layer {l} from x")
        print(f"layer {l}: max abs err {e_local:.2e} on its input, {e_chain:.2e} from x")
        cur = y.reshape(B * T, 256)
    assert binding.lstm_fault_status() == 0
