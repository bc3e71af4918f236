"""Benchmark of the four-layer bidirectional LSTM stack on GB300.

One step = one full forward pass of the stack (4 layers x (projection +
forward and reverse recurrences)) over one batch of windows already resident
in HBM.  The default workload is the batch-32 case (32 windows of 589 steps);
the single-window latency case (batch 1, T = 589) is reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
stack on its own GPU with its own batch of windows (weak scaling: windows are
independent, no data exchange); the step time is the maximum over ranks.

Timing: CUDA events on the launching stream around each step; between timed
steps a 256 MiB buffer is written to flush the 129 MB L2 (not timed).  Per-
kernel times come from the library's phase events, recorded on the stream
each kernel runs on, in a short instrumented pass right after the timed steps
(same input, same flush): the 24 event nodes add 4-9 % to a step, so the
timed steps run without them.  SM clocks are sampled with nvidia-smi during the timed
region.  ``--impl reference`` times the float64 CPU oracle on this machine's
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bidirectional_lstm_stack_gb300 import synthetic  # noqa: E402

WORKLOAD = "b32_t589"
LATENCY_WORKLOAD = "b1_t589"
METRIC = "4-layer BiLSTM windows/s and µs/step at B=1,32 (H=128, T=589, fp32)"
FLUSH_BYTES = 256 << 20
LAYERS = synthetic.LAYERS
H = synthetic.HIDDEN

# roofline denominators
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense rates (per GPU) used to scale the measured bf16 peak to TF32
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_TF32_TFLOPS = 1100.0
# FP32 FMA pipe: 152 SMs x 128 lanes x 2 flop per FMA at the SM clock
SMS = 152
FP32_LANES = 128


def peaks():
    try:
        with open(PEAKS_FILE) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def ncu_traffic(kernel: str, rows: int):
    """DRAM bytes per launch from the committed ncu capture of `kernel`, scaled
    to `rows` rows (the kernels' traffic grows in proportion to the rows they
    process); None when the kernel's source changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as fh:
            rec = json.load(fh)[kernel]
        with open(os.path.join(ROOT, rec["source"]), "rb") as fh:
            sha = hashlib.sha256(fh.read()).hexdigest()[:16]
    except (OSError, KeyError, ValueError):
        return None
    if sha != rec["sha256_16"]:
        return None
    return (rec["dram_read_bytes"] + rec["dram_write_bytes"]) * rows / rec["rows"]


def flops_projection(rows: int) -> float:
    """Algorithmic flops of the four projections: 2 * rows * 1024 * K_l."""
    return sum(2.0 * rows * 1024 * (60 if l == 0 else 256) for l in range(LAYERS))


def flops_heads(rows: int) -> float:
    """Algorithmic flops of the dense heads: 2 * rows * (256*128 + 128*128 + 128*7)."""
    return 2.0 * rows * (256 * 128 + 128 * 128 + 128 * 7)


def time_heads(heads, y, steps, warmup, flush, stream):
    """Per-call device time (ms) of the dense heads on the stack output y,
    L2 flushed between calls."""
    import torch
    out = torch.empty((*y.shape[:-1], 7), device=y.device)
    for _ in range(warmup):
        heads.forward(y, out, stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        with torch.cuda.stream(stream):
            flush.fill_(i)
            starts[i].record(stream)
            heads.forward(y, out, stream)
            ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_recurrence_layer(fn, g, rp, bias, y, batch, steps, reps, warmup, flush, stream):
    """Per-step device time (us) of one layer's recurrence, both directions
    in one launch as the stack runs them, through `fn` (lstm_recurrence or
    lstm_recurrence_floor), L2 flushed before each launch; the median over
    `reps` launches."""
    import torch
    from bidirectional_lstm_stack_gb300 import binding
    times = []
    for i in range(warmup + reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.fill_(i)
            e0.record(stream)
        fn(g, rp, bias, y, batch, steps, binding.LSTM_BOTH_DIRECTIONS, stream)
        e1.record(stream)
        e1.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1) * 1e3 / steps)
    return float(np.median(times))


def recurrence_floor(layer, x, stream, flush, reps=5, warmup=3):
    """The recurrence's per-step time and its latency floor on the same
    launch shape, both directions running together: the layer's projection
    of x feeds both; the floor is lstm_recurrence_floor (the same kernel with
    the step's arithmetic replaced by a trivial dependence on the received h).
    Returns (full us/step, floor us/step)."""
    import torch
    from bidirectional_lstm_stack_gb300 import binding
    B, T, F = x.shape
    kp = (F + 31) // 32 * 32
    wp_hi, wp_lo, rp, bias = binding.lstm_pack_layer(layer["w"], layer["r"], layer["b"], F, kp)
    dev = x.device
    whi, wlo = torch.from_numpy(wp_hi).to(dev), torch.from_numpy(wp_lo).to(dev)
    rp_d, bias_d = torch.from_numpy(rp).to(dev), torch.from_numpy(bias).to(dev)
    g = torch.empty((B * T, 1024), device=dev)
    y = torch.empty((B, T, 2 * H), device=dev)
    binding.lstm_projection(x, B * T, F, whi, wlo, kp, g, stream)
    torch.cuda.synchronize()
    full = time_recurrence_layer(binding.lstm_recurrence, g, rp_d, bias_d, y, B, T, reps, warmup,
                                 flush, stream)
    floor = time_recurrence_layer(binding.lstm_recurrence_floor, g, rp_d, bias_d, y, B, T, reps,
                                  warmup, flush, stream)
    # the floor's outputs are meaningless, but no wait of either kernel may
    # have run out (that would void both times)
    bits = binding.lstm_fault_status()
    if bits:
        raise RuntimeError(f"recurrence floor measurement: fault bits {bits:#x}")
    return full, floor


FLOOR_TABLE_BATCHES = (1, 8, 32, 48, 64, 80, 128, 192, 256)


def run_floor_table(args):
    """The recurrence against its per-step latency floor at every batch size
    of FLOOR_TABLE_BATCHES (T = 589, the default variant per batch, both
    directions in one launch, L2 flushed); one JSON line."""
    import torch
    from bidirectional_lstm_stack_gb300 import binding
    torch.cuda.set_device(0)
    layers = synthetic.stack_weights()
    stream = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    steps = synthetic.WORKLOADS[WORKLOAD].steps
    rows = []
    for batch in FLOOR_TABLE_BATCHES:
        x = torch.from_numpy(synthetic.random_matrix(batch, (batch, steps, 60))).cuda()
        full, floor = recurrence_floor(layers[0], x, stream, flush)
        rows.append({"batch": batch, "us_per_step": full, "floor_us_per_step": floor,
                     "vs_floor": full / floor})
    print(json.dumps({"floor_table": rows, "steps": steps,
                      "note": "lstm_recurrence vs lstm_recurrence_floor, both directions in "
                              "one launch, median of 5 after 3 warm-up launches"}))
    return 0


def flops_recurrence_launch(batch: int, steps: int, directions: int = 2) -> float:
    """Algorithmic flops of one recurrence launch (one layer; the stack runs
    both directions in one launch): the 512 x 128 matrix-vector product per
    window, step and direction."""
    return 2.0 * batch * steps * 4 * H * H * directions


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        # "under load": samples above the idle floor
        load = [r for r in rows if r[2] > 0.5 * max(x[2] for x in rows)] or rows
        return {"sm_mhz": float(np.median([r[0] for r in load])),
                "sm_max_mhz": float(max(r[1] for r in rows)),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": float(max(r[2] for r in rows))}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    """The float64 CPU oracle on this host's cores, on a bounded sample of the
    workload: each step runs `sample` windows of the workload's input."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl = synthetic.WORKLOADS[args.workload]
    layers = synthetic.stack_weights()
    x = synthetic.stack_input(wl)
    sample = min(wl.batch, args.reference_windows or wl.batch)
    xs = x[:sample]
    for _ in range(args.warmup):
        oracle.lstm_stack(xs[:1], layers)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.lstm_stack(xs, layers)
        times.append(time.perf_counter() - t0)
    per_step = float(np.mean(times))
    value = sample / per_step
    cores = oracle.threads()
    desc = f"{sample} of the {wl.batch} windows of {wl.name} per step (T={wl.steps}), float64"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "windows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "steps": wl.steps, "hidden": H,
                   "layers": LAYERS, "sample_windows": sample},
        "cpu_baseline": {"value": value, "unit": "windows/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "windows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def cpu_baseline(workload: str, max_seconds: float = 20.0):
    """The oracle as it stands on the host cores: whole windows of the
    workload, as many as fit about `max_seconds` (at least one)."""
    import oracle
    wl = synthetic.WORKLOADS[workload]
    layers = synthetic.stack_weights()
    x = synthetic.stack_input(wl)
    cores = oracle.threads()
    t0 = time.perf_counter()
    oracle.lstm_stack(x[:1], layers)
    one = time.perf_counter() - t0
    # windows run in parallel over (window, direction): estimate what fits
    n = int(max(1, min(wl.batch, (max_seconds / max(one, 1e-6)) * max(1, cores // 2))))
    t0 = time.perf_counter()
    oracle.lstm_stack(x[:n], layers)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "windows/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of the {wl.batch} windows of {wl.name} (T={wl.steps}), float64, "
                      f"{dt:.1f} s"}


def time_stack(stack, x, steps, warmup, flush, stream, with_phases=True, phase_steps=5):
    """Per-step device time (ms) of stack.forward on resident inputs, L2
    flushed between steps; then, in a separate pass (so the timed steps carry
    no extra events), the mean per-phase times."""
    import torch
    from bidirectional_lstm_stack_gb300 import binding
    y = torch.empty((x.shape[0], x.shape[1], 2 * H), device=x.device)
    for _ in range(warmup):
        stack.forward(x, y, stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        with torch.cuda.stream(stream):
            flush.fill_(i)
            starts[i].record(stream)
            stack.forward(x, y, stream)
            ends[i].record(stream)
    torch.cuda.synchronize()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ph = None
    if with_phases:
        binding.lstm_stack_enable_phase_timing(stack.handle, True)
        phases, totals = [], []
        for i in range(phase_steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                flush.fill_(i)
                e0.record(stream)
                stack.forward(x, y, stream)
                e1.record(stream)
            phases.append(binding.lstm_stack_phase_times(stack.handle))
            e1.synchronize()
            totals.append(e0.elapsed_time(e1))
        binding.lstm_stack_enable_phase_timing(stack.handle, False)
        ph = np.mean(np.stack(phases), axis=0)
        # the instrumented pass's own step time, for the gaps between phases
        ph_total = float(np.mean(totals))
        return ms, (ph, ph_total), y
    return ms, ph, y


def run_ours(args):
    import torch
    import torch.distributed as dist

    from bidirectional_lstm_stack_gb300 import binding
    from bidirectional_lstm_stack_gb300.sharding import max_over_ranks

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    wl = synthetic.WORKLOADS[args.workload]
    lat = synthetic.WORKLOADS[LATENCY_WORKLOAD]
    layers = synthetic.stack_weights()
    stack = binding.LSTMStack(layers, max(wl.batch, lat.batch), max(wl.steps, lat.steps), dev)
    stream = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    # weak scaling: every rank runs its own batch of the workload's windows
    x_host = synthetic.stack_input(wl)
    x = torch.from_numpy(x_host).cuda()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clocks:
        ms, (phases, phases_total), y = time_stack(stack, x, args.steps, args.warmup, flush,
                                                   stream)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
    total_s = max_over_ranks(sum(ms) / 1e3, device=torch.device("cuda", dev))
    ms_per_step = total_s * 1e3 / args.steps
    value = wl.batch * world * args.steps / total_s

    # latency case: one window of 589 steps
    x1 = torch.from_numpy(synthetic.stack_input(lat)).cuda()
    ms1, (ph1, ph1_total), _ = time_stack(stack, x1, max(args.steps, 10), args.warmup, flush,
                                          stream)
    ms1_step = max_over_ranks(float(np.mean(ms1)), device=torch.device("cuda", dev))

    # the one-window case with the projection fused into the recurrence
    binding.lstm_stack_set_fused_batches(stack.handle, 1)
    ms1f, (ph1f, _), _ = time_stack(stack, x1, max(args.steps, 10), args.warmup, flush, stream)
    binding.lstm_stack_set_fused_batches(stack.handle, 0)
    ms1f_step = max_over_ranks(float(np.mean(ms1f)), device=torch.device("cuda", dev))

    # the opt-in single-product TF32 projection mode on the same workload (the
    # fp32-accurate 3xTF32 mode above is the headline)
    binding.lstm_stack_set_math(stack.handle, binding.LSTM_MATH_TF32)
    ms_t, (ph_t, _), _ = time_stack(stack, x, args.steps, args.warmup, flush, stream)
    binding.lstm_stack_set_math(stack.handle, binding.LSTM_MATH_3XTF32)
    tf32_s = max_over_ranks(sum(ms_t) / 1e3, device=torch.device("cuda", dev))

    # the segmentation model's dense heads on this forward's output (3 launches)
    heads = binding.LSTMHeads(synthetic.heads_weights(), wl.batch * wl.steps, device=dev)
    ms_h = time_heads(heads, y, args.steps, args.warmup, flush, stream)
    heads.close()
    heads_ms = float(np.mean(ms_h))

    # the recurrence against its latency floor (same kernel and launch shape,
    # the step's arithmetic removed), both directions together, on the
    # workload and on the one-window latency case; and the tensor cores'
    # measured kind::tf32 rate, the projection's and the heads' denominator
    rec_full_us, rec_floor_us = recurrence_floor(layers[0], x, stream, flush)
    rec1_full_us, rec1_floor_us = recurrence_floor(layers[0], x1, stream, flush)
    tf32_rate = binding.lstm_tf32_rate(dev)

    # end to end through the host-buffer entry point (pinned host memory)
    xp = torch.from_numpy(x_host).pin_memory()
    yp = torch.empty((wl.batch, wl.steps, 2 * H), dtype=torch.float32).pin_memory()
    xn, yn = xp.numpy(), yp.numpy()
    for _ in range(args.warmup):
        binding.lstm_stack_forward_host(stack.handle, xn, yn, wl.batch, wl.steps, stream)
    e2e_s = []
    for i in range(args.steps):
        with torch.cuda.stream(stream):
            flush.fill_(i)
        stream.synchronize()
        t0 = time.perf_counter()
        binding.lstm_stack_forward_host(stack.handle, xn, yn, wl.batch, wl.steps, stream)
        e2e_s.append(time.perf_counter() - t0)
    e2e_total = max_over_ranks(sum(e2e_s), device=torch.device("cuda", dev))
    e2e_serial = wl.batch * world * args.steps / e2e_total
    # the same calls enqueued back to back (lstm_stack_forward_host_async):
    # each step still copies its input in and its result out, but one step's
    # output copy and the next step's input copy overlap a forward; results
    # alternate between two pinned output buffers, the L2 flush stays between
    # the forwards
    yp2 = [yp, torch.empty_like(yp).pin_memory()]
    yn2 = [t.numpy() for t in yp2]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        with torch.cuda.stream(stream):
            flush.fill_(i)
        binding.lstm_stack_forward_host_async(stack.handle, xn, yn2[i % 2], wl.batch, wl.steps,
                                              stream)
    binding.lstm_stack_host_sync(stack.handle)
    e2e_pipe_total = max_over_ranks(time.perf_counter() - t0, device=torch.device("cuda", dev))
    e2e_value = wl.batch * world * args.steps / e2e_pipe_total

    # dominant kernel: the recurrence (per launch = one direction of one layer)
    p, peak_kind = peaks()
    clk = clocks.summary()
    rec_ms = float(np.mean(phases[:, 1]))    # mean over layers (one launch, both directions)
    proj_ms = float(np.mean(phases[:, 0]))
    sm_mhz = clk.get("sm_mhz") or 2070.0
    fp32_peak_tflops = SMS * FP32_LANES * 2 * (clk.get("sm_max_mhz") or 2070.0) * 1e6 / 1e12
    rec_flops = flops_recurrence_launch(wl.batch, wl.steps)
    rec_achieved = rec_flops / (rec_ms * 1e-3) / 1e12
    tf32_peak = p["bf16_tflops"] * NOMINAL_TF32_TFLOPS / NOMINAL_BF16_TFLOPS
    proj_peak = tf32_peak / 3.0    # 3xTF32: three TF32 products per fp32 product
    proj_achieved = flops_projection(wl.batch * wl.steps) / LAYERS / (proj_ms * 1e-3) / 1e12
    us_per_layer_step = ms_per_step * 1e3 / (LAYERS * wl.steps)
    rec_us_per_step = rec_ms * 1e3 / wl.steps

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "windows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "steps": wl.steps, "hidden": H,
                   "layers": LAYERS, "inputs": wl.description,
                   "l2": "flushed: 256 MiB written between timed steps",
                   "parallelism": f"windows sharded, {wl.batch} per GPU" if world > 1
                   else "1 GPU"},
        "us_per_step": us_per_layer_step,
        "latency_b1": {"workload": lat.name, "ms_per_window": ms1_step,
                       "windows_per_s": 1e3 / ms1_step,
                       "us_per_step": ms1_step * 1e3 / (LAYERS * lat.steps),
                       "recurrence_us_per_step": float(np.mean(ph1[:, 1])) * 1e3 / lat.steps,
                       "phases_ms": {"projection": [round(float(v), 4) for v in ph1[:, 0]],
                                     "recurrence": [round(float(v), 4) for v in ph1[:, 1]]},
                       "gaps_ms": ph1_total - float(np.sum(ph1[:, 0]) +
                                                   np.sum(ph1[:, 1])),
                       "recurrence_pair_us_per_step": rec1_full_us,
                       "floor_us_per_step": rec1_floor_us,
                       "vs_floor": rec1_full_us / rec1_floor_us,
                       "fused_projection": {
                           "ms_per_window": ms1f_step, "windows_per_s": 1e3 / ms1f_step,
                           "recurrence_ms": [round(float(v), 4) for v in ph1f[:, 1]],
                           "mode": "lstm_stack_set_fused_batches: each layer one launch, the "
                                   "input projection computed inside the recurrence"},
                       "context": "pages: A100, TF32-projection stack, 3.21-4.13 ms per window"},
        "gaps_ms": phases_total - float(np.sum(phases[:, 0]) +
                                        np.sum(phases[:, 1])),
        "phases_pass_ms_per_step": phases_total,
        "phases_ms": {"projection": [round(float(v), 4) for v in phases[:, 0]],
                      "recurrence": [round(float(v), 4) for v in phases[:, 1]]},
        "roofline": {"kernel": "recurrence (one layer, both directions in one launch)",
                     "bound": "alu",
                     "achieved": rec_achieved, "peak": fp32_peak_tflops, "unit": "TFLOP/s",
                     "frac": rec_achieved / fp32_peak_tflops,
                     "traffic": ncu_traffic("recurrence", wl.batch * wl.steps),
                     "algorithmic_bytes": float(2 * wl.batch * wl.steps * (512 + 128) * 4),
                     "peak_source": "152 SMs x 128 FP32 lanes x 2 flop x max SM clock",
                     "us_per_step": rec_us_per_step,
                     "pair_us_per_step": rec_full_us,
                     "floor_us_per_step": rec_floor_us,
                     "vs_floor": rec_full_us / rec_floor_us,
                     "floor_source": "lstm_recurrence_floor: the same variant, grid, exchange "
                                     "and waits with the step's arithmetic removed; both "
                                     "directions in one launch, L2 flushed, median of 5"},
        "roofline_projection": {"kernel": "projection (one layer, both directions)",
                                "bound": "tensor", "achieved": proj_achieved, "peak": proj_peak,
                                "unit": "TFLOP/s", "frac": proj_achieved / proj_peak,
                                "traffic": ncu_traffic("projection", wl.batch * wl.steps),
                                "peak_source": f"{peak_kind} bf16 burst {p['bf16_tflops']} x "
                                               f"{NOMINAL_TF32_TFLOPS}/{NOMINAL_BF16_TFLOPS} "
                                               f"(TF32) / 3 (3xTF32)",
                                "tf32_measured_tflops": tf32_rate,
                                "frac_of_measured_tf32": proj_achieved / (tf32_rate / 3.0)},
        "tf32_mode": {"windows_per_s": wl.batch * world * args.steps / tf32_s,
                      "ms_per_step": tf32_s * 1e3 / args.steps,
                      "projection_ms": [round(float(v), 4) for v in ph_t[:, 0]]},
        "heads": {"kernels": "linear0+LeakyReLU, linear1+LeakyReLU, classifier+log-softmax",
                  "rows": wl.batch * wl.steps, "ms": heads_ms,
                  "achieved_tflops": flops_heads(wl.batch * wl.steps) / (heads_ms * 1e-3) / 1e12,
                  "frac_of_3xtf32_peak": flops_heads(wl.batch * wl.steps) / (heads_ms * 1e-3)
                  / 1e12 / proj_peak,
                  "frac_of_measured_3xtf32": flops_heads(wl.batch * wl.steps) / (heads_ms * 1e-3)
                  / 1e12 / (tf32_rate / 3.0)},
        "e2e": {"value": e2e_value, "unit": "windows/s",
                "h2d_bytes_per_step": int(xn.nbytes), "d2h_bytes_per_step": int(yn.nbytes),
                "mode": "forward_host_async, steps enqueued back to back (copies of one step "
                        "overlap the next forward), host clock around all steps",
                "serial_value": e2e_serial},
        "gpu_launches": 8 * args.steps,  # per forward: 4 projections, 4 two-direction recurrences
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl.name)
    if rank == 0:
        print(json.dumps(line))
    stack.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--reference-windows", type=int, default=0,
                    help="windows per step of the --impl reference run (default: the "
                         "workload's whole batch)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--floor-table", action="store_true",
                    help="print the recurrence's per-step time against its latency floor "
                         "for a range of batch sizes instead of the benchmark line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.floor_table:
        return run_floor_table(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
