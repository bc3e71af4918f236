"""Seeded synthetic weights and inputs for the LSTM stack.

This module only draws random numbers; it holds none of the method's
arithmetic, so both the CUDA path's tests and the float64 oracle can take their
inputs from it.

The shapes follow the stack the speakrs 0.6.0 pages describe (``lstmproj.rs``:
``FEATURES`` = 60 input features, ``HIDDEN`` = 128, four layers, two
directions; the source weight lengths in ``Oxide::with_recurrence``).  The
pages' model runs on 10 s audio windows of 589 frames (``lstmproj.rs``,
``driver_pin``); audio and trained weights are not available, so seeded random
data of the same shapes stands in for them:

* every W, R, Wb and Rb entry is i.i.d. U(-1/sqrt(128), 1/sqrt(128)) from the
  weight seed (the usual LSTM initialisation range for hidden size 128);
* inputs are N(0, 1) per feature, optionally scaled (x3 pushes the gates into
  saturation) and with whole frames zeroed with a given probability (silence).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

FEATURES = 60
HIDDEN = 128
LAYERS = 4
GATES = 4 * HIDDEN


@dataclass(frozen=True)
class Workload:
    """One synthetic configuration of the stack's input."""
    name: str
    batch: int
    steps: int
    scale: float = 1.0
    zero_frames: float = 0.0
    seed: int = 1
    description: str = ""


#: The five workloads: a small case, the single-window latency case, a
#: saturating case, the model's batch-32 case and a large-batch case.
WORKLOADS = {
    "b1_t64": Workload("b1_t64", 1, 64, seed=1,
                       description="batch 1, T=64, N(0,1)"),
    "b1_t589": Workload("b1_t589", 1, 589, seed=2,
                        description="batch 1, T=589 (one 10 s window), N(0,1)"),
    "b8_t589_x3": Workload("b8_t589_x3", 8, 589, scale=3.0, seed=3,
                           description="batch 8, T=589, 3*N(0,1) (saturating)"),
    "b32_t589": Workload("b32_t589", 32, 589, seed=4,
                         description="batch 32, T=589, N(0,1)"),
    "b256_t589_z5": Workload("b256_t589_z5", 256, 589, zero_frames=0.05,
                             seed=5,
                             description="batch 256, T=589, N(0,1), 5% of "
                                         "frames zeroed"),
}

WEIGHT_SEED = 0


def stack_weights(seed: int = WEIGHT_SEED, hidden: int = HIDDEN,
                  features: int = FEATURES, layers: int = LAYERS,
                  dtype=np.float32):
    """Random weights in the library's source layout.

    Returns a list of ``layers`` dicts with ``w`` ``[2, 4H, in_l]``, ``r``
    ``[2, 4H, H]`` and ``b`` ``[2, 8H]`` (per direction Wb[4H] then Rb[4H]),
    gate row blocks in the order i, f, g, o.  ``in_0 = features`` and
    ``in_l = 2H`` after the first layer.
    """
    rng = np.random.default_rng(seed)
    bound = 1.0 / np.sqrt(hidden)
    out = []
    for l in range(layers):
        inw = features if l == 0 else 2 * hidden
        w = rng.uniform(-bound, bound, size=(2, 4 * hidden, inw))
        r = rng.uniform(-bound, bound, size=(2, 4 * hidden, hidden))
        b = rng.uniform(-bound, bound, size=(2, 8 * hidden))
        out.append({"w": w.astype(dtype), "r": r.astype(dtype),
                    "b": b.astype(dtype)})
    return out


HEADS_SEED = 7


def heads_weights(seed: int = HEADS_SEED, dtype=np.float32):
    """Random weights of the segmentation model's dense heads, row-major
    ``[k, n]``: w0 ``[256, 128]``, w1 ``[128, 128]``, w2 ``[128, 7]`` and the
    biases ``[n]``, every entry U(-1/sqrt(k), 1/sqrt(k)) for its layer's
    input width k (the default range of a freshly initialised linear
    layer)."""
    rng = np.random.default_rng(seed)
    out = {}
    for name, (k, n) in (("0", (2 * HIDDEN, 128)), ("1", (128, 128)), ("2", (128, 7))):
        bound = 1.0 / np.sqrt(k)
        out["w" + name] = rng.uniform(-bound, bound, size=(k, n)).astype(dtype)
        out["b" + name] = rng.uniform(-bound, bound, size=(n,)).astype(dtype)
    return out


def stack_input(workload: Workload, features: int = FEATURES,
                dtype=np.float32) -> np.ndarray:
    """The input ``[B, T, features]`` of a workload, from its seed."""
    rng = np.random.default_rng(workload.seed)
    x = rng.standard_normal((workload.batch, workload.steps, features))
    x *= workload.scale
    if workload.zero_frames > 0.0:
        drop = rng.random((workload.batch, workload.steps)) < workload.zero_frames
        x[drop] = 0.0
    return x.astype(dtype)


def random_matrix(seed: int, shape, scale: float = 1.0,
                  dtype=np.float32) -> np.ndarray:
    """A seeded N(0, scale^2) array, for step-level tests."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(dtype)
