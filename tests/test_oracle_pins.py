"""Pins of the float64 oracle to things other than itself.

Each check is chosen so that a plausible mistake in the oracle (a dropped
bias, a swapped gate block, a transposed R, h_t used instead of h_{t-1}, the
reverse direction writing time-flipped rows, the concat halves swapped, a wrong
packed column) fails at least one of them:

* zero weights give exactly zero output (sigmoid(0)=1/2, tanh(0)=0);
* with R = 0 and the forget gate shut, every step has a closed form;
* with R = 0 and any forget gate, the cell state is the explicit
  product-sum  c_t = sum_s (prod_{r>s} f_r) i_s g_s;
* the reverse direction equals the forward one on time-reversed input, for a
  single direction and through all four layers;
* a saturated-gate counter whose hidden states are tanh of hand-derived
  integers (tests/golden/saturated_counter.json);
* agreement with torch.nn.LSTM in float64 (a library routine with the same
  i,f,g,o gate blocks and separate input/recurrent biases);
* brute force on H = 2, T = 3, input 2, both directions: every gate written
  out as scalar arithmetic;
* the packed projection against a one-hot W and against numpy's matmul;
* TF32 projection mode: the oracle's rounding against a definition written
  on the bit layout (keep sign, exponent and the top 10 mantissa bits; the
  dropped bits at or above half round the magnitude up), and the TF32 stack
  against the float64 stack run layer by layer on operands rounded that way.
"""
import json
import os

import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import synthetic

HERE = os.path.dirname(os.path.abspath(__file__))


def _layers(rng, H, in0, L, scale=0.3):
    out = []
    for l in range(L):
        inw = in0 if l == 0 else 2 * H
        out.append({
            "w": rng.uniform(-scale, scale, (2, 4 * H, inw)),
            "r": rng.uniform(-scale, scale, (2, 4 * H, H)),
            "b": rng.uniform(-scale, scale, (2, 8 * H)),
        })
    return out


def _sig(z):
    return 1.0 / (1.0 + np.exp(-z))


def test_zero_weights_give_exact_zero():
    rng = np.random.default_rng(10)
    H, in0, L, B, T = 8, 5, 4, 3, 11
    layers = [{k: np.zeros_like(v) for k, v in l.items()}
              for l in _layers(rng, H, in0, L)]
    x = rng.standard_normal((B, T, in0)) * 5
    y = oracle.lstm_stack(x, layers)
    assert y.shape == (B, T, 2 * H)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("reverse", [False, True])
def test_r_zero_forget_shut_closed_form(reverse):
    rng = np.random.default_rng(11)
    H, inw, T = 6, 4, 9
    W = rng.uniform(-1, 1, (4 * H, inw))
    Wb = rng.uniform(-1, 1, 4 * H)
    Rb = rng.uniform(-1, 1, 4 * H)
    Wb[H:2 * H] = -1.0e3  # forget gate exactly 0 in float64
    R = np.zeros((4 * H, H))
    x = rng.standard_normal((T, inw))
    h = oracle.lstm_direction(x, W, R, Wb, Rb, reverse)
    z = x @ W.T + Wb + Rb  # [T, 4H]
    zi, zg, zo = z[:, :H], z[:, 2 * H:3 * H], z[:, 3 * H:]
    expect = _sig(zo) * np.tanh(_sig(zi) * np.tanh(zg))
    np.testing.assert_allclose(h, expect, rtol=0, atol=1e-14)


@pytest.mark.parametrize("reverse", [False, True])
def test_r_zero_product_sum_cell(reverse):
    rng = np.random.default_rng(12)
    H, inw, T = 5, 3, 12
    W = rng.uniform(-1, 1, (4 * H, inw))
    Wb = rng.uniform(-1, 1, 4 * H)
    Rb = rng.uniform(-1, 1, 4 * H)
    R = np.zeros((4 * H, H))
    x = rng.standard_normal((T, inw))
    h = oracle.lstm_direction(x, W, R, Wb, Rb, reverse)
    z = x @ W.T + Wb + Rb
    i = _sig(z[:, :H])
    f = _sig(z[:, H:2 * H])
    g = np.tanh(z[:, 2 * H:3 * H])
    o = _sig(z[:, 3 * H:])
    order = list(range(T))[::-1] if reverse else list(range(T))
    expect = np.zeros((T, H))
    for n, t in enumerate(order):
        # c at the n-th visited step: sum over earlier visits s of
        # (product of the forget gates visited after s) * i_s * g_s
        c = np.zeros(H)
        for m in range(n + 1):
            s = order[m]
            prod = np.ones(H)
            for q in range(m + 1, n + 1):
                prod = prod * f[order[q]]
            c = c + prod * i[s] * g[s]
        expect[t] = o[t] * np.tanh(c)
    np.testing.assert_allclose(h, expect, rtol=0, atol=1e-13)


def test_reverse_is_forward_on_flipped_time_single_direction():
    rng = np.random.default_rng(13)
    H, inw, T = 7, 5, 10
    W = rng.uniform(-0.5, 0.5, (4 * H, inw))
    R = rng.uniform(-0.5, 0.5, (4 * H, H))
    Wb = rng.uniform(-0.5, 0.5, 4 * H)
    Rb = rng.uniform(-0.5, 0.5, 4 * H)
    x = rng.standard_normal((T, inw))
    rev = oracle.lstm_direction(x, W, R, Wb, Rb, True)
    fwd_flipped = oracle.lstm_direction(x[::-1], W, R, Wb, Rb, False)
    assert np.array_equal(rev, fwd_flipped[::-1])


def test_reverse_is_forward_on_flipped_time_whole_stack():
    # With W_rev = W_fwd (input-column halves swapped from the second layer
    # on, since the flipped input's layer outputs arrive with swapped halves),
    # R_rev = R_fwd and b_rev = b_fwd, the identity
    #     y(x)[t, H:] == y(flip x)[T-1-t, :H]
    # holds at every layer of the stack.
    rng = np.random.default_rng(14)
    H, in0, L, B, T = 6, 4, 4, 2, 8
    layers = _layers(rng, H, in0, L)
    for l, lay in enumerate(layers):
        w_f = lay["w"][0]
        if l == 0:
            w_r = w_f.copy()
        else:
            w_r = np.concatenate([w_f[:, H:], w_f[:, :H]], axis=1)
        lay["w"] = np.stack([w_f, w_r])
        lay["r"] = np.stack([lay["r"][0], lay["r"][0]])
        lay["b"] = np.stack([lay["b"][0], lay["b"][0]])
    x = rng.standard_normal((B, T, in0))
    y = oracle.lstm_stack(x, layers)
    yf = oracle.lstm_stack(x[:, ::-1], layers)
    np.testing.assert_allclose(y[:, :, H:], yf[:, ::-1, :H], rtol=0, atol=1e-13)
    np.testing.assert_allclose(y[:, :, :H], yf[:, ::-1, H:], rtol=0, atol=1e-13)


def _counts_from_rules(x):
    """The saturated counter's cell counts, derived from its sign rules."""
    sign = lambda v: int(v > 0) - int(v < 0)
    T = len(x)
    f0 = np.zeros((T, 2), int)
    c0 = c1 = 0
    for t in range(T):
        g1 = sign(f0[t - 1, 0]) if t > 0 else 0
        c0 += sign(x[t])
        c1 += g1
        f0[t] = (c0, c1)
    r0 = np.zeros((T, 2), int)
    c0 = c1 = 0
    for t in range(T - 1, -1, -1):
        g1 = sign(r0[t + 1, 0]) if t < T - 1 else 0
        c0 += -sign(x[t])
        c1 += g1
        r0[t] = (c0, c1)
    f1 = np.zeros((T, 2), int)
    c0 = c1 = 0
    for t in range(T):
        c0 += sign(r0[t, 0])
        c1 += sign(f0[t, 1])
        f1[t] = (c0, c1)
    r1 = np.zeros((T, 2), int)
    c0 = c1 = 0
    for t in range(T - 1, -1, -1):
        g1 = sign(r1[t + 1, 0]) if t < T - 1 else 0
        c0 += -sign(f0[t, 0])
        c1 += g1
        r1[t] = (c0, c1)
    return {"layer0_forward": f0, "layer0_reverse": r0,
            "layer1_forward": f1, "layer1_reverse": r1}


def test_saturated_counter_golden():
    with open(os.path.join(HERE, "golden", "saturated_counter.json")) as fh:
        doc = json.load(fh)
    x = np.array(doc["x"], dtype=np.float64)
    counts = {k: np.array(v) for k, v in doc["counts"].items()}
    derived = _counts_from_rules(x)
    for k in counts:
        assert np.array_equal(counts[k], derived[k]), k
    layers = [{k: np.array(v) for k, v in l.items()} for l in doc["layers"]]
    xin = x.reshape(1, -1, 1)
    y0 = oracle.lstm_stack(xin, layers[:1])[0]
    e0 = np.tanh(np.concatenate([counts["layer0_forward"],
                                 counts["layer0_reverse"]], axis=1))
    np.testing.assert_allclose(y0, e0, rtol=0, atol=1e-14)
    y1 = oracle.lstm_stack(xin, layers)[0]
    e1 = np.tanh(np.concatenate([counts["layer1_forward"],
                                 counts["layer1_reverse"]], axis=1))
    np.testing.assert_allclose(y1, e1, rtol=0, atol=1e-14)


def _torch_lstm(x, layers):
    torch = pytest.importorskip("torch")
    B, T, in0 = x.shape
    H = layers[0]["r"].shape[2]
    L = len(layers)
    m = torch.nn.LSTM(in0, H, num_layers=L, bidirectional=True,
                      batch_first=True, dtype=torch.float64)
    with torch.no_grad():
        for l, lay in enumerate(layers):
            for d, suffix in enumerate(["", "_reverse"]):
                getattr(m, f"weight_ih_l{l}{suffix}").copy_(
                    torch.from_numpy(np.asarray(lay["w"][d], np.float64)))
                getattr(m, f"weight_hh_l{l}{suffix}").copy_(
                    torch.from_numpy(np.asarray(lay["r"][d], np.float64)))
                getattr(m, f"bias_ih_l{l}{suffix}").copy_(
                    torch.from_numpy(np.asarray(lay["b"][d][:4 * H], np.float64)))
                getattr(m, f"bias_hh_l{l}{suffix}").copy_(
                    torch.from_numpy(np.asarray(lay["b"][d][4 * H:], np.float64)))
        y, _ = m(torch.from_numpy(np.asarray(x, np.float64)))
    return y.numpy()


def test_matches_torch_lstm_small():
    rng = np.random.default_rng(15)
    layers = _layers(rng, 16, 6, 4, scale=0.4)
    x = rng.standard_normal((3, 9, 6))
    np.testing.assert_allclose(oracle.lstm_stack(x, layers),
                               _torch_lstm(x, layers), rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", ["b1_t64", "b1_t589"])
def test_matches_torch_lstm_full_width(name):
    # the stack's real shape on the one-window workloads (T = 64 and 589)
    layers = synthetic.stack_weights()
    x = synthetic.stack_input(synthetic.WORKLOADS[name])
    np.testing.assert_allclose(oracle.lstm_stack(x, layers),
                               _torch_lstm(x, layers), rtol=0, atol=1e-12)


@pytest.mark.parametrize("d,k,u,j", [(0, 0, 0, 0), (0, 2, 5, 3), (1, 3, 7, 1),
                                     (1, 1, 2, 4)])
def test_projection_one_hot_column(d, k, u, j):
    rng = np.random.default_rng(16)
    H, inw, M = 8, 5, 7
    X = rng.standard_normal((M, inw))
    W = np.zeros((2, 4 * H, inw))
    W[d, k * H + u, j] = 1.0
    G = oracle.projection(X, W)
    col = d * 4 * H + 4 * u + k
    np.testing.assert_array_equal(G[:, col], X[:, j])
    G[:, col] = 0.0
    assert np.all(G == 0.0)


def test_projection_matches_matmul():
    rng = np.random.default_rng(17)
    H, inw, M = 16, 12, 33
    X = rng.standard_normal((M, inw))
    W = rng.standard_normal((2, 4 * H, inw))
    G = oracle.projection(X, W)
    for d in range(2):
        full = X @ W[d].T  # [M, 4H], source row order
        for k in range(4):
            np.testing.assert_allclose(
                G[:, d * 4 * H + k:(d + 1) * 4 * H:4], full[:, k * H:(k + 1) * H],
                rtol=0, atol=1e-12)


def test_recurrence_of_projection_is_the_layer():
    rng = np.random.default_rng(18)
    H, inw, B, T = 8, 6, 3, 10
    lay = _layers(rng, H, inw, 1)[0]
    x = rng.standard_normal((B, T, inw))
    G = oracle.projection(x.reshape(B * T, inw), lay["w"])
    y = oracle.recurrence(G, lay["r"], lay["b"], B, T)
    np.testing.assert_allclose(y, oracle.lstm_stack(x, [lay]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(y, _torch_lstm(x, [lay]), rtol=0, atol=1e-12)


def test_oracle_threads_positive():
    assert oracle.threads() >= 1


# ---- TF32 projection mode -------------------------------------------------

def _tf32_bits(v):
    """TF32 rounding of float64 values from their bit layout: keep the sign,
    the exponent and the top 10 of the 52 mantissa bits; if the 42 dropped
    bits are at least half of the kept unit, add one kept unit to the
    magnitude (the carry may run into the exponent).  Ties go away from 0."""
    b = np.ascontiguousarray(v, dtype=np.float64).view(np.uint64)
    unit = np.uint64(1) << np.uint64(42)
    low = b & (unit - np.uint64(1))
    kept = b - low
    out = np.where(low >= (unit >> np.uint64(1)), kept + unit, kept)
    return out.view(np.float64)


def test_tf32_rounding_against_bit_definition():
    rng = np.random.default_rng(31)
    # fp32 values over many binades, plus exact ties and values a hair off them
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-60, 60, 20000))).astype(np.float32)
    base = rng.integers(1 << 10, 1 << 11, 500).astype(np.float64)
    ties = np.concatenate([(base + 0.5) * 2.0 ** -10, -(base + 0.5) * 2.0 ** -3,
                           (base + 0.5 - 2.0 ** -20) * 2.0 ** 4, (base + 0.5 + 2.0 ** -20)])
    for vals in (v.astype(np.float64), ties, rng.standard_normal(5000)):
        got = oracle.tf32(vals)
        np.testing.assert_array_equal(got, _tf32_bits(vals))
    # hand cases: 1 + 2^-11 is a tie (away: 1 + 2^-10); 1 + 2^-12 rounds down
    np.testing.assert_array_equal(
        oracle.tf32([1 + 2.0 ** -11, 1 + 2.0 ** -12, -(1 + 2.0 ** -11), 2 - 2.0 ** -12, 0.0]),
        [1 + 2.0 ** -10, 1.0, -(1 + 2.0 ** -10), 2.0, 0.0])


def test_tf32_projection_is_projection_of_rounded_operands():
    rng = np.random.default_rng(32)
    H, inw, M = 8, 20, 17
    X = rng.standard_normal((M, inw)).astype(np.float32).astype(np.float64)
    W = rng.uniform(-0.2, 0.2, (2, 4 * H, inw)).astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(oracle.projection(X, W, tf32=True),
                                  oracle.projection(_tf32_bits(X), _tf32_bits(W)))
    assert np.abs(oracle.projection(X, W, tf32=True) - oracle.projection(X, W)).max() > 1e-6


def test_tf32_stack_is_float64_stack_on_rounded_operands():
    # layer by layer: each layer's TF32 products equal the float64 layer run
    # on its input and W rounded to TF32 (R and the biases untouched)
    rng = np.random.default_rng(33)
    H, in0, B, T = 6, 5, 2, 7
    lays = _layers(rng, H, in0, 3)
    x = rng.standard_normal((B, T, in0))
    cur = x
    for lay in lays:
        rounded = dict(lay, w=_tf32_bits(lay["w"]))
        cur = oracle.lstm_stack(_tf32_bits(cur), [rounded])
    y = oracle.lstm_stack(x, lays, projection="tf32")
    np.testing.assert_array_equal(y, cur)
    assert np.abs(y - oracle.lstm_stack(x, lays)).max() > 1e-6


# ---- dense heads (linear0, linear1, classifier) ----------------------------

def test_heads_zero_weights_closed_form():
    # all weights zero: z = b2, so out = b2 - log(sum(exp(b2))); with b2 = 0
    # every class gets exactly -log 7
    M = 3
    y = np.random.default_rng(40).standard_normal((M, 256))
    z = np.zeros
    out = oracle.heads(y, z((256, 128)), z(128), z((128, 128)), z(128), z((128, 7)), z(7))
    np.testing.assert_array_equal(out, np.full((M, 7), -np.log(7.0)))
    b2 = np.array([0.5, -1.0, 2.0, 0.0, 3.0, -2.5, 1.0])
    out = oracle.heads(y, z((256, 128)), z(128), z((128, 128)), z(128), z((128, 7)), b2)
    np.testing.assert_allclose(out, np.tile(b2 - np.log(np.exp(b2).sum()), (M, 1)),
                               rtol=0, atol=1e-15)


def test_heads_leaky_slope_and_orientation():
    # W0 routes input k to output perm[k] ([k, n] storage), W1 is the identity,
    # W2 picks outputs 0..6: with negative inputs both LeakyReLUs scale by the
    # slope, so z = slope^2 * y[perm^-1[0..6]]
    rng = np.random.default_rng(41)
    slope = 0.2
    perm = rng.permutation(128)
    W0 = np.zeros((256, 128))
    W0[np.arange(128), perm] = 1.0
    W1 = np.eye(128)
    W2 = np.zeros((128, 7))
    W2[np.arange(7), np.arange(7)] = 1.0
    y = -rng.uniform(0.5, 2.0, (4, 256))
    out = oracle.heads(y, W0, np.zeros(128), W1, np.zeros(128), W2, np.zeros(7), slope)
    inv = np.argsort(perm)
    zz = slope * slope * y[:, inv[:7]]
    ref = zz - np.log(np.exp(zz).sum(axis=1, keepdims=True))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-14)


def test_heads_match_torch_and_normalise():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(42)
    M = 9
    y = rng.standard_normal((M, 256))
    W0, b0 = rng.uniform(-0.06, 0.06, (256, 128)), rng.uniform(-0.06, 0.06, 128)
    W1, b1 = rng.uniform(-0.09, 0.09, (128, 128)), rng.uniform(-0.09, 0.09, 128)
    W2, b2 = rng.uniform(-0.09, 0.09, (128, 7)), rng.uniform(-0.09, 0.09, 7)
    out = oracle.heads(y, W0, b0, W1, b1, W2, b2)
    t = lambda a: torch.from_numpy(a)
    h = F.leaky_relu(t(y) @ t(W0) + t(b0), 0.01)
    h = F.leaky_relu(h @ t(W1) + t(b1), 0.01)
    ref = F.log_softmax(h @ t(W2) + t(b2), dim=1).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(np.exp(out).sum(axis=1), 1.0, rtol=0, atol=1e-14)
    # log-softmax is unchanged by a constant added to every logit
    np.testing.assert_allclose(oracle.heads(y, W0, b0, W1, b1, W2, b2 + 3.0), out,
                               rtol=0, atol=1e-13)


# ---- brute force: H = 2, T = 3, input 2, one layer, both directions -------

def _brute_h2_t3(x, W, R, Wb, Rb, reverse):
    """The LSTM written out scalar by scalar for two units: every gate's
    pre-activation spelled out (rows i0 i1 f0 f1 g0 g1 o0 o1), no loop over
    units or gates; the time loop (3 steps) is the only loop."""
    import math

    def sig(v):
        return 1.0 / (1.0 + math.exp(-v))

    h0 = h1 = c0 = c1 = 0.0
    out = {}
    for t in ((2, 1, 0) if reverse else (0, 1, 2)):
        x0, x1 = float(x[t][0]), float(x[t][1])

        def pre(r):
            return (W[r][0] * x0 + W[r][1] * x1 + Wb[r]
                    + R[r][0] * h0 + R[r][1] * h1 + Rb[r])

        i0, i1 = sig(pre(0)), sig(pre(1))
        f0, f1 = sig(pre(2)), sig(pre(3))
        g0, g1 = math.tanh(pre(4)), math.tanh(pre(5))
        o0, o1 = sig(pre(6)), sig(pre(7))
        c0 = f0 * c0 + i0 * g0
        c1 = f1 * c1 + i1 * g1
        h0 = o0 * math.tanh(c0)
        h1 = o1 * math.tanh(c1)
        out[t] = (h0, h1)
    return np.array([out[0], out[1], out[2]])


def test_brute_force_h2_t3_both_directions():
    rng = np.random.default_rng(50)
    lay = {"w": rng.uniform(-0.8, 0.8, (2, 8, 2)), "r": rng.uniform(-0.8, 0.8, (2, 8, 2)),
           "b": rng.uniform(-0.8, 0.8, (2, 16))}
    x = rng.standard_normal((1, 3, 2))
    y = oracle.lstm_stack(x, [lay])
    for d in range(2):
        ref = _brute_h2_t3(x[0], lay["w"][d], lay["r"][d], lay["b"][d][:8], lay["b"][d][8:],
                           reverse=d == 1)
        np.testing.assert_allclose(y[0, :, 2 * d:2 * d + 2], ref, rtol=0, atol=1e-15)
