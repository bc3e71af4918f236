"""Parity of the cluster recurrence (through the C ABI) with the float64
oracle's recurrence, given the same fp32 projection; and bitwise identity of
every kernel variant."""
import numpy as np
import pytest

import oracle
from bidirectional_lstm_stack_gb300 import binding, synthetic
from gpu_util import assert_within, cuda

pytestmark = pytest.mark.gpu

VARIANTS = [(16, 1, 1, 0), (16, 2, 1, 0), (16, 4, 1, 0), (16, 8, 1, 0), (8, 1, 1, 0),
            (8, 2, 1, 0), (8, 4, 1, 0), (8, 8, 1, 0), (4, 1, 1, 0), (4, 2, 1, 0), (2, 1, 1, 0),
            (4, 1, 2, 0), (4, 1, 4, 0), (4, 1, 8, 0), (4, 2, 2, 0), (4, 2, 4, 0), (4, 2, 8, 0),
            (8, 2, 4, 0), (8, 1, 1, 128), (8, 2, 1, 128), (16, 1, 1, 64), (16, 2, 1, 64),
            (4, 4, 1, 0), (4, 4, 2, 0), (4, 4, 4, 0), (4, 8, 1, 0), (4, 8, 2, 0),
            (8, 4, 1, 128), (8, 8, 1, 128), (8, 1, 1, 64), (8, 4, 1, 64), (8, 4, 2, 64),
            (4, 4, 1, 128), (4, 4, 2, 128), (8, 8, 1, 64), (4, 8, 1, 128), (8, 8, 2, 64),
            (8, 2, 1, 64), (8, 2, 2, 64), (4, 2, 1, 128), (4, 2, 2, 128), (4, 1, 1, 128),
            (2, 4, 2, 256), (2, 4, 1, 256)]
# two hidden units per 8-lane group: (cluster, threads) of these variants
TWO_UNIT = {(8, 64), (4, 128), (2, 256)}


def _layer_inputs(batch, steps, layer_index=0, seed=21, scale=1.0):
    layers = synthetic.stack_weights()
    lay = layers[layer_index]
    inw = lay["w"].shape[2]
    x = synthetic.random_matrix(seed, (batch * steps, inw), scale=scale)
    G = oracle.projection(x, lay["w"]).astype(np.float32)
    _, _, rp, bias = binding.lstm_pack_layer(lay["w"], lay["r"], lay["b"], inw,
                                            64 if inw == 60 else 256)
    return lay, G, rp, bias


def _run(G, rp, bias, batch, steps, variant=None):
    import torch
    g = cuda(G)
    rpt, bt = cuda(rp), cuda(bias)
    y = torch.full((batch, steps, 256), float("nan"), device="cuda")
    for d in range(2):
        if variant is None:
            binding.lstm_recurrence(g, rpt[d], bt[d], y, batch, steps, d)
        else:
            binding.lstm_recurrence_variant(g, rpt[d], bt[d], y, batch, steps, d, *variant)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("batch,steps", [(1, 1), (1, 2), (1, 64), (3, 37), (5, 100), (9, 20),
                                         (33, 12)])
def test_recurrence_matches_oracle(batch, steps):
    lay, G, rp, bias = _layer_inputs(batch, steps)
    y = _run(G, rp, bias, batch, steps)
    ref = oracle.recurrence(G.astype(np.float64), lay["r"], lay["b"], batch, steps)
    assert_within(y, ref, what=f"recurrence b{batch} t{steps}")
    assert binding.lstm_fault_status() == 0


def test_recurrence_saturated_gates():
    # large projections drive the gates into saturation (the x3 workload's regime)
    lay, G, rp, bias = _layer_inputs(4, 50, layer_index=1, scale=6.0)
    y = _run(G, rp, bias, 4, 50)
    ref = oracle.recurrence(G.astype(np.float64), lay["r"], lay["b"], 4, 50)
    assert_within(y, ref, what="recurrence saturated")


@pytest.mark.parametrize("variant", VARIANTS)
def test_every_variant_matches_oracle(variant):
    batch, steps = 13, 29
    lay, G, rp, bias = _layer_inputs(batch, steps, seed=22)
    y = _run(G, rp, bias, batch, steps, variant)
    ref = oracle.recurrence(G.astype(np.float64), lay["r"], lay["b"], batch, steps)
    assert_within(y, ref, what=f"variant {variant}")


@pytest.mark.parametrize("steps", [3, 4, 5, 6, 7, 8, 9, 10, 11])
@pytest.mark.parametrize("variant", [(8, 1, 1, 128), (4, 2, 4, 0), (4, 4, 4, 0), (4, 8, 2, 0),
                                     (8, 1, 1, 64), (4, 1, 1, 128), (4, 4, 1, 128),
                                     (4, 4, 2, 128), (8, 2, 1, 64), (8, 2, 2, 64)])
def test_every_tail_length(variant, steps):
    # the step loop runs groups of 4 steps (2 with four or more chunks per
    # lane) and checks for the sequence end only in the last two groups:
    # every remainder and every count of full groups before the tail
    batch = 6
    lay, G, rp, bias = _layer_inputs(batch, steps, seed=24)
    y = _run(G, rp, bias, batch, steps, variant)
    ref = oracle.recurrence(G.astype(np.float64), lay["r"], lay["b"], batch, steps)
    assert_within(y, ref, what=f"variant {variant} T={steps}")
    assert binding.lstm_fault_status() == 0


@pytest.mark.parametrize("batch", [1, 4, 5, 9, 17, 23])
@pytest.mark.parametrize("variant", [(4, 4, 2, 0), (4, 4, 4, 0), (4, 8, 2, 0), (8, 4, 1, 128),
                                     (4, 4, 2, 128), (8, 4, 2, 64), (4, 8, 1, 128),
                                     (8, 2, 2, 64), (4, 2, 2, 128), (2, 4, 2, 256)])
def test_partly_and_wholly_empty_chunks(variant, batch):
    # tiles whose last chunks hold no window of the batch (those chunks have
    # no barrier traffic at all in the chunk-major variants)
    steps = 13
    lay, G, rp, bias = _layer_inputs(batch, steps, seed=25)
    y = _run(G, rp, bias, batch, steps, variant)
    ref = oracle.recurrence(G.astype(np.float64), lay["r"], lay["b"], batch, steps)
    assert_within(y, ref, what=f"variant {variant} B={batch}")
    assert binding.lstm_fault_status() == 0


# tensor cores (tcgen05, 3xTF32, A in tensor memory): clusters of 4 CTAs of
# 128 threads, 16 windows per cluster; another summation order than the FFMA
# variants, so compared with the oracle only
TC_VARIANT = (4, 16, 1, 128)


@pytest.mark.parametrize("batch,steps", [(1, 1), (1, 2), (3, 5), (16, 7), (17, 33), (40, 64),
                                         (33, 3)])
def test_tensor_core_variant_matches_oracle(batch, steps):
    import torch
    lay, G, rp, bias = _layer_inputs(batch, steps, seed=26)
    ref = oracle.recurrence(G.astype(np.float64), lay["r"], lay["b"], batch, steps)
    apart = _run(G, rp, bias, batch, steps, TC_VARIANT)
    assert_within(apart, ref, what=f"tensor cores b{batch} t{steps}, directions apart")
    y = torch.full((batch, steps, 256), float("nan"), device="cuda")
    binding.lstm_recurrence_variant(cuda(G), cuda(rp), cuda(bias), y, batch, steps,
                                    binding.LSTM_BOTH_DIRECTIONS, *TC_VARIANT)
    torch.cuda.synchronize()
    assert_within(y.cpu().numpy(), ref, what=f"tensor cores b{batch} t{steps}, one launch")
    assert binding.lstm_fault_status() == 0


def test_tensor_core_variant_large_inputs():
    # inputs 30x larger: saturated gates, the TF32 lo parts carrying the
    # products' low bits
    batch, steps = 21, 19
    lay, G, rp, bias = _layer_inputs(batch, steps, seed=27, scale=30.0)
    y = _run(G, rp, bias, batch, steps, TC_VARIANT)
    ref = oracle.recurrence(G.astype(np.float64), lay["r"], lay["b"], batch, steps)
    assert_within(y, ref, what="tensor cores, large inputs")


def test_variants_are_bitwise_identical():
    batch, steps = 37, 41
    _, G, rp, bias = _layer_inputs(batch, steps, seed=23)
    outs = [_run(G, rp, bias, batch, steps, v) for v in VARIANTS]
    outs.append(_run(G, rp, bias, batch, steps, None))
    for v, o in zip(VARIANTS + [None], outs):
        assert np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)), v


@pytest.mark.parametrize("batch,steps", [(1, 37), (5, 40), (33, 11), (130, 9)])
def test_both_directions_in_one_launch(batch, steps):
    # the stack's launch: forward and reverse clusters alternate in one grid;
    # bitwise equal to the two directions launched one by one
    import torch
    lay, G, rp, bias = _layer_inputs(batch, steps, layer_index=1, seed=batch + steps)
    one_by_one = _run(G, rp, bias, batch, steps)
    g, rpt, bt = cuda(G), cuda(rp), cuda(bias)
    y = torch.full((batch, steps, 256), float("nan"), device="cuda")
    binding.lstm_recurrence(g, rpt, bt, y, batch, steps, binding.LSTM_BOTH_DIRECTIONS)
    torch.cuda.synchronize()
    both = y.cpu().numpy()
    assert np.array_equal(both.view(np.uint32), one_by_one.view(np.uint32))
    assert binding.lstm_fault_status() == 0


def test_unknown_variant_is_rejected():
    import torch
    g = torch.zeros((4, 1024), device="cuda")
    rp = torch.zeros((512, 128), device="cuda")
    b = torch.zeros(512, device="cuda")
    y = torch.zeros((1, 4, 256), device="cuda")
    with pytest.raises(binding.LSTMError) as e:
        binding.lstm_recurrence_variant(g, rp, b, y, 1, 4, 0, 3, 1, 1, 0)
    assert e.value.code == binding.LSTM_E_INVALID


@pytest.mark.parametrize("variant,batch", [((8, 1, 1, 128), 7), ((4, 1, 1, 128), 37),
                                           ((4, 2, 1, 128), 74), ((4, 4, 1, 128), 148),
                                           ((4, 4, 2, 128), 264), ((8, 4, 1, 128), 100),
                                           ((2, 4, 1, 256), 152), ((2, 4, 2, 256), 304)])
def test_chosen_variants_run_in_one_wave(variant, batch):
    # the batch sizes each variant is chosen for fit on the GPU at once, both
    # directions together (more registers or shared memory per CTA would
    # silently split them into two waves)
    c, nw, nch, threads = variant
    if (c, threads) in TWO_UNIT:
        tile = nw * nch
    else:
        tile = ((threads or 256) // 8) // (128 // c) * nw * nch
    need = 2 * -(-batch // tile)
    assert binding.lstm_recurrence_max_clusters(*variant) >= need, (variant, need)


def test_max_clusters_query():
    for v in VARIANTS + [TC_VARIANT]:
        n = binding.lstm_recurrence_max_clusters(*v)
        assert n >= 1, (v, n)
    with pytest.raises(binding.LSTMError):
        binding.lstm_recurrence_max_clusters(3, 1, 1, 0)
