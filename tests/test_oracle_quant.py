"""Pins of the oracle's grouped affine weight quantization (8 and 4 bits, groups of 64):
exact reconstruction on grid-aligned weights, the hand-computed codes of one group, code range
and the round-trip error bound, the zero-range group, and the dequantized provider. No GPU."""

import numpy as np
import pytest

import oracle
from oracle import quant


def _bf16(x):
    f = np.asarray(x, np.float32)
    u = f.view(np.uint32)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even
    return r


def test_grid_aligned_weights_reconstruct_exactly():
    # min 0, max 15/128: scale 1/128 exactly in fp16, codes = w * 128
    q = np.arange(64) % 16
    w = _bf16(q / 128.0).reshape(1, 64)
    codes, s, b = quant.quantize(w, 4)
    np.testing.assert_array_equal(codes[0], q)
    assert s[0, 0] == np.float16(1 / 128) and b[0, 0] == 0
    np.testing.assert_array_equal(quant.dequantize(codes, s, b)[0], q / 128.0)


def test_hand_computed_group():
    # values -0.5 .. 0.25 in steps of 0.75/255 rounded: 8-bit codes of the endpoints are 0, 255
    w = np.zeros(64)
    w[0], w[1], w[2] = -0.5, 0.25, 0.0
    codes, s, b = quant.quantize(_bf16(w).reshape(1, 64), 8)
    assert b[0, 0] == np.float16(-0.5)
    assert s[0, 0] == np.float16(np.float32(0.75) / np.float32(255))
    sc = np.float32(s[0, 0])
    assert codes[0, 0] == 0 and codes[0, 1] == 255
    assert codes[0, 2] == int(np.rint(np.float32(0.5) / sc))


@pytest.mark.parametrize("nbits", [8, 4])
def test_codes_in_range_and_round_trip_bound(nbits):
    rng = np.random.default_rng(nbits)
    w = _bf16(rng.normal(0, 0.02, (6, 256)))
    codes, s, b = quant.quantize(w, nbits)
    assert codes.max() <= 2 ** nbits - 1
    wf = quant._bf16_to_f32(w).astype(np.float64)
    deq = quant.dequantize(codes, s, b)
    # half a step, plus the fp16 rounding of the bias and of the step times the top code
    step = np.repeat(s.astype(np.float64), 64, axis=1)
    slack = np.repeat(np.abs(b.astype(np.float64)), 64, axis=1) * 2.0 ** -11 + step * (2 ** nbits) * 2.0 ** -11
    assert np.all(np.abs(deq - wf) <= step / 2 + slack + 1e-12)
    # every group uses both ends of its range
    g = codes.reshape(6, 4, 64)
    assert np.all(g.min(axis=2) == 0)
    assert np.all(g.max(axis=2) >= 2 ** nbits - 2)


def test_zero_range_group():
    w = _bf16(np.full((1, 64), 0.125))
    codes, s, b = quant.quantize(w, 4)
    assert s[0, 0] == 0 and np.all(codes == 0)
    np.testing.assert_array_equal(quant.dequantize(codes, s, b), np.full((1, 64), 0.125))


def test_quantized_provider_feeds_the_model():
    import dataclasses
    import synth
    shape = dataclasses.replace(synth.TINY, inter=128)  # every input width a multiple of 64
    w = synth.Weights(shape, seed=3)
    qw = quant.QuantizedWeights(w, 4)
    m = oracle.Model(qw)
    lw = m.layer(0)
    codes, s, b = quant.quantize(w.layer(0)["self_attn.q_proj.weight"], 4)
    np.testing.assert_array_equal(lw.wq, quant.dequantize(codes, s, b))
    np.testing.assert_array_equal(lw.in_norm, m.layer(0).in_norm)
    out = oracle.forward(m, [1, 2, 3], oracle.SeqCache(shape.n_layers))
    assert np.all(np.isfinite(out["logits"]))


def test_halfway_values_round_to_even_code():
    # min 0, max 15/128 (scale 1/128): w = k.5/128 lies exactly between codes k and k + 1, and
    # rint sends it to the even one (round half up would give 1, 2, 3, 4 here)
    w = np.zeros(64)
    w[1] = 15 / 128
    w[2:6] = np.array([0.5, 1.5, 2.5, 3.5]) / 128
    codes, s, b = quant.quantize(_bf16(w).reshape(1, 64), 4)
    assert s[0, 0] == np.float16(1 / 128) and b[0, 0] == 0
    assert codes[0, 2:6].tolist() == [0, 2, 2, 4]


def test_eight_bits_finer_than_four():
    rng = np.random.default_rng(7)
    w = _bf16(rng.normal(0, 0.02, (4, 128)))
    wf = quant._bf16_to_f32(w).astype(np.float64)
    err = {n: np.abs(quant.dequantize(*quant.quantize(w, n)) - wf).max() for n in (4, 8)}
    # 255 levels instead of 15 over the same range: the step is 17x finer
    assert err[8] < err[4] / 8
