"""The shared input generator follows its published definitions."""
import numpy as np

import synth


def test_splitmix64_reference_vector():
    # splitmix64 from state 0: the first output is 0xE220A8397B1DCDAF
    assert int(synth._mix(np.uint64(0) + synth._G)) == 0xE220A8397B1DCDAF


def test_counter_based_and_chunk_independent():
    a = synth.normal(3, 2, 1, 1001)
    b = synth.normal(3, 2, 1, 1001, chunk=7)
    assert np.array_equal(a, b)
    assert np.array_equal(synth.uniform(3, 2, 1, 10, offset=5), synth.uniform(3, 2, 1, 15)[5:])
    assert not np.array_equal(synth.normal(3, 2, 2, 10), synth.normal(3, 2, 1, 10))


def test_normal_moments():
    x = synth.normal(0, 0, 1, 400000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_bf16_round_to_nearest_even():
    v = np.array([1.0, 1.00390625, 1.01171875, -2.5, 0.0])
    assert list(synth.to_bf16_bits(v)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0]
    back = synth.bf16_bits_to_f32(synth.to_bf16_bits(v))
    assert list(back) == [1.0, 1.0, 1.0078125 + 0.0078125, -2.5, 0.0]


def test_gate_rows_scaled_per_neuron():
    wg, wu, wd = synth.layer_weights(0, 0, 64, 512, sigma=1.0)
    assert wg.shape == (512, 64) and wu.shape == (512, 64) and wd.shape == (64, 512)
    rs = synth.bf16_bits_to_f32(wg).std(axis=1)
    us = synth.bf16_bits_to_f32(wu).std(axis=1)
    # per-row spread of a LogNormal(0,1) scale is far wider than the up rows'
    assert np.log(rs).std() > 0.8 and np.log(us).std() < 0.2
