"""Pins of the seeded input generator that both sides draw their inputs from.

The generator holds none of the method's arithmetic. These tests check that it
follows its published definitions and draws the stated input recipe:

* SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): the first three outputs from
  state 0 are the algorithm's published reference sequence.
* FNV-1a 64 (the stream-name hash): the published test vectors.
* The int64 tensor form (wrapping multiplies, logical shifts) equals the
  Python-integer form, for counters up to 2^62.
* The recipe: codes are uniform over all 2^b values, scales lie in
  [0.005, 0.02], activations are N(0, 1), gamma is N(1, 0.1), and the
  outliers are +-50 on about 1 element in 1000.
* Row samples equal the same rows of the full matrix, so sampled parity
  checks see the real inputs.
"""
import numpy as np
import pytest
import torch

import synth

SEED = synth.DEFAULT_SEED


def test_splitmix64_reference_sequence():
    # state 0, then three steps of gamma 0x9E3779B97F4A7C15
    assert [synth.draw_int(0, i) for i in range(3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_fnv1a64_vectors():
    assert synth.fnv1a64(b"") == 0xCBF29CE484222325
    assert synth.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert synth.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_tensor_form_equals_integer_form():
    idx = [0, 1, 2, 31, 12345, (1 << 31) + 3, (1 << 40) + 7, 1 << 62]
    for key in (0, 1, synth.stream_key(SEED, "w.codes"), (1 << 63) + 5, synth.MASK64):
        got = synth.draws(key, torch.tensor(idx, dtype=torch.int64)).numpy().view(np.uint64)
        assert [int(v) for v in got] == [synth.draw_int(key, i) for i in idx]


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codes_uniform_over_all_values(bits):
    c = synth.codes(SEED, f"uni{bits}", 64, 4096, bits).numpy().astype(np.int64)
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    assert c.min() == lo and c.max() == hi
    counts = np.bincount((c - lo).ravel(), minlength=1 << bits)
    n, p = c.size, 1.0 / (1 << bits)
    sigma = np.sqrt(n * p * (1 - p))
    assert np.all(np.abs(counts - n * p) < 5 * sigma)


def test_scales_range_and_spread():
    s = synth.scales(SEED, "sc", 512, 64).numpy().astype(np.float64)
    assert s.min() >= np.float16(0.005) and s.max() <= np.float16(0.02)
    assert abs(s.mean() - 0.0125) < 2e-4
    # uniform on [0.005, 0.02]: standard deviation 0.015 / sqrt(12)
    assert abs(s.std() - 0.015 / np.sqrt(12)) < 2e-4


def test_activation_and_gamma_distributions():
    x = synth.normal_f16(SEED, "act", (1 << 18,)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    g = synth.normal_f16(SEED, "gam", (1 << 18,), mean=1.0, std=0.1).astype(np.float64)
    assert abs(g.mean() - 1.0) < 0.002 and abs(g.std() - 0.1) < 0.002


def test_outliers():
    n = 1 << 20
    v = synth.normal_f16(SEED, "out", (n,), outlier_every=1000).astype(np.float64)
    hit = np.abs(v) == 50.0
    p = 1.0 / 1000
    assert abs(hit.sum() - n * p) < 5 * np.sqrt(n * p)
    assert (v[hit] > 0).any() and (v[hit] < 0).any()
    # the same stream without outliers differs only at the hits
    w = synth.normal_f16(SEED, "out", (n,)).astype(np.float64)
    assert np.array_equal(v[~hit], w[~hit])


def test_row_samples_equal_full_rows():
    rows = np.array([0, 5, 63, 17])
    full = synth.codes(SEED, "rows", 64, 512, 2)
    assert torch.equal(synth.codes(SEED, "rows", 64, 512, 2, rows=rows), full[rows])
    fs = synth.scales(SEED, "rows", 64, 16)
    assert torch.equal(synth.scales(SEED, "rows", 64, 16, rows=rows).view(torch.int16),
                       fs[rows].view(torch.int16))
    ft = synth.ternary_codes(SEED, "rows", 64, 512)
    assert torch.equal(synth.ternary_codes(SEED, "rows", 64, 512, rows=rows), ft[rows])
    # chunking the draw changes nothing
    assert torch.equal(synth.codes(SEED, "rows", 64, 512, 2, chunk_elems=1000), full)


def test_streams_are_deterministic_and_distinct():
    a = synth.codes(SEED, "det", 8, 256, 4)
    assert torch.equal(a, synth.codes(SEED, "det", 8, 256, 4))
    assert not torch.equal(a, synth.codes(SEED, "det2", 8, 256, 4))
    assert not torch.equal(a, synth.codes(SEED + 1, "det", 8, 256, 4))
