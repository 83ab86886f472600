"""Ternary codes {-1, 0, 1} ("raw-metal-loop-playbook", ranked-targets table,
BitCPM-8B row: ternary unpack in the same decoder family as int2) are packed
as int2 fields: u = v + 2 in {1, 2, 3}.  Pins: a hand-derived word, the
round trip, and the synthetic generator's range and balance."""
import numpy as np

import oracle
import synth


def test_ternary_word_by_hand():
    # v = -1, 0, 1 repeated -> u = 1, 2, 3 repeated, LSB first, 2 bits each:
    # byte0 = 1 | 2<<2 | 3<<4 | 1<<6 = 0x79, byte1 = 2 | 3<<2 | 1<<4 | 2<<6 = 0x9E,
    # byte2 = 3 | 1<<2 | 2<<4 | 3<<6 = 0xE7, byte3 = 0x79
    v = np.array([[-1, 0, 1] * 5 + [-1]], np.int8)
    w = oracle.pack(v, 2)
    assert w.shape == (1, 1) and int(w[0, 0]) == 0x79E79E79
    assert np.array_equal(oracle.unpack(w, 16, 2), v)


def test_ternary_generator_range_and_round_trip():
    c = synth.ternary_codes(3, "tern", 64, 512).numpy()
    vals, counts = np.unique(c, return_counts=True)
    assert list(vals) == [-1, 0, 1]
    assert counts.min() > 0.3 * c.size
    w = oracle.pack(c, 2)
    assert np.array_equal(oracle.unpack(w, 512, 2), c)
    # no field ever holds u = 0 (the int2 value -2)
    u = (w[..., None] >> (2 * np.arange(16, dtype=np.uint32))) & 3
    assert not np.any(u == 0)
