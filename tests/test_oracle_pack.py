"""Oracle pins: packer and decoder.

Hand-decoded words from tests/golden/packed_words.txt (each with its
citation), field-level invariants, and range checks.
"""
import os

import numpy as np
import pytest


def _golden(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "packed_words.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            bits, codes, word = line.split()
            rows.append((int(bits), [int(c) for c in codes.split(",")], int(word, 16)))
    return rows


def test_golden_words(orc, golden_dir):
    rows = _golden(golden_dir)
    assert len(rows) >= 8
    for bits, codes, word in rows:
        assert len(codes) == 32 // bits
        got = orc.pack(np.array([codes], np.int8), bits)
        assert got.shape == (1, 1) and int(got[0, 0]) == word, (bits, codes, hex(int(got[0, 0])))
        back = orc.unpack(np.array([[word]], np.uint32), len(codes), bits)
        assert back[0].tolist() == codes


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_roundtrip_random(orc, bits):
    rng = np.random.default_rng(bits)
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1))
    codes = rng.integers(lo, hi, size=(37, 256), dtype=np.int64).astype(np.int8)
    words = orc.pack(codes, bits)
    assert words.shape == (37, 256 * bits // 32)
    assert np.array_equal(orc.unpack(words, 256, bits), codes)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_unpack_every_word_byte(orc, bits):
    # every byte value at every byte position decodes, and re-packs, to itself
    per_byte = 8 // bits
    vals = np.arange(256, dtype=np.uint32)
    for pos in range(4):
        words = (vals << (8 * pos)).reshape(-1, 1)
        codes = orc.unpack(words, 32 // bits, bits)
        assert np.array_equal(orc.pack(codes, bits), words)
        # the byte at `pos` holds codes pos*per_byte .. +per_byte-1, low field first
        for q in range(per_byte):
            u = (vals >> (bits * q)) & ((1 << bits) - 1)
            assert np.array_equal(codes[:, pos * per_byte + q].astype(np.int64),
                                  u.astype(np.int64) - (1 << (bits - 1)))


def test_int2_every_half_word(orc):
    # all 2^16 patterns of either 16-bit half of an int2 word: eight codes,
    # code j of the half at bits 2j..2j+1, value field - 2
    pat = np.arange(1 << 16, dtype=np.uint32)
    j = np.arange(8, dtype=np.uint32)
    want = ((pat[:, None] >> (2 * j)) & 3).astype(np.int64) - 2
    for half in (0, 1):
        words = (pat << (16 * half)).reshape(-1, 1)
        codes = orc.unpack(words, 16, 2).astype(np.int64)
        assert np.array_equal(codes[:, 8 * half:8 * half + 8], want)
        assert np.all(codes[:, 8 * (1 - half):8 * (1 - half) + 8] == -2)
        assert np.array_equal(orc.pack(codes.astype(np.int8), 2), words)


def test_int2_values_are_minus2_to_1(orc):
    codes = orc.unpack(np.array([[0xE4E4E4E4]], np.uint32), 16, 2)
    assert sorted(set(codes[0].tolist())) == [-2, -1, 0, 1]


@pytest.mark.parametrize("bits,bad", [(2, 2), (2, -3), (4, 8), (4, -9)])
def test_out_of_range_rejected(orc, bits, bad):
    codes = np.zeros((1, 32 // bits), np.int8)
    codes[0, 1] = bad
    with pytest.raises(ValueError):
        orc.pack(codes, bits)
