"""Pins of the oracle's tight packing of mixed-rate keys: each code at its
group's width, the groups' codes concatenated  [Block-GTQ, packed cache].

A hand-worked record (bytes derived bit by bit in the docstring), the record
size the bit budget implies (48 B at 3 bits per coordinate on average, 32 B at
2, against 64 B of nibbles), and round trips against the nibble record of the
same codes."""
import numpy as np
import pytest

from oracle import tq_oracle as O


def _spec(block_bits, tight=True):
    mats = {b: np.eye(cs.size) for b, cs in O.group_layout(block_bits)}
    return O.spec_group_dense(block_bits, mats, tight=tight)


def test_hand_record():
    """d = 8, RoPE blocks of widths (3, 1, 4, 2): record positions are the 1-bit
    group (block 1), the 2-bit group (block 3), then blocks 0 and 2, so the widths
    are 1 1 2 2 3 3 4 4 (20 bits, one 16-byte unit).  Codes 1 0 3 1 5 2 9 15 give
    the bit stream 1 0 | 11 | 10 | 101 | 010 | 1001 | 1111 (each code LSB first):
    bytes 0b01011101 = 0x5D, 0b10010101 = 0x95, 0b00001111 = 0x0F, then zeros."""
    spec = _spec([3, 1, 4, 2])
    np.testing.assert_array_equal(O.code_widths(spec), [1, 1, 2, 2, 3, 3, 4, 4])
    idx = np.array([[1, 0, 3, 1, 5, 2, 9, 15]])
    rec = O.pack(idx, spec)
    assert rec.shape == (1, 16)
    assert rec[0, :3].tolist() == [0x5D, 0x95, 0x0F] and not rec[0, 3:].any()
    np.testing.assert_array_equal(O.unpack(rec, spec, 8), idx)


@pytest.mark.parametrize("avg,nbytes", [(3, 48), (2, 32), (4, 64)])
def test_record_size_follows_the_budget(avg, nbytes):
    """The greedy allocation spends exactly avg * 64 block bits, i.e. avg * 128
    code bits: the tight record is avg * 16 bytes."""
    rng = np.random.default_rng(avg)
    s = rng.lognormal(0, 2, 64)
    bb = O.greedy_bit_alloc(s, 1, 4, avg * 64)
    spec = _spec(bb)
    assert int(O.code_widths(spec).sum()) == avg * 128
    idx = np.stack([rng.integers(0, 1 << O.code_widths(spec)) for _ in range(5)])
    rec = O.pack(idx, spec)
    assert rec.shape == (5, nbytes)
    np.testing.assert_array_equal(O.unpack(rec, spec, 128), idx)
    # the same codes in nibbles: 64 bytes, and the same codes back
    nib = _spec(bb, tight=False)
    assert O.pack(idx, nib).shape == (5, 64)
    np.testing.assert_array_equal(O.unpack(O.pack(idx, nib), nib, 128), O.unpack(rec, spec, 128))


def test_uneven_total_rounds_up():
    """A total that is not a multiple of 128 bits is padded with zero bits to the
    next 16-byte unit."""
    bb = np.array([1] * 63 + [2])          # 130 code bits
    spec = _spec(bb)
    idx = np.ones((2, 128), dtype=np.int64)
    rec = O.pack(idx, spec)
    assert rec.shape == (2, 32)
    bits = np.unpackbits(rec, axis=1, bitorder="little")
    assert bits[:, 130:].sum() == 0
    np.testing.assert_array_equal(O.unpack(rec, spec, 128), idx)
