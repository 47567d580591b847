"""The 16-token tile layout of include/tq.h, as the harness restates it for the
GPU tests: every bit of a tile belongs to exactly one (token, field, bit), every
norm element to one (token, slot); conversions round-trip; each key word and each
value half belongs to one token (so appends never rewrite another token's bits).
CPU only."""
import numpy as np
import pytest

from gpu_harness import CacheLayout, norm_positions, tile_bit_map


@pytest.mark.parametrize("which", ["k", "v"])
@pytest.mark.parametrize("bits", [3, 4])
def test_bit_map_is_a_bijection(which, bits):
    M = tile_bit_map(which, bits)
    nb = 48 if bits == 3 else 64
    assert np.array_equal(np.sort(M.ravel()), np.arange(16 * nb * 8))


@pytest.mark.parametrize("which", ["k", "v"])
@pytest.mark.parametrize("bits", [3, 4])
def test_token_ownership_of_words(which, bits):
    """Key words (32 bits) and value halves (16 bits) hold bits of one token only."""
    M = tile_bit_map(which, bits)
    unit = 32 if which == "k" else 16
    owner = {}
    for t in range(16):
        for u in np.unique(M[t] // unit):
            assert owner.setdefault(int(u), t) == t


def test_key_slots_of_lane_zero():
    """Spot values from the header's text: token 0, lane 0 (r = 0, c = 0): field
    s = 0 (pair 0) is byte 0 of word 0; field 2 (pair 8) byte 2; field 4 (pair 16)
    sits in word 1 (bits 0-1 of the field at byte bits 0-1, bits 2-5 at 4-7); field
    12 (pair 48) is spread over bits 6-7 / 2-3 / 6-7 of byte 0 of words 0, 1, 2;
    token 8 starts at word 3 (byte 12 of lane 0); lane 1 starts at byte 16."""
    M = tile_bit_map("k", 3)
    assert list(M[0, 0]) == list(range(6))
    assert list(M[0, 8]) == [16 + k for k in range(6)]
    assert list(M[0, 16]) == [32, 33, 36, 37, 38, 39]
    assert list(M[0, 48]) == [6, 7, 34, 35, 70, 71]
    assert M[8, 0, 0] == 8 * 12
    assert M[0, 1, 0] == 8 * 16     # pair 1: lane column c = 1 -> lane 1
    M4 = tile_bit_map("k", 4)
    assert list(M4[8, 0]) == [8 * (512 + 0) + k for k in range(8)]   # token 8, word 4 of lane 0
    V = tile_bit_map("v", 3)
    assert list(V[0, 0]) == list(range(6))                    # token 0 = low half of lane 0's word 0
    assert list(V[1, 0]) == [16 + k for k in range(6)]        # token 1 = high half
    assert V[2, 0, 0] == 8 * 16                               # token 2: lane column c = 1


@pytest.mark.parametrize("which,slots", [("k", 1), ("v", 1), ("k", 4), ("v", 4)])
def test_norm_positions_are_a_permutation(which, slots):
    P = norm_positions(which, slots)
    assert np.array_equal(np.sort(P.ravel()), np.arange(16 * slots))


class _Desc:
    def __init__(self, bits, slots, t_alloc, k_mixed=0):
        self.layout = 1
        self.k_mixed = k_mixed
        self.t_alloc = t_alloc
        self.k_code_bytes = self.v_code_bytes = 48 if bits == 3 else 64
        self.k_norm_slots = self.v_norm_slots = slots


@pytest.mark.parametrize("bits,slots", [(3, 1), (4, 4), (3, 4)])
def test_round_trip(bits, slots):
    rng = np.random.default_rng(3)
    lay = CacheLayout(_Desc(bits, slots, 48))
    nb = 48 if bits == 3 else 64
    for which in ("k", "v"):
        rec = rng.integers(0, 256, size=(48, nb), dtype=np.uint8)
        raw = lay.raw(rec, which)
        assert raw.shape == (48 * nb,)
        assert np.array_equal(lay.records(raw, which), rec)
        nrm = rng.standard_normal((48, slots)).astype(np.float16)
        assert np.array_equal(lay.norms(lay.raw_norms(nrm, which), which), nrm)


class _Seg:
    def __init__(self, start, length, bits):
        self.start, self.length, self.bits = start, length, bits


class _Spec:
    def __init__(self, segs):
        self.segments = segs


def test_mixed_key_offsets():
    """Mixed-rate keys in the tile layout: a b-bit code c (b < 4) is stored as
    c + 2^b, so every stored nibble of a 1..3-bit group lies in [2^b, 2^(b+1))
    and names its group; 4-bit codes are stored as they are."""
    rng = np.random.default_rng(5)
    segs = [_Seg(0, 10, 1), _Seg(10, 30, 2), _Seg(40, 50, 3), _Seg(90, 38, 4)]
    spec = _Spec(segs)
    width = np.zeros(128, dtype=np.int64)
    for sg in segs:
        width[sg.start:sg.start + sg.length] = sg.bits
    codes = rng.integers(0, 1 << width, size=(48, 128)).astype(np.uint8)   # [T][d] codes of each width
    rec = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)        # nibble records
    mixed = CacheLayout(_Desc(4, 4, 48, k_mixed=1))
    raw = mixed.raw(rec, "k", spec)
    assert np.array_equal(mixed.records(raw, "k", spec), rec)
    stored = CacheLayout(_Desc(4, 4, 48)).records(raw, "k")                 # the nibbles as stored
    nib = np.stack([stored & 15, stored >> 4], axis=2).reshape(48, 128).astype(np.int64)
    lo_b = np.where(width < 4, 1 << width, 0)
    hi_b = np.where(width < 4, 2 << width, 16)
    assert np.all((nib >= lo_b) & (nib < hi_b))
    assert np.array_equal(nib - lo_b, codes.astype(np.int64))
    # values are not offset; a never-written (zero) row reads back as zero
    assert np.array_equal(mixed.records(mixed.raw(rec, "v", spec), "v", spec), rec)
    assert not mixed.records(np.zeros(48 * 64, dtype=np.uint8), "k", spec).any()
