"""Pins for the oracle's ZipFusion codec: the pages' two worked examples
(exponent 127 in a block of exponents 120..133 gives d = 3 and restores exactly;
code byte 0xD0 with b/2 = 63 gives high bytes 0xBF and 0xC1), the compression
rule at its edges, the 12-bit size, lossless round trips on random and special
bf16 values, and the high-byte identity the register restore rests on."""
import numpy as np
import pytest

from oracle import tq_oracle as O


def bf16(sign, exp, mant):
    return np.uint16((sign << 15) | (exp << 7) | mant)


def _block_with(exps, rng, signs=None):
    """512 bf16 patterns whose exponent fields cycle through `exps`."""
    e = np.resize(np.asarray(exps, dtype=np.int64), O.ZF_BLOCK)
    s = rng.integers(0, 2, O.ZF_BLOCK) if signs is None else np.resize(signs, O.ZF_BLOCK)
    m = rng.integers(0, 128, O.ZF_BLOCK)
    return ((s << 15) | (e << 7) | m).astype(np.uint16)


def test_worked_example_exponent_127():
    rng = np.random.default_rng(0)
    blk = _block_with(range(120, 134), rng)
    blk[5] = bf16(0, 127, 0x35)
    assert O.zf_base(blk) == 120 and O.zf_compressible(blk)
    half, low, codes = O.zf_encode_block(blk)
    assert half == 60
    d = codes[4 * 0 + 1] >> 3 & 7          # value 5 = group 0, k = 5: bits 3-5 of byte 1
    assert d == 3                          # offset 7 = 0b0111: the low bit stays in the low byte
    assert (int(low[5]) >> 7) & 1 == 1
    assert 2 * half + 2 * d + 1 == 127
    np.testing.assert_array_equal(O.zf_decode_block(half, low, codes), blk)


def test_worked_example_code_byte_0xD0():
    assert O.zf_high_bytes(0xD0, 63) == (0xBF, 0xC1)
    # the same through the encoder: value 0 (sign 1, d 0) and value 4 (sign 1, d 2), b = 126
    rng = np.random.default_rng(1)
    blk = _block_with([126, 127, 128, 130], rng, signs=[0])
    blk[0] = bf16(1, 126, 3)
    blk[4] = bf16(1, 130, 9)
    half, low, codes = O.zf_encode_block(blk)
    assert half == 63 and codes[0] == 0xD0
    restored = O.zf_decode_block(half, low, codes)
    assert restored[0] >> 8 == 0xBF and restored[4] >> 8 == 0xC1


@pytest.mark.parametrize("lo,hi,ok", [(120, 135, True), (120, 136, False), (121, 135, True), (121, 136, False),
                                      (0, 15, True), (240, 254, True), (7, 7, True)])
def test_compression_rule(lo, hi, ok):
    """All exponents in [b, b + 15] with b the minimum rounded down to even."""
    rng = np.random.default_rng(2)
    blk = _block_with([lo, hi], rng)
    assert O.zf_base(blk) == lo // 2 * 2
    assert O.zf_compressible(blk) == ok


def test_twelve_bits_per_value():
    rng = np.random.default_rng(3)
    half, low, codes = O.zf_encode_block(_block_with(range(118, 130), rng))
    assert low.nbytes + codes.nbytes == 768 == 0.75 * 2 * O.ZF_BLOCK


def test_lossless_round_trip_random_and_special():
    rng = np.random.default_rng(4)
    for trial in range(20):
        x = rng.standard_normal(O.ZF_BLOCK).astype(np.float32) * np.float32(10.0 ** rng.uniform(-3, 3))
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        if O.zf_compressible(bits):
            np.testing.assert_array_equal(O.zf_decode_block(*O.zf_encode_block(bits)), bits)
    # signed zeros and subnormals (exponent 0), the largest finite exponent
    blk = _block_with([0, 1, 2, 14], rng)
    blk[0], blk[1] = bf16(0, 0, 0), bf16(1, 0, 0)
    np.testing.assert_array_equal(O.zf_decode_block(*O.zf_encode_block(blk)), blk)
    blk = _block_with([240, 254], rng)
    np.testing.assert_array_equal(O.zf_decode_block(*O.zf_encode_block(blk)), blk)


def test_high_byte_identity():
    """High byte = 128 sign + (exponent >> 1) = 128 sign + b/2 + d: the one addition
    of the register restore never carries into the sign (b/2 + d <= 127)."""
    rng = np.random.default_rng(5)
    blk = _block_with(range(200, 215), rng)
    half, low, codes = O.zf_encode_block(blk)
    e = O.zf_exponent(blk)
    for i in range(O.ZF_BLOCK):
        g, k = divmod(i, 8)
        byte = int(codes[4 * g + k % 4])
        d = byte & 7 if k < 4 else (byte >> 3) & 7
        assert half + d == e[i] >> 1 <= 127


@pytest.mark.parametrize("which", ["k", "v"])
def test_page_is_four_blocks_and_round_trips(which):
    """A 16-token page of one head (128 coordinates) is four 512-value blocks (the
    pages: four key blocks per head and page) that partition it; incompressible
    blocks stay raw and the page restores exactly."""
    rng = np.random.default_rng(6)
    page = (rng.standard_normal((16, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    page[12, 3] = bf16(0, 3, 1)                     # one block spans exponents far apart
    blocks = O.zf_page_blocks(page, which)
    assert blocks.shape == (4, 512)
    seen = np.zeros((16, 128), dtype=int)
    for grp in O.zf_block_groups(which):
        for t, d0 in grp:
            seen[t, d0:d0 + 8] += 1
    assert np.all(seen == 1)
    np.testing.assert_array_equal(O.zf_page_unblocks(blocks, which), page)
    assert sum(not O.zf_compressible(b) for b in blocks) == 1
    np.testing.assert_array_equal(O.zf_page_roundtrip(page, which), page)


def test_block_groups_follow_the_lanes():
    """Block q of K holds lane (r, c)'s keys of tokens r and r + 8 at coordinates
    32c + 8q .. +7, next to each other; V block 2e + q lane (r, c)'s values of
    tokens 2c + 8e and 2c + 8e + 1 at coordinates 16r + 8q .. +7."""
    gk, gv = O.zf_block_groups("k"), O.zf_block_groups("v")
    L = 4 * 5 + 3   # lane r = 5, c = 3
    assert gk[2][2 * L] == (5, 32 * 3 + 16) and gk[2][2 * L + 1] == (13, 32 * 3 + 16)
    assert gv[3][2 * L] == (8 + 6, 16 * 5 + 8) and gv[3][2 * L + 1] == (8 + 7, 16 * 5 + 8)
