"""Pins for the oracle's rotations, quantiser and packer: an independent
library Hadamard, Hamilton's rules, the SO(3) special case printed on the
RotaryQuant page, hand-derived records, and the sizes the pages print."""
import math

import numpy as np
import pytest
import scipy.linalg

from conftest import read_golden_kv
from oracle import tq_oracle as O


@pytest.mark.parametrize("n", [1, 2, 4, 32, 128])
def test_hadamard_matches_scipy(n):
    np.testing.assert_allclose(O.hadamard(n), scipy.linalg.hadamard(n) / math.sqrt(n), atol=1e-15)


def test_hadamard_properties():
    H = O.hadamard(128)
    np.testing.assert_allclose(H @ H.T, np.eye(128), atol=1e-13)
    np.testing.assert_allclose(H, H.T, atol=0)
    np.testing.assert_allclose(H @ H, np.eye(128), atol=1e-13)
    np.testing.assert_allclose(H[:, 0], np.full(128, 1 / math.sqrt(128)), atol=1e-15)


def test_hamilton_rules():
    one, i, j, k = np.eye(4)
    np.testing.assert_allclose(O.quat_mul(i, i), -one)
    np.testing.assert_allclose(O.quat_mul(j, j), -one)
    np.testing.assert_allclose(O.quat_mul(k, k), -one)
    np.testing.assert_allclose(O.quat_mul(i, j), k)
    np.testing.assert_allclose(O.quat_mul(j, k), i)
    np.testing.assert_allclose(O.quat_mul(k, i), j)
    np.testing.assert_allclose(O.quat_mul(j, i), -k)


def _left(q):
    # textbook matrix of v -> q v
    w, x, y, z = q
    return np.array([[w, -x, -y, -z], [x, w, -z, y], [y, z, w, -x], [z, -y, x, w]])


def _right(q):
    # textbook matrix of v -> v q
    w, x, y, z = q
    return np.array([[w, -x, -y, -z], [x, w, z, -y], [y, -z, w, x], [z, y, -x, w]])


def test_so4_block_against_textbook_matrices():
    rng = np.random.default_rng(3)
    for _ in range(20):
        qL = rng.standard_normal(4)
        qL /= np.linalg.norm(qL)
        qR = rng.standard_normal(4)
        qR /= np.linalg.norm(qR)
        M = O.so4_block_matrix(qL, qR)
        qRc = np.array([qR[0], -qR[1], -qR[2], -qR[3]])
        np.testing.assert_allclose(M, _left(qL) @ _right(qRc), atol=1e-14)
        np.testing.assert_allclose(M @ M.T, np.eye(4), atol=1e-14)
        assert abs(np.linalg.det(M) - 1.0) < 1e-12


def test_so3_special_case_fixes_real_axis():
    # [RotaryQuant] Key design 2 / ablation: a single-quaternion conjugation
    # v -> q v conj(q) (q_L = q_R) leaves the real axis fixed, so 1 of 4 dims
    # is not rotated.
    rng = np.random.default_rng(5)
    q = rng.standard_normal(4)
    q /= np.linalg.norm(q)
    M = O.so4_block_matrix(q, q)
    np.testing.assert_allclose(M[:, 0], [1, 0, 0, 0], atol=1e-14)
    np.testing.assert_allclose(M[0, :], [1, 0, 0, 0], atol=1e-14)
    np.testing.assert_allclose(O.so4_block_matrix(np.array([1., 0, 0, 0]), np.array([1., 0, 0, 0])), np.eye(4))


def test_page_op_and_parameter_counts():
    p = {k: float(v[0]) for k, v in read_golden_kv("pages_numbers.txt").items()}
    d = 128
    assert d * math.log2(d) == p["wht_fma_128"]
    assert (d // 4) * 16 == p["so4_fma_128"]
    assert p["wht_fma_128"] + p["so4_fma_128"] == p["total_fma_128"]
    assert d * d == p["dense_params"]
    assert round(p["dense_params"] / p["total_fma_128"], 1) == p["dense_over_total"]
    quats = np.zeros((d // 4, 2, 4))
    assert quats.size == p["so4_params_per_head"]
    assert p["dense_params"] / p["so4_params_per_head"] == p["params_ratio"]


def _all_specs(rng, bits=3):
    d = 128
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    g = rng.standard_normal((32, 2, 4))
    quats = g / np.linalg.norm(g, axis=-1, keepdims=True)
    block_bits = rng.integers(1, 5, size=64)
    mats = {}
    for b, cs in O.group_layout(block_bits):
        a = rng.standard_normal((cs.size, cs.size))
        qm, r = np.linalg.qr(a)
        mats[b] = qm * np.sign(np.diag(r))
    return [O.spec_wht128(signs, bits), O.spec_wht32(signs, bits), O.spec_so4_wht128(quats, bits),
            O.spec_group_dense(block_bits, mats)]


def test_rotations_orthogonal_and_preserve_inner_products():
    rng = np.random.default_rng(9)
    for spec in _all_specs(rng):
        R = spec.R
        np.testing.assert_allclose(R @ R.T, np.eye(128), atol=1e-12)
        q, k = rng.standard_normal((2, 128))
        assert abs((R @ q) @ (R @ k) - q @ k) < 1e-12
        # segments tile the record exactly
        cover = np.zeros(128, dtype=int)
        for s in spec.segments:
            cover[s.start:s.start + s.length] += 1
        assert np.all(cover == 1)
        # each segment's stored norm is over coordinates whose image is that segment
        for s, cs in zip(spec.segments, spec.seg_coords):
            x = np.zeros(128)
            x[cs] = rng.standard_normal(cs.size)
            y = R @ x
            outside = np.delete(y, np.arange(s.start, s.start + s.length))
            assert np.allclose(outside, 0, atol=1e-12)


def test_group_layout_blocks_to_coordinates():
    bb = np.array([4, 1, 4, 2])
    lay = O.group_layout(bb)
    assert [b for b, _ in lay] == [1, 2, 4]
    np.testing.assert_array_equal(lay[0][1], [2, 3])
    np.testing.assert_array_equal(lay[1][1], [6, 7])
    np.testing.assert_array_equal(lay[2][1], [0, 1, 4, 5])


def test_unit_basis_record_hand_derived():
    g = read_golden_kv("tq3_unit_e0.txt")
    spec = O.spec_wht128(np.ones(128), 3)
    for sign, key in ((1.0, "pos"), (-1.0, "neg")):
        x = np.zeros((1, 128))
        x[0, 0] = sign
        idx, nrm, y = O.quantize(x, spec, "f32")
        assert float(nrm[0, 0]) == float(g["norm"][0])
        assert np.all(idx == int(g[f"index_{key}"][0]))
        rec = O.pack_3bit(idx)
        assert rec.shape == (1, 48)
        want = bytes(int(b, 16) for b in g[f"bytes_{key}"]) * 16
        assert rec.tobytes() == want


def test_zero_vector():
    for spec in _all_specs(np.random.default_rng(1)):
        idx, nrm, y = O.quantize(np.zeros((2, 128)), spec, "f16")
        assert np.all(nrm == 0) and np.all(y == 0)
        for s in spec.segments:
            assert np.all(idx[:, s.start:s.start + s.length] == (1 << (s.bits - 1)) - 1)


def test_tie_goes_to_lower_cell():
    # A coordinate exactly on a boundary is not "greater", so it takes the lower
    # index ([TQ-MNN §3.4] counts strict greater-than comparisons).
    for bits in (3, 4):
        cb = O.codebook(128, bits)
        b32 = cb.boundaries.astype(np.float32).astype(np.float64)
        np.testing.assert_array_equal(O.codebook_search(b32, cb), np.arange(b32.size))
        above = np.nextafter(b32.astype(np.float32), np.float32(1)).astype(np.float64)
        np.testing.assert_array_equal(O.codebook_search(above, cb), np.arange(1, b32.size + 1))
        assert O.codebook_search(np.array([-1.0]), cb)[0] == 0
        assert O.codebook_search(np.array([1.0]), cb)[0] == (1 << bits) - 1


@pytest.mark.parametrize("bits", [3, 4])
def test_pack_roundtrip_and_bit_positions(bits):
    rng = np.random.default_rng(2)
    idx = rng.integers(0, 1 << bits, size=(50, 128))
    if bits == 3:
        rec = O.pack_3bit(idx)
        assert rec.shape == (50, 48)
        np.testing.assert_array_equal(O.unpack_3bit(rec, 128), idx)
        # bit 3i+j of the little-endian stream is bit j of index i
        stream = np.unpackbits(rec, axis=1, bitorder="little")
        for i in (0, 7, 8, 63, 127):
            for j in range(3):
                np.testing.assert_array_equal(stream[:, 3 * i + j], (idx[:, i] >> j) & 1)
    else:
        rec = O.pack_4bit(idx)
        assert rec.shape == (50, 64)
        np.testing.assert_array_equal(O.unpack_4bit(rec, 128), idx)
        np.testing.assert_array_equal(rec[:, 5], idx[:, 10] | (idx[:, 11] << 4))


def test_page_sizes_and_ratios():
    p = {k: float(v[0]) for k, v in read_golden_kv("pages_numbers.txt").items()}
    assert O.pack_3bit(np.zeros((1, 128), dtype=int)).shape[1] == p["tq3_bytes_per_128"]
    assert round(256 / 48, 1) == p["fp16_over_tq3_128"]
    assert O.pack_3bit(np.zeros((1, 8), dtype=int)).shape[1] == 3  # 8 indices in 3 bytes
    # block-32 with one fp16 norm per block: 64 B of fp16 vs codes + 2 B
    tq3 = 64 / (O.pack_3bit(np.zeros((1, 32), dtype=int)).shape[1] + 2)
    tq4 = 64 / (O.pack_4bit(np.zeros((1, 32), dtype=int)).shape[1] + 2)
    assert round(tq3, 1) == p["block32_tq3_ratio"]
    assert round(tq4, 1) == p["block32_tq4_ratio"]
    # record sizes including norms: 56 B (TQ3) and 72 B (TQ4) per block-32 vector
    assert 48 + 4 * 2 == 56 and 64 + 4 * 2 == 72


def test_norm_rounding_and_dtype():
    spec = O.spec_wht128(np.ones(128), 3)
    x = np.full((1, 128), 1.0 / 3.0)
    _, n16, _ = O.quantize(x, spec, "f16")
    _, n32, _ = O.quantize(x, spec, "f32")
    exact = math.sqrt(128) / 3
    assert n16.dtype == np.float16 and n16[0, 0] == np.float16(exact)
    assert n32.dtype == np.float32 and n32[0, 0] == np.float32(exact)


def test_sign_flip_before_transform():
    g = read_golden_kv("tq3_unit_e0.txt")
    rng = np.random.default_rng(12)
    signs = np.where(rng.random(128) < 0.5, -1.0, 1.0)
    signs[0] = -1.0
    x = np.zeros((1, 128))
    x[0, 0] = 3.0
    idx, nrm, _ = O.quantize(x, O.spec_wht128(signs, 3), "f32")
    assert np.all(idx == int(g["first_sign_negative_index"][0]))
    assert nrm[0, 0] == 3.0


def test_so4_after_transform_hand_derived():
    g = read_golden_kv("tq3_unit_e0.txt")
    quats = np.zeros((32, 2, 4))
    quats[:, :, 1] = 1.0          # q_L = q_R = i
    x = np.zeros((1, 128))
    x[0, 0] = 1.0
    idx, _, _ = O.quantize(x, O.spec_so4_wht128(quats, 3), "f32")
    want = np.tile([int(v) for v in g["so4_conj_i_indices"]], 32)
    np.testing.assert_array_equal(idx[0], want)


def test_group_segment_is_its_own_encoder():
    rng = np.random.default_rng(13)
    bb = rng.integers(1, 5, size=64)
    mats = {}
    for b, cs in O.group_layout(bb):
        a = rng.standard_normal((cs.size, cs.size))
        qm, r = np.linalg.qr(a)
        mats[b] = qm * np.sign(np.diag(r))
    spec = O.spec_group_dense(bb, mats)
    x = rng.standard_normal((3, 128))
    idx, nrm, y = O.quantize(x, spec, "f32")
    for (b, cs), seg in zip(O.group_layout(bb), spec.segments):
        n = np.linalg.norm(x[:, cs], axis=1)
        np.testing.assert_allclose(nrm[:, b - 1], n.astype(np.float32))
        want_y = (x[:, cs] @ mats[b].T) / n[:, None]
        np.testing.assert_allclose(y[:, seg.start:seg.start + seg.length], want_y, atol=1e-13)
        assert seg.cb_dim == cs.size and seg.bits == b
