"""Pins for the oracle's compressed-domain attention, key-axis split merge,
block energies and greedy bit allocation: the rotated/dequantised identity of
the RotaryQuant page, split invariance, degenerate cases with known answers,
and brute force over all allocations on tiny inputs."""
import itertools
import math

import numpy as np
import pytest

from oracle import tq_oracle as O


def _rand_specs(rng, k_bits=3, v_bits=3):
    d = 128
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    g = rng.standard_normal((32, 2, 4))
    quats = g / np.linalg.norm(g, axis=-1, keepdims=True)
    bb = rng.integers(1, 5, size=64)
    mats = {}
    for b, cs in O.group_layout(bb):
        a = rng.standard_normal((cs.size, cs.size))
        qm, r = np.linalg.qr(a)
        mats[b] = qm * np.sign(np.diag(r))
    return [
        (O.spec_wht128(signs, k_bits), O.spec_wht128(signs, v_bits)),
        (O.spec_wht32(signs, k_bits), O.spec_wht32(signs, v_bits)),
        (O.spec_so4_wht128(quats, k_bits), O.spec_so4_wht128(quats, v_bits)),
        (O.spec_group_dense(bb, mats), O.spec_wht128(signs, v_bits)),
    ]


def _encode(rng, spec, T, scale=1.0):
    x = rng.standard_normal((T, 128)) * scale
    idx, nrm, _ = O.quantize(x, spec, "f16")
    return idx, nrm.astype(np.float64)


@pytest.mark.parametrize("kind", range(4))
def test_rotated_domain_equals_dequantize_then_attend(kind):
    # [RotaryQuant] Key design 3: <Rq, Rk> = q^T k and o~ = R o, so attention in
    # the rotated domain with one inverse rotation equals conventional
    # attention on the dequantised keys and values.
    rng = np.random.default_rng(100 + kind)
    ks, vs = _rand_specs(rng)[kind]
    T, G = 37, 4
    ki, kn = _encode(rng, ks, T)
    vi, vn = _encode(rng, vs, T)
    q = rng.standard_normal((G, 128))
    for L in (1, 5, T):
        a = O.attend_rotated(q, ki, kn, ks, vi, vn, vs, L)
        b = O.attend_dequantized(q, ki, kn, ks, vi, vn, vs, L)
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)


def test_seq_len_one_returns_dequantized_v0():
    rng = np.random.default_rng(1)
    for ks, vs in _rand_specs(rng):
        ki, kn = _encode(rng, ks, 4)
        vi, vn = _encode(rng, vs, 4)
        q = rng.standard_normal((3, 128))
        o = O.attend_rotated(q, ki, kn, ks, vi, vn, vs, 1)
        v0 = O.dequantize(vi[:1], vn[:1], vs)[0]
        np.testing.assert_allclose(o, np.broadcast_to(v0, o.shape), atol=1e-13)


def test_equal_logits_give_mean_of_values():
    # With every key identical the softmax is uniform: o is the mean of the
    # dequantised values.
    rng = np.random.default_rng(2)
    ks, vs = _rand_specs(rng)[0]
    T = 20
    ki, kn = _encode(rng, ks, 1)
    ki = np.repeat(ki, T, axis=0)
    kn = np.repeat(kn, T, axis=0)
    vi, vn = _encode(rng, vs, T)
    q = rng.standard_normal((2, 128))
    o = O.attend_rotated(q, ki, kn, ks, vi, vn, vs, T)
    want = O.dequantize(vi, vn, vs).mean(axis=0)
    np.testing.assert_allclose(o, np.broadcast_to(want, o.shape), atol=1e-13)


def test_dominant_key_selects_its_value():
    # A key aligned with q and a large norm takes (numerically) all the weight.
    rng = np.random.default_rng(4)
    ks, vs = _rand_specs(rng)[0]
    T = 16
    x = rng.standard_normal((T, 128)) * 0.01
    q = rng.standard_normal((1, 128))
    x[9] = q[0] * 50
    ki, kn, _ = O.quantize(x, ks, "f32")
    vi, vn = _encode(rng, vs, T)
    o = O.attend_rotated(q, ki, kn.astype(np.float64), ks, vi, vn, vs, T)
    np.testing.assert_allclose(o[0], O.dequantize(vi[9:10], vn[9:10], vs)[0], atol=1e-9)


@pytest.mark.parametrize("kind", range(4))
def test_lse_merge_equals_unsplit(kind):
    # [Block-GTQ]: key-axis sections merged by log-sum-exp give the unsplit
    # result; empty sections (m = -inf, l = 0) are skipped.
    rng = np.random.default_rng(20 + kind)
    ks, vs = _rand_specs(rng)[kind]
    T, G = 50, 3
    ki, kn = _encode(rng, ks, T)
    vi, vn = _encode(rng, vs, T)
    q = rng.standard_normal((G, 128))
    full = O.attend_rotated(q, ki, kn, ks, vi, vn, vs, T)
    for cuts in ([0, 50], [0, 1, 50], [0, 7, 7, 30, 49, 50], [0, 25, 50, 50]):
        bounds = list(zip(cuts[:-1], cuts[1:]))
        parts = O.split_partials(q, ki, kn, ks, vi, vn, vs, bounds)
        np.testing.assert_allclose(O.lse_merge(parts, vs), full, atol=1e-13)


def test_exact_attention_error_is_small_statistic():
    # Reported statistic (not a gate): the 3-bit path stays close to exact
    # fp64 attention on the unquantised inputs.
    rng = np.random.default_rng(5)
    ks, vs = _rand_specs(rng)[0]
    T = 256
    K = rng.standard_normal((T, 128))
    V = rng.standard_normal((T, 128))
    ki, kn, _ = O.quantize(K, ks, "f32")
    vi, vn, _ = O.quantize(V, vs, "f32")
    q = rng.standard_normal((4, 128))
    o = O.attend_rotated(q, ki, kn.astype(np.float64), ks, vi, vn.astype(np.float64), vs, T)
    ex = O.attend_exact(q, K, V, T)
    assert np.max(np.abs(o - ex)) < 0.25 * np.max(np.abs(ex)) + 0.05


# ---------------------------------------------------------------------------
# block energy and allocation  [Block-GTQ]
# ---------------------------------------------------------------------------
def test_block_energy_hand_computed():
    # q = 1 everywhere, k = 2 everywhere: each 2-dim block has ||q||^2 = 2 and
    # ||k||^2 = 8, so s_i = (2 + 8) / 2 = 5.
    q = np.ones((3, 2, 8))
    k = np.full((3, 8), 2.0)
    np.testing.assert_allclose(O.block_energy(q, k), np.full(4, 5.0))
    # only block 1 of k is nonzero
    k = np.zeros((2, 8))
    k[:, 2:4] = [3.0, 4.0]
    s = O.block_energy(np.zeros((2, 1, 8)), k)
    np.testing.assert_allclose(s, [0, 12.5, 0, 0])


def _brute(s, bmin, bmax, B):
    best = math.inf
    for b in itertools.product(range(bmin, bmax + 1), repeat=len(s)):
        if sum(b) == B:
            best = min(best, O.allocation_objective(s, b))
    return best


@pytest.mark.parametrize("seed", range(30))
def test_greedy_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 7))
    bmin = int(rng.integers(0, 3))
    bmax = int(rng.integers(bmin, 5))
    B = int(rng.integers(L * bmin, L * bmax + 1))
    s = rng.lognormal(0, 2, size=L)
    if seed % 5 == 0:
        s[:] = s[0]          # ties
    b = O.greedy_bit_alloc(s, bmin, bmax, B)
    assert b.sum() == B and b.min() >= bmin and b.max() <= bmax
    assert abs(O.allocation_objective(s, b) - _brute(s, bmin, bmax, B)) <= 1e-12 * max(1.0, _brute(s, bmin, bmax, B))


def test_greedy_special_cases():
    s = np.array([1.0, 1.0, 1.0, 1.0])
    np.testing.assert_array_equal(O.greedy_bit_alloc(s, 1, 4, 4), [1, 1, 1, 1])
    np.testing.assert_array_equal(O.greedy_bit_alloc(s, 1, 4, 16), [4, 4, 4, 4])
    np.testing.assert_array_equal(O.greedy_bit_alloc(s, 1, 4, 6), [2, 2, 1, 1])   # ties -> lowest index
    # one bit more for a block is worth 4x less: a block 4x hotter gets exactly one more bit
    np.testing.assert_array_equal(O.greedy_bit_alloc([4.0, 1.0], 1, 4, 5), [3, 2])
    with pytest.raises(ValueError):
        O.greedy_bit_alloc(s, 1, 4, 3)
    with pytest.raises(ValueError):
        O.greedy_bit_alloc(s, 1, 4, 17)


def test_expected_energy_allocation_shape():
    # Energies decaying by 10^(-i/16) (the long-context workload's block scale
    # squared): hot blocks get 4 bits, cold blocks 1, average exactly 3.
    s = 10.0 ** (-np.arange(64) / 16.0)
    b = O.greedy_bit_alloc(s, 1, 4, 192)
    assert b.sum() == 192
    assert np.all(np.diff(b) <= 0)          # monotone in energy
    assert b[0] == 4 and b[-1] == 1


def test_softmax_scale_is_inverse_sqrt_d():
    # Two keys whose logits differ by D give weights in ratio exp(D / sqrt(128)).
    rng = np.random.default_rng(6)
    ks, vs = _rand_specs(rng)[0]
    ki, kn = _encode(rng, ks, 2)
    vi, vn = _encode(rng, vs, 2)
    q = rng.standard_normal((1, 128))
    K = O.dequantize(ki, kn, ks)
    V = O.dequantize(vi, vn, vs)
    o = O.attend_rotated(q, ki, kn, ks, vi, vn, vs, 2)[0]
    # o = a0 v0 + (1 - a0) v1  ->  a0 by least squares
    dv = V[0] - V[1]
    a0 = float((o - V[1]) @ dv / (dv @ dv))
    D = float(q[0] @ (K[0] - K[1]))
    assert abs(a0 / (1 - a0) - math.exp(D / math.sqrt(128))) < 1e-9 * math.exp(abs(D) / 11)
