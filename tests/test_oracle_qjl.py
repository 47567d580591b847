"""Pins of the oracle's two-stage key code (a (b-1)-bit MSE code plus a 1-bit
QJL code of its residual)  [TQ-MNN §2.4].

The page fixes what the second stage is for: an unbiased estimate of the
inner product from the signs of a random projection.  The pins below check that
property itself (over many independent projections, with the variance the
sign estimator must have), hand-worked examples whose numbers come from closed
forms (the 1-bit codebook of the d = 4 coordinate density is +-4 / (3 pi)), the
residual energy the Lloyd-Max conditions imply, the bit layout, and attention
by brute force on a tiny case."""
import math

import numpy as np
import pytest

from oracle import tq_oracle as O


def _one_score(x, q, qs, norm_dtype="f32"):
    idx, sb, nr, y, z = O.qjl_quantize(np.asarray([x], dtype=np.float64), qs, norm_dtype)
    return float(O.qjl_scores(np.asarray([q], dtype=np.float64), idx, sb, nr.astype(np.float64), qs)[0, 0])


def test_hand_example_qjl_only():
    """b = 1: no MSE code; the whole normalised vector is the residual.  x = (3,
    0, 4, 0): n = 5, y = r = (0.6, 0, 0.8, 0), rho = 1; with S = I the signs of z = r
    are all +1 (a zero counts as +1).  For q = (1, 2, 3, 4):
    estimate = 5 * 1 * sqrt(pi/2) / 4 * (1 + 2 + 3 + 4) = 12.5 sqrt(pi/2)."""
    qs = O.QjlSpec(np.eye(4), 0, np.eye(4))
    idx, sb, nr, y, z = O.qjl_quantize(np.array([[3.0, 0.0, 4.0, 0.0]]), qs, "f32")
    assert idx.tolist() == [[0, 0, 0, 0]]
    assert sb.tolist() == [[1, 1, 1, 1]]
    assert nr.astype(np.float64).tolist() == [[5.0, 5.0]]
    est = O.qjl_scores(np.array([[1.0, 2.0, 3.0, 4.0]]), idx, sb, nr.astype(np.float64), qs)
    assert est[0, 0] == pytest.approx(12.5 * math.sqrt(math.pi / 2), rel=1e-12)


def test_hand_example_two_stage():
    """b = 2 in d = 4: the 1-bit Lloyd-Max codebook of the density (1 - t^2)^(1/2)
    is +-c with c = E|t| = (1/3) / (pi/4) = 4 / (3 pi).  x = (3, 0, 4, 0): y = (0.6,
    0, 0.8, 0), codes (1, 0, 1, 0) (0 is not > 0), y^ = (c, -c, c, -c), r = y - y^.
    With S = [[1,0,0,0], [0,-1,0,0], [1,1,0,0], [0,0,1,-1]]: z = (0.6 - c, -c, 0.6,
    0.8 - 2c), signs (+, -, +, -).  For q = (1, 2, 3, 4) (R = I): the MSE term is
    5 c (1 - 2 + 3 - 4) = -10 c; S q = (1, -2, 3, -1) against the signs gives 7; so
    estimate = -10 c + 5 rho sqrt(pi/2) / 4 * 7."""
    c = 4.0 / (3.0 * math.pi)
    S = np.array([[1, 0, 0, 0], [0, -1, 0, 0], [1, 1, 0, 0], [0, 0, 1, -1]], dtype=np.float64)
    qs = O.QjlSpec(np.eye(4), 1, S)
    np.testing.assert_allclose(O.codebook(4, 1).centroids, [-c, c], rtol=1e-12)
    idx, sb, nr, y, z = O.qjl_quantize(np.array([[3.0, 0.0, 4.0, 0.0]]), qs, "f32")
    assert idx.tolist() == [[1, 0, 1, 0]]
    r = np.array([0.6 - c, c, 0.8 - c, c])
    np.testing.assert_allclose(z[0], [0.6 - c, -c, 0.6, 0.8 - 2 * c], rtol=1e-12, atol=1e-15)
    assert sb.tolist() == [[1, 0, 1, 0]]
    rho = math.sqrt(float(r @ r))
    np.testing.assert_allclose(nr.astype(np.float64)[0], [5.0, np.float32(5.0 * rho)], rtol=1e-7)
    est = O.qjl_scores(np.array([[1.0, 2.0, 3.0, 4.0]]), idx, sb, nr.astype(np.float64), qs)
    want = -10.0 * c + float(np.float32(5.0 * rho)) * math.sqrt(math.pi / 2) / 4.0 * 7.0
    assert est[0, 0] == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("b", [1, 2])
def test_unbiased_over_projections(b):
    """The defining property: over independent Gaussian projections S the estimate
    averages to <q, x>, and its variance is the sign estimator's
      n^2 rho^2 / d * ((pi/2) ||q~||^2 - <q~, r / rho>^2)
    (each row contributes E[(s.a) sign(s.r)] = sqrt(2/pi) <a, r> / ||r|| and
    E[(s.a)^2] = ||a||^2).  A dropped residual, a wrong sqrt(pi/2) or 1/d, or a
    flipped sign convention moves the mean by many standard errors."""
    d, M = 64, 3000
    rng = np.random.default_rng([7, b])
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    R = O.hadamard(d) @ np.diag(signs)
    x = rng.standard_normal(d) * np.linspace(0.5, 3.0, d)
    q = rng.standard_normal(d) + 0.8 * x / np.linalg.norm(x)
    est = np.empty(M)
    for m in range(M):
        qs = O.QjlSpec(R, b - 1, rng.standard_normal((d, d)))
        est[m] = _one_score(x, q, qs)
    truth = float(q @ x)
    # the variance from closed forms of the same encoding (independent of S)
    qs0 = O.QjlSpec(R, b - 1, np.eye(d))
    idx, sb, nr, y, z = O.qjl_quantize(x[None], qs0, "f32")
    n = float(np.linalg.norm(x))
    yhat = O.codebook(d, b - 1).centroids[idx[0]] if b > 1 else np.zeros(d)
    r = y[0] - yhat
    rho = float(np.linalg.norm(r))
    qt = R @ q
    var = n * n * rho * rho / d * (math.pi / 2 * float(qt @ qt) - float(qt @ (r / rho)) ** 2)
    se = math.sqrt(var / M)
    assert abs(est.mean() - truth) < 4.0 * se, (est.mean(), truth, se)
    assert est.var(ddof=1) == pytest.approx(var, rel=0.15)


def test_residual_energy_matches_lloyd_max():
    """With a 1-bit MSE stage the centroid is the conditional mean, c = E|y|, so
    E||r||^2 = 1 - 2 c E sum|y_i| + d c^2 = 1 - d c^2 over uniformly random unit
    vectors; with no MSE stage r = y and rho = 1 exactly."""
    d, N = 128, 4000
    rng = np.random.default_rng(11)
    x = rng.standard_normal((N, d))
    qs = O.QjlSpec(np.eye(d), 1, np.eye(d))
    idx, sb, nr, y, z = O.qjl_quantize(x, qs, "f32")
    c = O.codebook(d, 1).centroids[1]
    rho2 = (nr[:, 1].astype(np.float64) / nr[:, 0].astype(np.float64)) ** 2
    assert rho2.mean() == pytest.approx(1.0 - d * c * c, rel=0.01)
    _, _, nr0, _, _ = O.qjl_quantize(x, O.QjlSpec(np.eye(d), 0, np.eye(d)), "f32")
    np.testing.assert_allclose(nr0[:, 1], nr0[:, 0], rtol=1e-7)


def test_zero_vector():
    """A zero key stores norms (0, 0) and contributes score 0."""
    d = 16
    qs = O.QjlSpec(np.eye(d), 1, np.random.default_rng(1).standard_normal((d, d)))
    idx, sb, nr, y, z = O.qjl_quantize(np.zeros((1, d)), qs, "f16")
    assert nr.astype(np.float64).tolist() == [[0.0, 0.0]]
    assert O.qjl_scores(np.ones((1, d)), idx, sb, nr.astype(np.float64), qs)[0, 0] == 0.0


def test_mse_term_is_the_one_stage_code():
    """With S = 0 the QJL term vanishes and the score is the one-stage 1-bit
    code's <q~, n C[idx]> (the pinned one-stage dequantiser)."""
    d = 128
    rng = np.random.default_rng(3)
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    spec = O.spec_wht128(signs, 1)
    qs = O.QjlSpec(spec.R, 1, np.zeros((d, d)))
    x = rng.standard_normal((20, d))
    q = rng.standard_normal((3, d))
    idx, sb, nr, y, z = O.qjl_quantize(x, qs, "f32")
    idx1, nr1, _ = O.quantize(x, spec, "f32")
    np.testing.assert_array_equal(idx, idx1)
    want = (q @ spec.R.T) @ O.dequantize_rotated(idx1, nr1.astype(np.float64), spec).T
    got = O.qjl_scores(q, idx, sb, nr.astype(np.float64), qs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_record_layout():
    """MSE codes LSB first, then the sign bits: for d = 16 and b = 2, codes set at
    positions 0, 8, 9, 15 give bytes 0x01, 0x83; signs all +1 but position 3 give
    0xF7, 0xFF.  Record sizes: 16 (b = 1) and 32 (b = 2) bytes at d = 128."""
    idx = np.zeros((1, 16), dtype=np.int64)
    idx[0, [0, 8, 9, 15]] = 1
    sb = np.ones((1, 16), dtype=np.int64)
    sb[0, 3] = 0
    rec = O.qjl_pack(idx, sb, 1)
    assert rec.tolist() == [[0x01, 0x83, 0xF7, 0xFF]]
    i2, s2 = O.qjl_unpack(rec, 1, 16)
    np.testing.assert_array_equal(i2, idx)
    np.testing.assert_array_equal(s2, sb)
    assert O.qjl_record_bytes(0) == 16 and O.qjl_record_bytes(1) == 32
    rng = np.random.default_rng(5)
    idx = rng.integers(0, 2, (7, 128))
    sb = rng.integers(0, 2, (7, 128))
    for mb in (0, 1):
        rec = O.qjl_pack(idx * mb, sb, mb)
        assert rec.shape == (7, O.qjl_record_bytes(mb))
        i2, s2 = O.qjl_unpack(rec, mb, 128)
        np.testing.assert_array_equal(i2, idx * mb)
        np.testing.assert_array_equal(s2, sb)


def test_attention_brute_force():
    """attend_qjl against per-token loops on a tiny case (d = 8, T = 5, 2 heads):
    each score summed coordinate by coordinate and projection row by row,
    softmax, values dequantised one by one and rotated back."""
    d, T = 8, 5
    rng = np.random.default_rng(9)
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    R = O.hadamard(d) @ np.diag(signs)
    S = rng.standard_normal((d, d))
    qs = O.QjlSpec(R, 1, S)
    vspec = O.HeadSpec(R, [O.Segment(0, d, d, 3, 0)], [np.arange(d)], 1, False)
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    q = rng.standard_normal((2, d))
    idx, sb, nr, y, z = O.qjl_quantize(K, qs, "f32")
    vidx, vnr, _ = O.quantize(V, vspec, "f32")
    got = O.attend_qjl(q, idx, sb, nr.astype(np.float64), qs, vidx, vnr.astype(np.float64), vspec, T)
    C1 = O.codebook(d, 1).centroids
    C3 = O.codebook(d, 3).centroids
    for g in range(2):
        qt = [sum(R[i, c] * q[g, c] for c in range(d)) for i in range(d)]
        u = [sum(S[j, i] * qt[i] for i in range(d)) for j in range(d)]
        s = []
        for t in range(T):
            n, nrho = float(nr[t, 0]), float(nr[t, 1])
            mse = sum(qt[i] * n * C1[idx[t, i]] for i in range(d))
            qj = sum(u[j] * (1.0 if sb[t, j] else -1.0) for j in range(d))
            s.append((mse + nrho * math.sqrt(math.pi / 2) / d * qj) / math.sqrt(d))
        mx = max(s)
        w = [math.exp(v - mx) for v in s]
        tot = sum(w)
        ot = [sum(w[t] / tot * float(vnr[t, 0]) * C3[vidx[t, i]] for t in range(T)) for i in range(d)]
        o = [sum(R[i, c] * ot[i] for i in range(d)) for c in range(d)]
        np.testing.assert_allclose(got[g], o, rtol=1e-10, atol=1e-12)
