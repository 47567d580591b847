"""Pins for the oracle's attention over an unquantised block of tokens plus the
packed cache (fp16 prefill kept as is [RotaryQuant, deferred prefill]; the
recent-token buffer [Block-GTQ]): the two degenerate cases reduce to the pinned
packed-cache attention and to plain softmax attention (scipy), the general case
equals attention over the concatenated keys computed the conventional way, and
a worked case with equal keys has a closed form."""
import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import tq_oracle as O
from test_oracle_attention_alloc import _encode, _rand_specs


def _softmax_attention(q, K, V):
    """Reference by a library routine: softmax(q K^T / sqrt(d)) V."""
    a = softmax(q @ K.T / math.sqrt(q.shape[-1]), axis=1)
    return a @ V


def _fp16_values(rng, n, scale=1.0):
    return (rng.standard_normal((n, 128)) * scale).astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("kind", range(4))
def test_empty_prefix_is_packed_attention(kind):
    rng = np.random.default_rng(40 + kind)
    ks, vs = _rand_specs(rng)[kind]
    T = 37
    ki, kn = _encode(rng, ks, T)
    vi, vn = _encode(rng, vs, T)
    q = rng.standard_normal((4, 128))
    empty = np.zeros((0, 128))
    got = O.attend_prefix_packed(q, empty, empty, ki, kn, ks, vi, vn, vs, T)
    ref = O.attend_rotated(q, ki, kn, ks, vi, vn, vs, T)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_prefix_only_is_softmax_attention():
    rng = np.random.default_rng(7)
    ks, vs = _rand_specs(rng)[0]
    K = _fp16_values(rng, 50, 3.0)
    V = _fp16_values(rng, 50)
    q = rng.standard_normal((3, 128))
    ki = np.zeros((0, 128), dtype=np.int64)
    kn = np.zeros((0, 1))
    got = O.attend_prefix_packed(q, K, V, ki, kn, ks, ki, kn, vs, 0)
    np.testing.assert_allclose(got, _softmax_attention(q, K, V), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind", range(4))
def test_union_equals_attention_over_concatenated_keys(kind):
    """The log-sum-exp merge of the two parts against one softmax over the
    concatenation [K_pre; dequantised packed keys] (dequantise-then-attend)."""
    rng = np.random.default_rng(60 + kind)
    ks, vs = _rand_specs(rng)[kind]
    T, P = 29, 21
    ki, kn = _encode(rng, ks, T, 2.0)
    vi, vn = _encode(rng, vs, T)
    K = _fp16_values(rng, P, 2.0)
    V = _fp16_values(rng, P)
    q = rng.standard_normal((8, 128))
    got = O.attend_prefix_packed(q, K, V, ki, kn, ks, vi, vn, vs, T)
    Kc = np.concatenate([K, O.dequantize(ki, kn, ks)])
    Vc = np.concatenate([V, O.dequantize(vi, vn, vs)])
    np.testing.assert_allclose(got, _softmax_attention(q, Kc, Vc), rtol=1e-10, atol=1e-12)
    # only the first seq_len packed tokens take part
    got5 = O.attend_prefix_packed(q, K, V, ki, kn, ks, vi, vn, vs, 5)
    Kc5 = np.concatenate([K, O.dequantize(ki[:5], kn[:5], ks)])
    Vc5 = np.concatenate([V, O.dequantize(vi[:5], vn[:5], vs)])
    np.testing.assert_allclose(got5, _softmax_attention(q, Kc5, Vc5), rtol=1e-10, atol=1e-12)


def test_equal_keys_give_the_mean_value():
    """All P unquantised keys equal and no packed token: every weight is 1/P, so
    the output is the mean of the values, whatever q."""
    rng = np.random.default_rng(3)
    ks, vs = _rand_specs(rng)[0]
    P = 6
    K = np.tile(_fp16_values(rng, 1), (P, 1))
    V = _fp16_values(rng, P)
    q = rng.standard_normal((2, 128)) * 10
    e = np.zeros((0, 128), dtype=np.int64)
    got = O.attend_prefix_packed(q, K, V, e, np.zeros((0, 1)), ks, e, np.zeros((0, 1)), vs, 0)
    np.testing.assert_allclose(got, np.tile(V.mean(axis=0), (2, 1)), rtol=1e-13, atol=1e-14)


def test_both_parts_empty_give_zero():
    rng = np.random.default_rng(4)
    ks, vs = _rand_specs(rng)[0]
    e = np.zeros((0, 128))
    q = rng.standard_normal((2, 128))
    got = O.attend_prefix_packed(q, e, e, e.astype(np.int64), np.zeros((0, 1)), ks, e.astype(np.int64),
                                 np.zeros((0, 1)), vs, 0)
    assert not got.any()
