"""Pins for the oracle's single-precision building blocks of the sampled
acceptance: the exponential, the canonical summation tree, the tree-descent
sampler and the canonical softmax.

What fixes them: the mathematics (e^x to within 2 ulp, checked against the
double-precision exponential; sums within the pairwise-summation error
bound; inverse-CDF sampling hitting each token with its weight's share), and
hand-derived cases in which summation order changes the rounded result.
"""
import math

import numpy as np
import pytest

import oracle


def _ulp32(x: float) -> float:
    x = abs(float(x))
    if x < 2.0 ** -126:
        return 2.0 ** -149
    return 2.0 ** (math.frexp(x)[1] - 24)


def test_exp_error_bound_dense_sweep():
    rng = np.random.default_rng(3)
    xs = np.concatenate([
        np.linspace(-104.0, 0.0, 400001, dtype=np.float32),
        rng.uniform(-104.0, 0.0, size=400000).astype(np.float32),
        rng.uniform(-1.0, 0.0, size=200000).astype(np.float32),
        -np.abs(rng.standard_normal(100000)).astype(np.float32) * 1e-3,
    ])
    got = oracle.exp32_array(xs).astype(np.float64)
    ref = np.exp(xs.astype(np.float64))
    ulps = np.array([_ulp32(r) for r in ref[::97]])
    err = np.abs(got[::97] - ref[::97]) / ulps
    assert err.max() <= 2.0, err.max()
    # full set, relative form for the normal range
    normal = ref > 2.0 ** -126
    rel = np.abs(got[normal] - ref[normal]) / ref[normal]
    assert rel.max() <= 2.0 * 2.0 ** -23


def test_exp_special_values():
    assert oracle.exp32(0.0) == 1.0
    assert oracle.exp32(-0.0) == 1.0
    assert oracle.exp32(-math.inf) == 0.0
    assert math.isnan(oracle.exp32(math.nan))
    assert oracle.exp32(-104.5) == 0.0
    assert oracle.exp32(-200.0) == 0.0
    # subnormal range stays within 2 units of the smallest subnormal
    for x in (-88.0, -95.0, -100.0, -103.0):
        assert abs(oracle.exp32(x) - math.exp(x)) <= 2 * 2.0 ** -149 + 2 * _ulp32(math.exp(x))


def test_canon_sum_error_bound():
    rng = np.random.default_rng(5)
    for n in (1, 2, 3, 5, 64, 1000, 4097, 151936):
        x = rng.exponential(size=n).astype(np.float32)
        exact = math.fsum(float(v) for v in x)
        levels = max(1, math.ceil(math.log2(n))) if n > 1 else 0
        bound = levels * 2.0 ** -24 * exact * 1.0001 + 1e-30
        assert abs(oracle.canon_sum(x) - exact) <= bound


def test_canon_sum_contiguous_pairing():
    e = 2.0 ** -24
    # contiguous pairs: (e + e) + (1 + 0) = 1 + 2^-23 exactly;
    # pairs (i, i + n/2) would give (e + 1) + (e + 0) = 1 (ties to even).
    assert oracle.canon_sum(np.array([e, e, 1.0, 0.0], np.float32)) == 1.0 + 2.0 ** -23
    # left to right: 1 + e rounds back to 1 each time -> 1.0.
    # tree: (1+e)=1, (e+e)=2e -> 1+2e; (e+0)+(0+0)=e -> (1+2e)+e = 1 + 1.5 ulp -> ties to even
    # -> 1 + 2^-22.
    x = np.array([1.0, e, e, e, e, 0.0, 0.0, 0.0], np.float32)
    assert oracle.canon_sum(x) == 1.0 + 2.0 ** -22
    # n not a power of two: padding with zeros does not move the result.
    x5 = np.array([1.0, e, e, e, e], np.float32)
    assert oracle.canon_sum(x5) == 1.0 + 2.0 ** -22


def test_canon_sum_zero_padding_invariance():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(3001) ** 2).astype(np.float32)
    s = oracle.canon_sum(x)
    for pad in (1, 95, 1095, 262144 - 3001):
        assert oracle.canon_sum(np.concatenate([x, np.zeros(pad, np.float32)])) == s


def test_canon_sum_trivial():
    assert oracle.canon_sum(np.array([3.5], np.float32)) == 3.5
    assert oracle.canon_sum(np.zeros(17, np.float32)) == 0.0


def test_tree_sample_full_enumeration_matches_weights():
    x = np.array([0.1, 0.0, 0.35, 0.05, 0.5], np.float32)
    us = (np.arange(2 ** 24, dtype=np.float64) * 2.0 ** -24).astype(np.float32)
    tok = oracle.tree_sample_batch(x, us)
    counts = np.bincount(tok, minlength=5)
    assert counts[1] == 0
    S = float(oracle.canon_sum(x))
    share = counts / 2 ** 24
    # each boundary is placed within one rounding of S, so per-token error is
    # a few 2^-24 grid steps
    assert np.all(np.abs(share - x.astype(np.float64) / S) <= 4 * 2.0 ** -24)


def test_tree_sample_is_monotone_inverse_cdf():
    rng = np.random.default_rng(8)
    x = rng.exponential(size=37).astype(np.float32)
    x[rng.integers(0, 37, 9)] = 0.0
    us = np.sort(rng.random(20000).astype(np.float32))
    tok = oracle.tree_sample_batch(x, us)
    assert np.all(np.diff(tok) >= 0)
    assert np.all(x[tok] > 0)
    assert oracle.tree_sample(x, 0.0) == int(np.flatnonzero(x)[0])
    assert oracle.tree_sample(x, 1.0 - 2.0 ** -24) == int(np.flatnonzero(x)[-1])


@pytest.mark.parametrize("T", [1.0, 0.7, 2.0])
def test_softmax_close_to_double(T):
    rng = np.random.default_rng(9)
    l = (rng.standard_normal(151936) * 3).astype(np.float32)
    p = oracle.softmax(l, T).astype(np.float64)
    z = l.astype(np.float64) / T
    ref = np.exp(z - z.max())
    ref /= ref.sum()
    assert abs(p.sum() - 1.0) < 1e-5
    big = ref > 1e-30
    assert np.max(np.abs(p[big] - ref[big]) / ref[big]) < 1e-5


def test_softmax_one_hot_and_uniform():
    l = np.zeros(10, np.float32)
    l[3] = 200.0
    p = oracle.softmax(l)
    assert p[3] == 1.0 and p.sum() == 1.0
    u = oracle.softmax(np.zeros(8, np.float32))
    assert np.all(u == 0.125)
