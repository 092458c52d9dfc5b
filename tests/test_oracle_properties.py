"""Randomised invariants of the oracle's building blocks (hypothesis; CPU).

Each property follows from the definition alone, so it pins the oracle against
something other than itself on inputs nobody chose by hand."""
import math

import numpy as np
import pytest

import oracle as O

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings

finite = st.floats(min_value=-1e30, max_value=1e30, allow_nan=False, allow_infinity=False)
small = st.floats(min_value=-8.0, max_value=8.0, allow_nan=False, allow_infinity=False)


@settings(max_examples=300, deadline=None)
@given(st.lists(finite, min_size=2, max_size=16))
def test_bf16_rounding_is_monotone_idempotent_and_within_half_an_ulp(xs):
    x = np.sort(np.asarray(xs, dtype=np.float64))
    r = O.round_to_bf16(x)
    assert np.all(np.diff(r) >= 0)                                   # order kept
    assert np.array_equal(O.round_to_bf16(r), r)                     # bf16 values are fixed points
    for v, q in zip(x, r):
        if v == 0 or not math.isfinite(q):
            continue
        e = max(math.frexp(v)[1], -125)                              # spacing 2^(e - 8), subnormals flat
        assert abs(q - v) <= 2.0 ** (e - 9) * (1 + 1e-12)


@settings(max_examples=200, deadline=None)
@given(st.lists(small, min_size=4, max_size=4).filter(lambda v: sum(t * t for t in v) > 1e-6),
       st.floats(min_value=1e-3, max_value=1e3))
def test_rms_norm_is_scale_invariant_with_zero_eps(x, c):
    x = np.asarray(x)
    w = np.array([1.0, -2.0, 0.5, 3.0])
    a = O.rms_norm(c * x, w, 0.0)
    b = O.rms_norm(x, w, 0.0)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    assert math.isclose(float(np.sqrt(np.mean((b / w) ** 2))), 1.0, rel_tol=1e-12)


@settings(max_examples=200, deadline=None)
@given(st.lists(small, min_size=8, max_size=8), st.lists(small, min_size=8, max_size=8),
       st.integers(0, 5000), st.integers(0, 5000), st.integers(-1000, 1000))
def test_rope_scores_depend_on_the_position_difference_only(q, k, m, n, shift):
    q, k = np.asarray(q), np.asarray(k)
    d, theta = 8, 1e6
    s1 = O.rope_apply(q, O.rope_angles(m, d, theta)) @ O.rope_apply(k, O.rope_angles(n, d, theta))
    m2, n2 = m + shift + 1000, n + shift + 1000
    s2 = O.rope_apply(q, O.rope_angles(m2, d, theta)) @ O.rope_apply(k, O.rope_angles(n2, d, theta))
    assert math.isclose(s1, s2, rel_tol=1e-9, abs_tol=1e-9 * (1 + np.abs(q).sum() * np.abs(k).sum()))
    # and a rotation keeps the norm
    assert math.isclose(float(np.linalg.norm(O.rope_apply(q, O.rope_angles(m, d, theta)))),
                        float(np.linalg.norm(q)), rel_tol=1e-12, abs_tol=1e-12)


@settings(max_examples=100, deadline=None)
@given(st.integers(1, 9), st.integers(0, 2 ** 31 - 1))
def test_attention_ignores_the_order_of_cached_positions(T, seed):
    rng = np.random.default_rng(seed)
    Hq, Hkv, d = 4, 2, 8
    q = rng.standard_normal((Hq, d))
    K = rng.standard_normal((Hkv, T, d))
    V = rng.standard_normal((Hkv, T, d))
    perm = rng.permutation(T)
    a = O.attention_decode(q, K, V, Hq, Hkv)
    b = O.attention_decode(q, K[:, perm], V[:, perm], Hq, Hkv)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    # each output is a convex combination of its kv head's values
    for j in range(Hq):
        g = j // (Hq // Hkv)
        assert np.all(a[j] <= V[g].max(axis=0) + 1e-12) and np.all(a[j] >= V[g].min(axis=0) - 1e-12)


@settings(max_examples=200, deadline=None)
@given(st.lists(st.integers(-3, 3), min_size=1, max_size=12))
def test_argmax_takes_the_lowest_index_of_the_maximum(v):
    x = np.asarray(v, dtype=np.float64)
    assert O.argmax_lowest(x) == min(i for i, t in enumerate(v) if t == max(v))
