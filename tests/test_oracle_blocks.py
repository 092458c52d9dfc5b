"""Pins for the oracle's building blocks.

Each test checks an oracle function against something other than itself: a
bit pattern fixed by the bf16 format, a value worked by hand, a closed form, an
invariant, or brute force with Python loops on a tiny case.  The hand-worked
values live in ``tests/golden/*.txt`` with their derivations.
"""
import math
import os
import struct

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------- bf16

def test_bf16_widening_bit_patterns():
    rows = _golden("bf16_values.txt")
    assert len(rows) >= 9
    for bits, value in rows:
        got = O.bf16_bits_to_f64(np.array([int(bits, 16)], dtype=np.uint16))[0]
        want = float.fromhex(value)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (bits, got)


def test_bf16_rounding_ties_to_even():
    rows = _golden("bf16_rounding.txt")
    assert len(rows) >= 9
    for x, y in rows:
        got = O.round_to_bf16(np.array([float.fromhex(x)]))[0]
        assert got == float.fromhex(y), (x, got, y)


def test_bf16_rounding_is_exact_on_bf16_values():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    v = O.bf16_bits_to_f64(bits)
    fin = np.isfinite(v)
    assert np.array_equal(O.round_to_bf16(v[fin]), v[fin])


def test_bf16_rounding_matches_torch_from_float32():
    # torch's float32 -> bfloat16 conversion rounds to nearest even; on values
    # that are exactly float32 the oracle must agree bit for bit.
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_to_bf16(x32.astype(np.float64)), ref)


def test_bf16_rounding_error_bound():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(10000) * 10.0 ** rng.uniform(-20, 20, 10000)
    r = O.round_to_bf16(x)
    # at most half an ulp: 2^-8 relative to the leading power of two
    assert np.all(np.abs(r - x) <= np.abs(x) * 2.0 ** -8 * (1 + 1e-12))


# ------------------------------------------------------------------ RMSNorm

def test_rms_norm_hand_values():
    # x = (3, 4): mean(x^2) = 12.5
    out = O.rms_norm([3.0, 4.0], [1.0, 1.0], 0.0)
    assert np.allclose(out, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    out = O.rms_norm([3.0, 4.0], [2.0, 0.5], 0.0)          # per-element gain
    assert np.allclose(out, [6 / math.sqrt(12.5), 2 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    # eps sits inside the root: x = (1e-3, 0): mean = 5e-7, plus 1e-6 = 1.5e-6
    out = O.rms_norm([1e-3, 0.0], [1.0, 1.0], 1e-6)
    assert out[0] == pytest.approx(1e-3 / math.sqrt(1.5e-6), rel=1e-14)
    assert out[1] == 0.0


def test_rms_norm_identities():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 64)) * 7
    w = np.ones(64)
    y = O.rms_norm(x, w, 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, atol=1e-13)          # unit RMS
    assert np.allclose(O.rms_norm(3.7 * x, w, 0.0), y, atol=1e-13)          # scale invariant
    assert np.array_equal(O.rms_norm(np.zeros(8), np.ones(8), 1e-6), np.zeros(8))
    g = rng.uniform(0.5, 1.5, 64)
    assert np.allclose(O.rms_norm(x, g, 0.0), y * g, atol=1e-13)            # gain is elementwise
    # rows are independent
    assert np.allclose(O.rms_norm(x[2], w, 0.0), y[2], atol=1e-15)


# --------------------------------------------------------------------- SiLU

def test_silu_values():
    # 1/(1+e^-1) = 0.7310585786300049; silu(-1) = -1/(1+e) = -0.2689414213699951
    assert O.silu(0.0) == 0.0
    assert O.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert O.silu(-1.0) == pytest.approx(-0.2689414213699951, rel=1e-15)
    assert O.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(O.silu(-40.0)) < 1e-15
    z = np.linspace(-5, 5, 101)
    assert np.allclose(O.silu(z) - O.silu(-z), z, atol=1e-14)             # silu(z) - silu(-z) = z


# --------------------------------------------------------------------- RoPE

def test_rope_frequencies_hand_values():
    phi = O.rope_angles(1000, 128, 1e6)
    assert phi[0] == 1000.0
    rows = _golden("rope_angles.txt")
    assert len(rows) >= 5
    for theta, d, pos, i, angle in rows:
        phi = O.rope_angles(int(pos), int(d), float(theta))
        assert phi[int(i)] == pytest.approx(float(angle), rel=1e-12), (theta, d, pos, i)


def test_rope_rotate_half_pairing_and_direction():
    d = 8
    for i in range(d // 2):
        phi = np.zeros(d // 2)
        phi[i] = 1.0                      # rotate pair i by one radian
        e = np.zeros(d)
        e[i] = 1.0
        want = np.zeros(d)
        want[i] = math.cos(1.0)           # a -> a cos - b sin   (b = 0)
        want[i + d // 2] = math.sin(1.0)  # b -> b cos + a sin   (b = 0)
        assert np.allclose(O.rope_apply(e, phi), want, atol=1e-16)
        e2 = np.zeros(d)
        e2[i + d // 2] = 1.0
        want2 = np.zeros(d)
        want2[i] = -math.sin(1.0)
        want2[i + d // 2] = math.cos(1.0)
        assert np.allclose(O.rope_apply(e2, phi), want2, atol=1e-16)


def test_rope_invariants():
    rng = np.random.default_rng(4)
    d = 64
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    assert np.array_equal(O.rope_apply(q, O.rope_angles(0, d, 1e6)), q)   # position 0 = identity
    for p in (1, 17, 4000):                                                # norm preserved
        assert np.linalg.norm(O.rope_apply(q, O.rope_angles(p, d, 1e6))) == pytest.approx(
            np.linalg.norm(q), rel=1e-13)

    def dot(m, n):
        return O.rope_apply(q, O.rope_angles(m, d, 1e6)) @ O.rope_apply(k, O.rope_angles(n, d, 1e6))
    for m, n in ((3, 1), (10, 2), (7, 7)):                                 # relative position only
        assert dot(m, n) == pytest.approx(dot(m + 5, n + 5), rel=1e-11, abs=1e-11)
    assert abs(dot(3, 1) - dot(4, 1)) > 1e-3


def test_mrope_equal_streams_is_rope():
    d, sec = 128, (24, 20, 20)
    for p in (0, 5, 511):
        assert np.array_equal(O.rope_angles(p, d, 1e6), O.rope_angles((p, p, p), d, 1e6, sec))


def test_interleaved_mrope_layout():
    # the interleaved reading, checked pair by pair at the talker's (24, 20, 20):
    # streams take turns 0, 1, 2, 0, 1, 2, ... until streams 1 and 2 have their
    # 20 pairs each (pairs 58 and 59 are the last), then pairs 60..63 are stream 0
    d, sec = 128, (24, 20, 20)
    st = O.decoder.pair_streams(d, sec, interleaved=True)
    assert list(st[:9]) == [0, 1, 2, 0, 1, 2, 0, 1, 2]
    assert list(st[56:64]) == [2, 0, 1, 2, 0, 0, 0, 0]
    assert [int((st == k).sum()) for k in range(3)] == [24, 20, 20]
    # equal streams reduce it to plain RoPE; a perturbed stream moves only its pairs
    for p in (0, 7, 300):
        assert np.array_equal(O.rope_angles(p, d, 1e6), O.rope_angles((p, p, p), d, 1e6, sec, True))
    base = O.rope_angles((10, 10, 10), d, 1e6, sec, True)
    for stream in range(3):
        p3 = [10, 10, 10]
        p3[stream] = 77
        changed = np.nonzero(O.rope_angles(tuple(p3), d, 1e6, sec, True) != base)[0]
        assert changed.size == sec[stream]
        assert all(st[i] == stream for i in changed)
    # with sections (32, 0, 0) nothing interleaves
    assert not O.decoder.pair_streams(64, (32, 0, 0), interleaved=True).any()


def test_mrope_sections_are_local():
    d, sec = 128, (24, 20, 20)
    base = O.rope_angles((10, 10, 10), d, 1e6, sec)
    for stream, (lo, hi) in enumerate(((0, 24), (24, 44), (44, 64))):
        p = [10, 10, 10]
        p[stream] = 99
        changed = np.nonzero(O.rope_angles(tuple(p), d, 1e6, sec) != base)[0]
        assert changed.min() == lo and changed.max() == hi - 1 and changed.size == hi - lo
    # each pair uses one angle for both of its elements (i and i + d/2)
    rng = np.random.default_rng(5)
    v = rng.standard_normal(d)
    phi = O.rope_angles((3, 40, 900), d, 1e6, sec)
    out = O.rope_apply(v, phi)
    for i in range(d // 2):
        a, b = v[i], v[i + d // 2]
        c, s = math.cos(phi[i]), math.sin(phi[i])
        assert out[i] == pytest.approx(a * c - b * s, abs=1e-13)
        assert out[i + d // 2] == pytest.approx(b * c + a * s, abs=1e-13)
    with pytest.raises(ValueError):
        O.rope_angles((1, 2, 3), d, 1e6, (24, 20, 21))


# ---------------------------------------------------------------- attention

def _brute_attention(q, K, V, Hq, Hkv):
    d = len(q[0])
    out = []
    for j in range(Hq):
        g = j // (Hq // Hkv)
        scores = [sum(q[j][i] * K[g][t][i] for i in range(d)) / math.sqrt(d) for t in range(len(K[g]))]
        m = max(scores)
        e = [math.exp(s - m) for s in scores]
        z = sum(e)
        out.append([sum(e[t] / z * V[g][t][i] for t in range(len(e))) for i in range(d)])
    return np.array(out)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(6)
    for (Hq, Hkv, d, T) in ((4, 2, 8, 1), (4, 2, 8, 6), (6, 3, 4, 5), (2, 2, 8, 3), (4, 1, 8, 4)):
        q = rng.standard_normal((Hq, d))
        K = rng.standard_normal((Hkv, T, d))
        V = rng.standard_normal((Hkv, T, d))
        got = O.attention_decode(q, K, V, Hq, Hkv)
        want = _brute_attention(q.tolist(), K.tolist(), V.tolist(), Hq, Hkv)
        assert np.allclose(got, want, atol=1e-13), (Hq, Hkv, d, T)


def test_attention_closed_forms():
    rng = np.random.default_rng(7)
    d = 4
    q = rng.standard_normal((2, d)) * 30
    K = rng.standard_normal((1, 1, d))
    V = rng.standard_normal((1, 1, d))
    # one key: the output is that value, whatever the query
    assert np.allclose(O.attention_decode(q, K, V, 2, 1), np.repeat(V[0], 2, axis=0), atol=1e-15)
    # identical keys: the mean of the values
    K = np.repeat(rng.standard_normal((1, 1, d)), 5, axis=1)
    V = rng.standard_normal((1, 5, d))
    assert np.allclose(O.attention_decode(q, K, V, 2, 1)[0], V[0].mean(axis=0), atol=1e-14)
    # two keys with scores (1, 0): q = 2 e0, k1 = e0, k2 = 0, scale 1/sqrt(4)
    q = np.array([[2.0, 0, 0, 0]])
    K = np.array([[[1.0, 0, 0, 0], [0, 0, 0, 0]]])
    V = np.array([[[1.0, 0, 0, 0], [0, 1.0, 0, 0]]])
    out = O.attention_decode(q, K, V, 1, 1)[0]
    assert out[0] == pytest.approx(math.e / (math.e + 1), rel=1e-15)    # 0.7310585786300049
    assert out[1] == pytest.approx(1 / (math.e + 1), rel=1e-15)
    # large scores do not overflow (the maximum is subtracted)
    q = np.array([[1000.0, 0, 0, 0]])
    K = np.array([[[10.0, 0, 0, 0], [9.0, 0, 0, 0]]])
    out = O.attention_decode(q, K, V, 1, 1)[0]
    assert np.all(np.isfinite(out)) and out[0] == pytest.approx(1.0)


def test_attention_group_mapping():
    # Hq = 4, Hkv = 2: heads 0,1 read kv head 0 and heads 2,3 read kv head 1
    d, T = 8, 3
    q = np.random.default_rng(8).standard_normal((4, d))
    K = np.random.default_rng(9).standard_normal((2, T, d))
    V = np.zeros((2, T, d))
    V[1] = 1.0
    out = O.attention_decode(q, K, V, 4, 2)
    assert np.allclose(out[:2], 0.0) and np.allclose(out[2:], 1.0)


# ------------------------------------------------------------ argmax, sum17

def test_argmax_lowest_index_and_errors():
    assert O.argmax_lowest([1.0, 3.0, 3.0, 2.0]) == 1
    assert O.argmax_lowest([-5.0]) == 0
    assert O.argmax_lowest([0.0, -0.0]) == 0
    with pytest.raises(FloatingPointError):
        O.argmax_lowest([1.0, float("nan")])
    with pytest.raises(FloatingPointError):
        O.argmax_lowest([1.0, float("inf")])


def test_embed_sum17_brute_force():
    rng = np.random.default_rng(10)
    H = 16
    books = rng.integers(0, 1 << 16, size=(16, 32, H), dtype=np.uint16) & np.uint16(0x3FFF)
    text = rng.integers(0, 1 << 16, size=(50, H), dtype=np.uint16) & np.uint16(0x3FFF)
    codes = rng.integers(0, 32, size=(3, 16))
    tids = rng.integers(0, 50, size=3)
    got = O.embed_sum17(books, text, codes, tids)

    def widen(b):
        return struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]
    for r in range(3):
        for c in range(H):
            acc = 0.0
            for j in range(16):
                acc += widen(books[j, codes[r, j], c])
            acc += widen(text[tids[r], c])
            assert got[r, c] == acc
