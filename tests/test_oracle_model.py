"""Model-level pins for the oracle decoder.

Hand-worked forwards on 2-wide models (values derived in the comments),
structural invariants that a dropped term, a wrong index or a transposed
operand would break, and agreement between the oracle's two separately written
paths (token-by-token with a KV cache, and all-positions-at-once with a causal
mask).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W


def _bits(a):
    """bf16 bit patterns of values that bf16 holds exactly."""
    a32 = np.asarray(a, dtype=np.float32)
    b = a32.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def _shape(**kw):
    base = dict(n_layers=1, hidden=2, n_q_heads=1, n_kv_heads=1, head_dim=2, intermediate=1,
                vocab=3, vocab_in=3, tied=False, rms_eps=0.0, rope_theta=1e6, mrope_sections=None)
    base.update(kw)
    return O.DecoderShape(**base)


def _layer(H=2, d=2, Hq=1, Hkv=1, I=1, **over):
    lw = {
        "attn_norm": np.ones(H), "wq": np.eye(Hq * d, H), "wk": np.eye(Hkv * d, H),
        "wv": np.zeros((Hkv * d, H)), "q_norm": np.ones(d), "k_norm": np.ones(d),
        "wo": np.zeros((H, Hq * d)), "mlp_norm": np.ones(H), "w_gate": np.zeros((I, H)),
        "w_up": np.zeros((I, H)), "w_down": np.zeros((H, I)),
    }
    lw.update(over)
    return {k: _bits(v) for k, v in lw.items()}


def _bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


# ------------------------------------------------------------ hand examples

def test_mlp_hand_example():
    # x = embed[0] = (1, 1): RMS 1, so h = (1, 1) with eps 0 and unit gain.
    # v = 0 makes attention add nothing.  gate = (1, 0).h = 1, up = (0, 2).h = 2,
    # u = silu(1) * 2 = 1.4621171572600098, down = (1, -1)^T -> x += (u, -u).
    s = _shape()
    w = {"embed": _bits([[1, 1], [0, 0], [0, 0]]), "final_norm": _bits([1, 1]),
         "lm_head": _bits([[1, 0], [0, 1], [1, 1]]),
         "layers": [_layer(w_gate=[[1, 0]], w_up=[[0, 2]], w_down=[[1], [-1]])]}
    dec = O.Decoder(s, w, max_seq=4)
    logits, hid = dec.forward_embedding(O.bf16_bits_to_f64(w["embed"][0]))
    u = 2 * 0.7310585786300049
    assert np.allclose(hid[0], [1, 1], atol=0)
    assert np.allclose(hid[1], [1 + u, 1 - u], rtol=0, atol=1e-15)


def test_attention_hand_example_two_positions():
    # Wq = Wk = I, Wv = diag(0.5, 0.25), Wo = I, no MLP.  d = 2: one rotary pair
    # with omega = 1, so position p rotates by p radians.
    # step 0, x = (1, 1): one key, so o = v0 = (0.5, 0.25); x1 = (1.5, 1.25).
    # step 1, x = (1, -1): q = k1 = R(1)(1, -1) = (cos1 + sin1, sin1 - cos1);
    #   k0 = (1, 1) (rotation 0); s0 = q.k0 / sqrt2 = sqrt2 sin1,
    #   s1 = q.bf16(k1) / sqrt2 (keys are cached in bf16; |k1|^2 = 2 before rounding);
    #   v1 = (0.5, -0.25); o = softmax(s0, s1) . (v0, v1); x1 = (1, -1) + o.
    s = _shape()
    w = {"embed": _bits([[1, 1], [1, -1], [0, 0]]), "final_norm": _bits([1, 1]),
         "lm_head": _bits([[1, 0], [0, 1], [1, 1]]),
         "layers": [_layer(wv=[[0.5, 0], [0, 0.25]], wo=np.eye(2))]}
    dec = O.Decoder(s, w, max_seq=4)
    _, hid0 = dec.forward_embedding(O.bf16_bits_to_f64(w["embed"][0]))
    assert np.array_equal(hid0[1], [1.5, 1.25])
    _, hid1 = dec.forward_embedding(O.bf16_bits_to_f64(w["embed"][1]))
    c, sn = math.cos(1.0), math.sin(1.0)
    q = np.array([c + sn, sn - c])
    k1 = _bf16(q)
    s0 = math.sqrt(2) * sn
    s1 = float(q @ k1) / math.sqrt(2)
    a0 = 1.0 / (1.0 + math.exp(s1 - s0))
    a1 = 1.0 - a0
    o = a0 * np.array([0.5, 0.25]) + a1 * np.array([0.5, -0.25])
    assert np.allclose(hid1[1], np.array([1.0, -1.0]) + o, rtol=0, atol=1e-14)
    # the cache holds the rotated, bf16-rounded keys
    assert np.array_equal(dec.K[0, 0, 0], [1.0, 1.0])
    assert np.array_equal(dec.K[0, 0, 1], k1)


def test_norm_gains_rotation_order_and_value_rounding_hand_example():
    # One layer, d = 2 (one rotary pair, omega = 1), eps 0.  attn_norm = (1, 1),
    # q_norm = (1, 2), k_norm = (2, 1): QK-norm is applied before the rotation,
    # queries and keys with their own gains.  Wq = Wk = Wo = I,
    # Wv = [[1, -2^-9], [0, 1/2]].  mlp_norm = (2, 1/2), gate row (1, 0), up row
    # (0, 1), down column (1, 0): x += (silu(h0) h1, 0) with h = rmsnorm(x) (2, 1/2).
    # step 0, x = (1, 1): h = (1, 1); v = (1 - 2^-9, 1/2) is cached in bf16 as
    #   (1, 1/2) (1 - 2^-9 is the midpoint of 1 - 2^-8 and 1: ties to even);
    #   one key, so o = (1, 1/2) and x = (2, 3/2); then the MLP with rms sqrt(3.125).
    # step 1, x = (1, -1): h = (1, -1); q = R(1)(1, -2) = (c + 2s, s - 2c),
    #   k1 = bf16(R(1)(2, -1)) = bf16((2c + s, 2s - c)), k0 = (2, 1);
    #   v1 = bf16((1 + 2^-9, -1/2)) = (1, -1/2); scores q.k / sqrt2.
    s = _shape()
    lw = _layer(wv=[[1, -2.0 ** -9], [0, 0.5]], wo=np.eye(2), q_norm=[1, 2], k_norm=[2, 1],
                mlp_norm=[2, 0.5], w_gate=[[1, 0]], w_up=[[0, 1]], w_down=[[1], [0]])
    w = {"embed": _bits([[1, 1], [1, -1], [0, 0]]), "final_norm": _bits([1, 1]),
         "lm_head": _bits([[1, 0], [0, 1], [1, 1]]), "layers": [lw]}

    def mlp(x):
        r = math.sqrt((x[0] ** 2 + x[1] ** 2) / 2)
        h0, h1 = 2 * x[0] / r, 0.5 * x[1] / r
        return np.array([x[0] + h0 / (1 + math.exp(-h0)) * h1, x[1]])

    dec = O.Decoder(s, w, max_seq=4)
    _, hid0 = dec.forward_embedding(O.bf16_bits_to_f64(w["embed"][0]))
    assert np.array_equal(dec.V[0, 0, 0], [1.0, 0.5])
    assert np.allclose(hid0[1], mlp(np.array([2.0, 1.5])), rtol=0, atol=1e-14)
    _, hid1 = dec.forward_embedding(O.bf16_bits_to_f64(w["embed"][1]))
    c, sn = math.cos(1.0), math.sin(1.0)
    q = np.array([c + 2 * sn, sn - 2 * c])
    k0 = np.array([2.0, 1.0])
    k1 = _bf16([2 * c + sn, 2 * sn - c])
    s0, s1 = float(q @ k0) / math.sqrt(2), float(q @ k1) / math.sqrt(2)
    a0 = 1.0 / (1.0 + math.exp(s1 - s0))
    o = a0 * np.array([1.0, 0.5]) + (1.0 - a0) * np.array([1.0, -0.5])
    assert np.array_equal(dec.K[0, 0, 1], k1)
    assert np.array_equal(dec.V[0, 0, 1], [1.0, -0.5])
    assert np.allclose(hid1[1], mlp(np.array([1.0, -1.0]) + o), rtol=0, atol=1e-14)


def test_eps_inside_every_model_norm_hand_example():
    # eps = 3 (large on purpose), one layer, d = 2, unit norm gains except the
    # final norm (1, 2).  Wq = Wk = Wv = Wo = I; gate row (1, 0), up row (0, 2),
    # down column (1, -1).  Every RMSNorm is x / sqrt(mean(x^2) + 3) * gain.
    # step 0, x = (1, 1): h = (1, 1)/2; one key, so o = v = (1/2, 1/2), x = (3/2, 3/2).
    # step 1, x = (1, -1): h = (1, -1)/2; q = k = R(1)((1, -1)/2 / sqrt(1/4 + 3));
    #   k0 = bf16((1, 1)/2 / sqrt(3.25)), k1 = bf16(k); v0 = (1/2, 1/2), v1 = (1/2, -1/2).
    # After attention: m = rmsnorm(x), x += (silu(m0) 2 m1, -silu(m0) 2 m1);
    # logits = head . (x / sqrt(mean(x^2) + 3) * (1, 2)).
    e = 3.0
    s = _shape(rms_eps=e)
    lw = _layer(wv=np.eye(2), wo=np.eye(2), w_gate=[[1, 0]], w_up=[[0, 2]], w_down=[[1], [-1]])
    head = np.array([[1, 0], [0, 1], [1, 1]], dtype=float)
    w = {"embed": _bits([[1, 1], [1, -1], [0, 0]]), "final_norm": _bits([1, 2]),
         "lm_head": _bits(head), "layers": [lw]}

    def rn(x):
        return np.asarray(x) / math.sqrt(float(np.mean(np.square(x))) + e)

    def after_attention(x):
        m = rn(x)
        u = m[0] / (1 + math.exp(-m[0])) * 2 * m[1]
        return x + np.array([u, -u])

    dec = O.Decoder(s, w, max_seq=4)
    lg0, hid0 = dec.forward_embedding(O.bf16_bits_to_f64(w["embed"][0]))
    x0 = after_attention(np.array([1.5, 1.5]))
    assert np.allclose(hid0[1], x0, rtol=0, atol=1e-14)
    assert np.allclose(lg0, head @ (rn(x0) * np.array([1.0, 2.0])), rtol=0, atol=1e-14)
    lg1, hid1 = dec.forward_embedding(O.bf16_bits_to_f64(w["embed"][1]))
    c, sn = math.cos(1.0), math.sin(1.0)
    kn = np.array([0.5, -0.5]) / math.sqrt(0.25 + e)
    q = np.array([kn[0] * c - kn[1] * sn, kn[1] * c + kn[0] * sn])
    k0 = _bf16(np.array([0.5, 0.5]) / math.sqrt(0.25 + e))
    k1 = _bf16(q)
    s0, s1 = float(q @ k0) / math.sqrt(2), float(q @ k1) / math.sqrt(2)
    a0 = 1.0 / (1.0 + math.exp(s1 - s0))
    o = a0 * np.array([0.5, 0.5]) + (1.0 - a0) * np.array([0.5, -0.5])
    x1 = after_attention(np.array([1.0, -1.0]) + o)
    assert np.array_equal(dec.K[0, 0, 0], k0) and np.array_equal(dec.K[0, 0, 1], k1)
    assert np.allclose(hid1[1], x1, rtol=0, atol=1e-14)
    assert np.allclose(lg1, head @ (rn(x1) * np.array([1.0, 2.0])), rtol=0, atol=1e-14)


def test_final_norm_and_head_hand_example():
    # x = (3, 4): RMS sqrt(12.5); gain (1, 2) -> (3, 8)/sqrt(12.5) = (0.8485, 2.2627);
    # head rows (1,0), (0,1), (1,1) -> logits (0.8485, 2.2627, 3.1113); argmax 2.
    s = _shape()
    w = {"embed": _bits([[3, 4], [0, 0], [0, 0]]), "final_norm": _bits([1, 2]),
         "lm_head": _bits([[1, 0], [0, 1], [1, 1]]), "layers": [_layer()]}
    dec = O.Decoder(s, w, max_seq=2)
    ids, logits, hid = dec.generate([0], 0)
    r = math.sqrt(12.5)
    assert np.allclose(logits[0], [3 / r, 8 / r, 11 / r], rtol=0, atol=1e-15)
    assert ids[0] == 2
    assert np.array_equal(hid[0, 1], [3, 4])      # zero mixers leave the residual alone


def test_untied_head_is_not_the_embedding_and_tied_is():
    s_unt = _shape()
    s_tied = _shape(tied=True)
    emb = [[3, 4], [4, 3], [0, 1]]
    w = {"embed": _bits(emb), "final_norm": _bits([1, 1]),
         "lm_head": _bits([[1, 0], [0, 1], [1, 1]]), "layers": [_layer()]}
    _, lu, _ = O.Decoder(s_unt, w, 2).generate([0], 0)
    _, lt, _ = O.Decoder(s_tied, w, 2).generate([0], 0)
    x = np.array([3.0, 4.0]) / math.sqrt(12.5)
    assert np.allclose(lt[0], np.array(emb, dtype=float) @ x, atol=1e-15)
    assert np.allclose(lu[0], np.array([[1, 0], [0, 1], [1, 1]], dtype=float) @ x, atol=1e-15)


# ----------------------------------------------------------- random models

def _tiny(name="tiny", **over):
    s = W.shape(name)
    s.update(over)
    return s, W.make_weights(s, seed=0)


def test_zero_mixers_keep_embedding_and_tied_greedy_repeats():
    # Wo = Wd = 0: every hidden state is the input embedding.  With a tied head,
    # unit final gain and orthogonal equal-norm embedding rows, logits_j is
    # proportional to e_j . e_id, so greedy decode repeats the input token.
    s = W.shape("tiny")
    s.update(tied=True, vocab=256, vocab_in=256)
    w = W.make_weights(s, seed=0)
    emb = np.zeros((256, 256))
    emb[np.arange(256), np.arange(256)] = 0.5
    w["embed"] = _bits(emb)
    w["final_norm"] = _bits(np.ones(256))
    for lw in w["layers"]:
        lw["wo"] = np.zeros_like(lw["wo"])
        lw["w_down"] = np.zeros_like(lw["w_down"])
    dec = O.Decoder(s, w, max_seq=8)
    ids, logits, hid = dec.generate([37], 3)
    assert list(ids) == [37, 37, 37, 37]
    for f in range(4):
        for l in range(s["n_layers"] + 1):
            assert np.array_equal(hid[f, l], emb[37])


def test_incremental_equals_prefix():
    s, w = _tiny()
    toks = W.make_prompt(s["vocab_in"], 12, seed=1)
    dec = O.Decoder(s, w, max_seq=16)
    ids, logits, hid = dec.generate(toks, 0)
    pl, ph, pk, pv = O.prefix_forward(s, w, toks)
    assert np.allclose(logits, pl, rtol=0, atol=1e-10)
    assert np.allclose(hid, ph, rtol=0, atol=1e-10)
    assert np.allclose(dec.K[:, :, :12], pk, rtol=0, atol=1e-10)
    assert np.allclose(dec.V[:, :, :12], pv, rtol=0, atol=1e-10)


def test_causal_mask_in_prefix_path():
    s, w = _tiny()
    toks = W.make_prompt(s["vocab_in"], 8, seed=1)
    other = toks.copy()
    other[5] = (other[5] + 1) % s["vocab_in"]
    a, _, _, _ = O.prefix_forward(s, w, toks)
    b, _, _, _ = O.prefix_forward(s, w, other)
    assert np.array_equal(a[:5], b[:5])
    assert not np.allclose(a[5], b[5])


def test_gqa_equals_mha_with_repeated_kv_heads():
    # grouped heads: q head j reads kv head j // group.  The same model written
    # as multi-head attention repeats each kv head's rows group times.
    s, w = _tiny("gqa4")               # Hq 8, Hkv 2, d 64
    d, group = s["head_dim"], s["n_q_heads"] // s["n_kv_heads"]
    s_mha = dict(s, n_kv_heads=s["n_q_heads"])
    w_mha = {k: v for k, v in w.items() if k != "layers"}
    w_mha["layers"] = []
    for lw in w["layers"]:
        m = dict(lw)
        for key in ("wk", "wv"):
            heads = lw[key].reshape(s["n_kv_heads"], d, -1)
            m[key] = np.repeat(heads, group, axis=0).reshape(s["n_q_heads"] * d, -1)
        w_mha["layers"].append(m)
    toks = W.make_prompt(s["vocab_in"], 6, seed=1)
    ids_a, la, ha = O.Decoder(s, w, 8).generate(toks, 2)
    ids_b, lb, hb = O.Decoder(s_mha, w_mha, 8).generate(toks, 2)
    assert np.array_equal(ids_a, ids_b)
    assert np.allclose(la, lb, rtol=0, atol=1e-12)


def test_sentinel_equals_explicit_17way_sum():
    s, w = _tiny()
    H = s["hidden"]
    tables = W.make_tts_tables(H, seed=3, codebook_size=64, text_vocab=100)
    codes, text = W.make_tts_codes(5, seed=2, codebook_size=64, text_vocab=100)
    E = O.embed_sum17(tables["codebooks"], tables["text"], codes, text)
    ids, logits, hid = O.Decoder(s, w, 8).generate(W.sentinel_ids(5), 0, sentinel_rows=E)
    dec = O.Decoder(s, w, 8)
    for r in range(5):
        x = sum(O.bf16_bits_to_f64(tables["codebooks"][j, codes[r, j]]) for j in range(16))
        x = x + O.bf16_bits_to_f64(tables["text"][text[r]])
        lr, hr = dec.forward_embedding(x)
        assert np.array_equal(hr, hid[r]) and np.array_equal(lr, logits[r])
    # a sentinel row that equals embed[t] behaves exactly like id t
    t = 11
    E2 = O.bf16_bits_to_f64(w["embed"][[t]])
    _, la, _ = O.Decoder(s, w, 4).generate([-1], 1, sentinel_rows=E2)
    _, lb, _ = O.Decoder(s, w, 4).generate([t], 1)
    assert np.array_equal(la, lb)


def test_mrope_model_equal_streams_and_sections():
    s, w = _tiny("mrope_small")
    toks = W.make_prompt(s["vocab_in"], 5, seed=1)
    plain = dict(s, mrope_sections=None)
    _, l_none, _ = O.Decoder(s, w, 8).generate(toks, 0)
    _, l_eq, _ = O.Decoder(s, w, 8).generate(toks, 0, pos3=W.make_pos3(0, 5, distinct=False))
    _, l_rope, _ = O.Decoder(plain, w, 8).generate(toks, 0)
    assert np.array_equal(l_none, l_eq) and np.array_equal(l_none, l_rope)
    _, l_d, _ = O.Decoder(s, w, 8).generate(toks, 0, pos3=W.make_pos3(0, 5, distinct=True))
    # position 0 attends to one key, so rotation cannot change it; later ones differ
    assert np.array_equal(l_d[0], l_none[0])
    assert all(not np.allclose(l_d[t], l_none[t]) for t in range(1, 5))
    # the prefix path follows the same streams
    pl, _, _, _ = O.prefix_forward(s, w, toks, pos3=W.make_pos3(0, 5, distinct=True))
    assert np.allclose(pl, l_d, rtol=0, atol=1e-10)


def test_interleaved_mrope_model():
    # equal streams: the interleaved layout is plain RoPE; distinct streams
    # differ from the sectioned layout (other pairs take the moved angles);
    # the prefix path follows the same interleaving
    s, w = _tiny("mrope_small")
    si = dict(s, mrope_interleaved=True)
    toks = W.make_prompt(s["vocab_in"], 5, seed=1)
    _, l_none, _ = O.Decoder(s, w, 8).generate(toks, 0)
    _, l_ieq, _ = O.Decoder(si, w, 8).generate(toks, 0, pos3=W.make_pos3(0, 5, distinct=False))
    assert np.array_equal(l_none, l_ieq)
    p3 = W.make_pos3(0, 5, distinct=True)
    _, l_sec, _ = O.Decoder(s, w, 8).generate(toks, 0, pos3=p3)
    _, l_int, _ = O.Decoder(si, w, 8).generate(toks, 0, pos3=p3)
    assert all(not np.allclose(l_int[t], l_sec[t]) for t in range(1, 5))
    pl, _, _, _ = O.prefix_forward(si, w, toks, pos3=p3)
    assert np.allclose(pl, l_int, rtol=0, atol=1e-10)


def test_generate_feeds_back_greedy_ids():
    s, w = _tiny()
    toks = W.make_prompt(s["vocab_in"], 3, seed=1)
    dec = O.Decoder(s, w, 16)
    ids, logits, _ = dec.generate(toks, 4)
    assert len(ids) == 7
    assert all(ids[i] == int(np.argmax(logits[i])) for i in range(7))
    ref = O.Decoder(s, w, 16)
    feed = list(toks) + list(ids[2:6])
    ids2, logits2, _ = ref.generate(feed, 0)
    assert np.array_equal(ids, ids2) and np.array_equal(logits, logits2)
    # a later call with no inputs continues from the last id and cursor
    more, ml, _ = dec.generate([], 2)
    ids3, l3, _ = ref.generate([ids[-1]], 1)
    assert more[0] == ids3[0] and np.array_equal(ml[0], l3[0])
    assert dec.pos == 9


def test_cache_full_is_an_error():
    s, w = _tiny()
    dec = O.Decoder(s, w, 2)
    dec.generate([1, 2], 0)
    with pytest.raises(IndexError):
        dec.generate([3], 0)
