"""Batched prompt prefill (``mk_prefill``): the prompt's forwards as batched
tensor-core GEMMs plus the library's own attention / norm kernels, checked
against the oracle's all-positions path (``prefix_forward``) and against the
oracle's step path for the decode that continues after it."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity_util import assert_close, assert_ids

pytestmark = pytest.mark.gpu

mk = pytest.importorskip("persistent_transformer_megakernel_gb300")


def _prefill_then_decode(name, T, n_steps, max_seq, pos3_mode=None, sentinel=False):
    s = W.shape(name)
    w = W.make_weights(s, seed=0)
    n = T + n_steps
    pos3 = None if pos3_mode is None else W.make_pos3(0, n, distinct=(pos3_mode == "distinct"))
    shp = O.DecoderShape.from_dict(s)
    Wt = O.decoder.Weights(shp, w)
    if sentinel:
        rng = np.random.default_rng(11)
        E = rng.standard_normal((T, s["hidden"])) * 0.02
        prompt = W.sentinel_ids(T)
    else:
        E = None
        prompt = W.make_prompt(s["vocab_in"], T, seed=1)
    pl, ph, Kp, Vp = O.prefix_forward(shp, None, prompt, sentinel_rows=E,
                                      pos3=None if pos3 is None else pos3[:, :T], weights=Wt)
    ids_pre = np.array([O.argmax_lowest(r) for r in pl])
    # the oracle's step path continues from the prefix state
    ref = O.Decoder(shp, None, max_seq=max_seq, weights=Wt)
    ref.K[:, :, :T] = Kp
    ref.V[:, :, :T] = Vp
    ref.pos = T
    ref.last_id = int(ids_pre[-1])
    ids_ref, lg_ref, hd_ref = ref.generate([], n_steps, pos3=None if pos3 is None else pos3[:, T:])
    # GPU: prefill, then teacher-forced decode of the oracle's greedy ids
    dec = mk.Decoder(s, w, max_seq=max_seq)
    lg = torch.full((T, s["vocab"]), float("nan"), device="cuda:0")
    hd = torch.full((T, s["n_layers"] + 1, s["hidden"]), float("nan"), device="cuda:0")
    d_E = None if E is None else torch.as_tensor(E, dtype=torch.float32, device="cuda:0").contiguous()
    p3 = None if pos3 is None else torch.as_tensor(pos3[:, :T].copy(), device="cuda:0").contiguous()
    ids = dec.prefill(prompt, embeds=d_E, pos3=p3, logits=lg, hidden=hd).cpu().numpy()
    torch.cuda.synchronize()
    assert_close(lg.double().cpu().numpy(), pl, name + " prefill logits")
    hdn = hd.double().cpu().numpy()
    for l in range(s["n_layers"] + 1):
        assert_close(hdn[:, l], ph[:, l], "%s prefill hidden[%d]" % (name, l))
    assert_ids(ids, ids_pre, pl, name + " prefill ids")
    if n_steps:
        feed = np.concatenate([[ids_pre[-1]], ids_ref[:n_steps - 1]]).astype(np.int32)
        lg2 = torch.full((n_steps, s["vocab"]), float("nan"), device="cuda:0")
        p3d = None if pos3 is None else torch.as_tensor(pos3[:, T:].copy(), device="cuda:0").contiguous()
        ids2 = dec.decode(feed, 0, logits=lg2, pos3=p3d).cpu().numpy()
        torch.cuda.synchronize()
        assert_close(lg2.double().cpu().numpy(), lg_ref, name + " decode after prefill")
        assert_ids(ids2, ids_ref, lg_ref, name + " decode ids")
    dec.close()


@pytest.mark.parametrize("name,T,n_steps,max_seq", [
    ("tiny", 8, 8, 32),
    ("mid", 40, 12, 64),        # 0.6B-wide layers
    ("gqa4", 20, 8, 40),        # group 4, head_dim 64, tied head
    ("tiny", 300, 4, 320),      # two chunks of the 256-token scratch
    ("mha", 70, 6, 96),         # group 1, head_dim 128: three query tiles, two cache tiles
    ("mha64", 100, 4, 128),     # group 1, head_dim 64, ragged last query tile
    ("mid", 700, 4, 720),       # the third chunk ends past 512 positions: positions split over 4 CTAs + merge
    ("gqa4", 600, 3, 640),      # the same with group 4, head_dim 64
])
def test_prefill_parity(name, T, n_steps, max_seq):
    _prefill_then_decode(name, T, n_steps, max_seq)


@pytest.mark.parametrize("name", ["mrope_small", "mrope_small_interleaved"])
def test_prefill_mrope_distinct_streams(name):
    _prefill_then_decode(name, 10, 6, 24, pos3_mode="distinct")


def test_prefill_sentinel_rows():
    _prefill_then_decode("mid", 12, 4, 24, sentinel=True)


def test_prefill_graph_replay_for_new_calls_and_positions():
    # the launch sequence of a prompt length is captured once and replayed: a
    # replay with other ids, another cursor and other output buffers must give
    # what a first (capturing) call gives, and the oracle's prefix result
    s = W.shape("mid")
    w = W.make_weights(s, seed=0)
    p1 = W.make_prompt(s["vocab_in"], 16, seed=1)
    p2 = W.make_prompt(s["vocab_in"], 16, seed=7)
    a = mk.Decoder(s, w, max_seq=40)
    a.prefill(p1)                                   # captures the 16-token graph
    la = torch.full((16, s["vocab"]), float("nan"), device="cuda:0")
    ia = a.prefill(p2, logits=la).cpu().numpy()     # replay at position 16
    b = mk.Decoder(s, w, max_seq=40)
    b.prefill(p1, all_ids=False)                    # another graph (last id only)
    lb = torch.full((16, s["vocab"]), float("nan"), device="cuda:0")
    ib = b.prefill(p2, logits=lb).cpu().numpy()     # first all-ids call on b: captured now
    torch.cuda.synchronize()
    assert np.array_equal(ia, ib) and torch.equal(la, lb)
    pl, _, _, _ = O.prefix_forward(s, w, np.concatenate([p1, p2]))
    assert_close(la.double().cpu().numpy(), pl[16:], "replayed prefill at position 16")


def test_prefill_last_id_only_and_errors():
    # without ids only the last token's logits are computed; decode continues
    # from its greedy id exactly as after a one-token-per-forward prompt
    s = W.shape("mid")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 16, seed=1)
    a = mk.Decoder(s, w, max_seq=40)
    full = a.prefill(prompt).cpu().numpy()
    a_next = a.decode(None, 6).cpu().numpy()
    b = mk.Decoder(s, w, max_seq=40)
    assert b.prefill(prompt, all_ids=False) is None
    b_next = b.decode(None, 6).cpu().numpy()
    assert np.array_equal(a_next, b_next)
    assert b.info()["position"] == 22
    # a bad id is reported, not faulted; the KV-full check is on the host
    c = mk.Decoder(s, w, max_seq=40)
    bad = prompt.copy()
    bad[3] = s["vocab_in"]
    with pytest.raises(mk.MKError):
        c.prefill(bad)
    d = mk.Decoder(s, w, max_seq=10)
    with pytest.raises(mk.MKError):
        d.prefill(prompt)
    del full


def test_prefill_graph_cache_stays_bounded_and_correct():
    # more prompt lengths than the per-handle graph cache keeps (8): the least
    # recently used graphs are replaced, and a length whose graph was dropped
    # is captured again and still matches the oracle
    s = W.shape("tiny")
    w = W.make_weights(s, seed=0)
    dec = mk.Decoder(s, w, max_seq=64)
    lengths = list(range(3, 14))                    # 11 lengths
    for n in lengths:
        dec.reset()
        dec.prefill(W.make_prompt(s["vocab_in"], n, seed=n),
                    logits=torch.empty((n, s["vocab"]), device="cuda:0"))
    p = W.make_prompt(s["vocab_in"], 3, seed=3)     # the first length: its graph was replaced
    dec.reset()
    lg = torch.full((3, s["vocab"]), float("nan"), device="cuda:0")
    dec.prefill(p, logits=lg)
    torch.cuda.synchronize()
    pl, _, _, _ = O.prefix_forward(s, w, p)
    assert_close(lg.double().cpu().numpy(), pl, "prefill after the graph cache turned over")
    dec.close()
