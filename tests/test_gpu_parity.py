"""Parity of the CUDA megakernel (through the C ABI) with the CPU oracle.

Every case draws its inputs from ``workloads`` (seeded), runs the oracle on the
CPU, then runs the library on cuda:0 in the launch configuration the bench
uses (one CTA per SM, one cooperative launch per call) and compares logits,
the layer-by-layer hidden states and the greedy ids.  Teacher-forced runs feed
the oracle's own id stream so that one near-tie flip cannot make later
forwards incomparable.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity_util import assert_close, assert_ids, first_near_tie

pytestmark = pytest.mark.gpu

mk = pytest.importorskip("persistent_transformer_megakernel_gb300")


def _run_gpu(dec, feed, n_steps=0, embeds=None, pos3=None, per_op=False, attn_chunks=0, talker=None):
    s = dec.shape
    n = len(feed) + n_steps
    logits = torch.full((n, s["vocab"]), float("nan"), dtype=torch.float32, device="cuda:0")
    hidden = torch.full((n, s["n_layers"] + 1, s["hidden"]), float("nan"), dtype=torch.float32,
                        device="cuda:0")
    ids = dec.decode(feed, n_steps, logits=logits, hidden=hidden, embeds=embeds, pos3=pos3,
                     per_op=per_op, attn_chunks=attn_chunks, talker=talker)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), logits.double().cpu().numpy(), hidden.double().cpu().numpy()


# the decode kernel mk_create picks: 1 = compiled for hidden 1024 / MLP 3072 /
# 16:8 heads of 128 (every phase inline), 0 = the general kernel
PLAN = {"mid": 1, "qwen3_0p6b": 1, "tts_talker": 1, "qwen3_1p7b": 2}


def _teacher_forced(name, n_prompt, n_steps, max_seq=64, pos3_mode=None, per_op=False,
                    attn_chunks=0):
    s = W.shape(name)
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], n_prompt, seed=1)
    n = n_prompt + n_steps
    pos3 = None if pos3_mode is None else W.make_pos3(0, n, distinct=(pos3_mode == "distinct"))
    ref = O.Decoder(s, w, max_seq=max_seq)
    ids_ref, lg_ref, hd_ref = ref.generate(prompt, n_steps, pos3=pos3)
    feed = np.concatenate([prompt, ids_ref[n_prompt - 1:n - 1]]).astype(np.int32)
    dec = mk.Decoder(s, w, max_seq=max_seq)
    assert dec.info()["plan"] == PLAN.get(name, 0)
    p3 = None if pos3 is None else torch.as_tensor(pos3, device="cuda:0")
    ids, lg, hd = _run_gpu(dec, feed, 0, pos3=p3, per_op=per_op, attn_chunks=attn_chunks)
    assert_close(lg, lg_ref, name + " logits")
    for l in range(s["n_layers"] + 1):
        assert_close(hd[:, l], hd_ref[:, l], "%s hidden[%d]" % (name, l))
    assert_ids(ids, ids_ref, lg_ref, name + " ids")
    dec.close()
    return ids, lg, hd


@pytest.mark.parametrize("name,n_prompt,n_steps", [
    ("tiny", 8, 16),          # the tiny oracle-check workload
    ("mid", 5, 70),           # 0.6B-wide layers: several tiles per CTA, ragged vocab, 75 positions
    ("gqa4", 6, 20),          # group 4, head_dim 64, tied head
    ("mha", 6, 20),           # group 1 (multi-head attention), head_dim 128
    ("mha64", 5, 24),         # group 1, head_dim 64, attention width 384 != hidden, tied head
])
def test_teacher_forced_parity(name, n_prompt, n_steps):
    _teacher_forced(name, n_prompt, n_steps, max_seq=n_prompt + n_steps + 4)


@pytest.mark.parametrize("mode", ["equal", "distinct"])
def test_mrope_parity(mode):
    _teacher_forced("mrope_small", 6, 10, max_seq=24, pos3_mode=mode)


def test_interleaved_mrope_parity():
    # streams taking turns pair by pair (rope_mode 2), distinct position streams
    _teacher_forced("mrope_small_interleaved", 6, 10, max_seq=24, pos3_mode="distinct")


def test_free_running_greedy_matches_until_a_near_tie():
    s = W.shape("tiny")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 8, seed=1)
    ids_ref, lg_ref, _ = O.Decoder(s, w, max_seq=40).generate(prompt, 16)
    dec = mk.Decoder(s, w, max_seq=40)
    ids = dec.decode(prompt, 16).cpu().numpy()
    k = first_near_tie(lg_ref)
    assert np.array_equal(ids[:k], ids_ref[:k])
    assert dec.position == 24


def test_sentinel_rows_from_gpu_embed_sum():
    # talker-style input: every forward is a negative id selecting a summed row
    s = W.shape("mrope_small")
    w = W.make_weights(s, seed=0)
    n = 12
    tables = W.make_tts_tables(s["hidden"], seed=3, codebook_size=256, text_vocab=1000)
    codes, text = W.make_tts_codes(n, seed=2, codebook_size=256, text_vocab=1000)
    E_ref = O.embed_sum17(tables["codebooks"], tables["text"], codes, text)
    books = torch.from_numpy(tables["codebooks"].view(np.int16)).view(torch.bfloat16).cuda()
    txt = torch.from_numpy(tables["text"].view(np.int16)).view(torch.bfloat16).cuda()
    E = mk.embed_sum(books, txt, torch.as_tensor(codes).cuda(), torch.as_tensor(text).cuda())
    torch.cuda.synchronize()
    assert_close(E.double().cpu().numpy(), E_ref, "17-way embedding sum")
    sid = W.sentinel_ids(n)
    pos3 = W.make_pos3(0, n, distinct=True)
    ids_ref, lg_ref, hd_ref = O.Decoder(s, w, max_seq=16).generate(sid, 0, sentinel_rows=E_ref, pos3=pos3)
    dec = mk.Decoder(s, w, max_seq=16)
    ids, lg, hd = _run_gpu(dec, sid, 0, embeds=E, pos3=torch.as_tensor(pos3, device="cuda:0"))
    assert_close(lg, lg_ref, "sentinel logits")
    assert_close(hd, hd_ref, "sentinel hidden")
    assert_ids(ids, ids_ref, lg_ref)


def _oracle_feed(name, n_prompt, n_steps, max_seq):
    """The oracle's greedy run and the teacher-forced feed that replays it."""
    s = W.shape(name)
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], n_prompt, seed=1)
    ids_ref, lg_ref, hd_ref = O.Decoder(s, w, max_seq=max_seq).generate(prompt, n_steps)
    feed = np.concatenate([prompt, ids_ref[n_prompt - 1:n_prompt + n_steps - 1]]).astype(np.int32)
    return s, w, prompt, feed, ids_ref, lg_ref, hd_ref


def _assert_oracle(s, ids, lg, hd, ids_ref, lg_ref, hd_ref, what):
    assert_close(lg, lg_ref, what + " logits")
    for l in range(s["n_layers"] + 1):
        assert_close(hd[:, l], hd_ref[:, l], "%s hidden[%d]" % (what, l))
    assert_ids(ids, ids_ref, lg_ref, what + " ids")


def test_per_op_path_matches_the_oracle_and_the_persistent_kernel():
    # the launch-overhead ablation (one launch per phase): oracle parity on a
    # teacher-forced run, and the same bits as the persistent kernel
    s, w, prompt, feed, ids_ref, lg_ref, hd_ref = _oracle_feed("mid", 6, 10, 32)
    a = mk.Decoder(s, w, max_seq=32)
    b = mk.Decoder(s, w, max_seq=32)
    ia, la, ha = _run_gpu(a, feed)
    ib, lb, hb = _run_gpu(b, feed, per_op=True)
    _assert_oracle(s, ib, lb, hb, ids_ref, lg_ref, hd_ref, "per-op")
    assert np.array_equal(ia, ib) and np.array_equal(la, lb) and np.array_equal(ha, hb)
    # free-running greedy through the per-op path, up to the oracle's first near tie
    b.reset()
    free = b.decode(prompt, 10, per_op=True).cpu().numpy()
    k = first_near_tie(lg_ref)
    assert np.array_equal(free[:k], ids_ref[:k])


def test_per_op_graph_replay_matches_the_oracle_and_the_persistent_kernel():
    # the per-op ablation replayed from a captured graph of one forward: call
    # fields read from the device call block; a second call reuses the graph
    # at a new position.  Oracle parity on both calls (teacher-forced), and
    # the same bits as the persistent kernel.
    s, w, prompt, feed, ids_ref, lg_ref, hd_ref = _oracle_feed("mid", 6, 16, 40)
    a = mk.Decoder(s, w, max_seq=40)
    b = mk.Decoder(s, w, max_seq=40)
    ia, la, ha = _run_gpu(a, feed[:16])
    ib, lb, hb = _run_gpu(b, feed[:16], per_op="graph")
    _assert_oracle(s, ib, lb, hb, ids_ref[:16], lg_ref[:16], hd_ref[:16], "graph replay")
    assert np.array_equal(ia, ib) and np.array_equal(la, lb) and np.array_equal(ha, hb)
    ia2, la2, ha2 = _run_gpu(a, feed[16:])
    ib2, lb2, hb2 = _run_gpu(b, feed[16:], per_op="graph")
    _assert_oracle(s, ib2, lb2, hb2, ids_ref[16:], lg_ref[16:], hd_ref[16:], "graph replay, second call")
    assert np.array_equal(ia2, ib2) and np.array_equal(la2, lb2) and np.array_equal(ha2, hb2)


def test_in_kernel_talker_sum_equals_the_sentinel_buffer_path():
    # negative ids with code rows: the kernel sums 16 codebook rows and a text
    # row itself, in the order mk_embed_sum uses -> bitwise the same forwards
    s = W.shape("mrope_small")
    w = W.make_weights(s, seed=0)
    n = 12
    tables = W.make_tts_tables(s["hidden"], seed=3)
    codes, text = W.make_tts_codes(n, seed=2)
    books = torch.from_numpy(tables["codebooks"].view(np.int16)).view(torch.bfloat16).cuda()
    txt = torch.from_numpy(tables["text"].view(np.int16)).view(torch.bfloat16).cuda()
    codes_d = torch.as_tensor(codes, dtype=torch.int32).cuda().contiguous()
    text_d = torch.as_tensor(text, dtype=torch.int32).cuda().contiguous()
    E = mk.embed_sum(books, txt, codes_d, text_d)
    sid = W.sentinel_ids(n)
    pos3 = torch.as_tensor(W.make_pos3(0, n, distinct=True), dtype=torch.int32).cuda().contiguous()
    a = mk.Decoder(s, w, max_seq=32)
    ia, la, ha = _run_gpu(a, sid, 3, embeds=E, pos3=None)
    b = mk.Decoder(s, w, max_seq=32)
    ib, lb, hb = _run_gpu(b, sid, 3, talker=(books, txt, codes_d, text_d))
    assert np.array_equal(ia, ib) and np.array_equal(la, lb) and np.array_equal(ha, hb)
    # distinct MRoPE streams too, through the per-op path
    a.reset(); b.reset()
    p3 = torch.as_tensor(W.make_pos3(0, n, distinct=True), dtype=torch.int32).cuda().contiguous()
    ia, la, ha = _run_gpu(a, sid, 0, embeds=E, pos3=p3)
    ib, lb, hb = _run_gpu(b, sid, 0, pos3=p3, per_op=True, talker=(books, txt, codes_d, text_d))
    assert np.array_equal(ia, ib) and np.array_equal(la, lb) and np.array_equal(ha, hb)
    # a code out of range is a bad token, reported without a fault
    bad = codes_d.clone()
    bad[5, 3] = books.shape[1]
    c = mk.Decoder(s, w, max_seq=32)
    with pytest.raises(mk.MKError):
        _run_gpu(c, sid, 0, talker=(books, txt, bad, text_d))
    del pos3


def test_streaming_mailbox_publishes_every_id_while_the_launch_runs():
    # each greedy id reaches the host-mapped mailbox as soon as it is chosen:
    # the stream equals the oracle's greedy ids up to its first near tie and
    # the ids of a plain decode everywhere, and the first id is seen before
    # the last one exists
    s = W.shape("mid")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 4, seed=1)
    ids_orc, lg_orc, _ = O.Decoder(s, w, max_seq=256).generate(prompt, 200)
    ref = mk.Decoder(s, w, max_seq=256)
    ids_ref = ref.decode(prompt, 200).cpu().numpy()
    dec = mk.Decoder(s, w, max_seq=256)
    got = list(dec.decode_stream(prompt, 200))
    assert [g[0] for g in got] == list(range(204))
    streamed = np.array([g[1] for g in got])
    k = first_near_tie(lg_orc)
    assert k > 0 and np.array_equal(streamed[:k], ids_orc[:k]), "stream differs from the oracle before forward %d" % k
    assert np.array_equal(streamed, ids_ref)
    assert got[0][2] < got[-1][2]
    # the per-op path publishes the same stream
    dec.reset()
    got2 = list(dec.decode_stream(prompt, 20, per_op=True))
    assert np.array_equal(np.array([g[1] for g in got2]), ids_ref[:24])
    # a second start without a wait is refused; the wait then succeeds
    dec.reset()
    dec.decode_start(prompt, 2)
    with pytest.raises(mk.MKError):
        dec.decode_start(prompt, 2)
    dec.decode_wait()


def test_repeat_runs_are_deterministic_and_reset_works():
    s = W.shape("mid")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 4, seed=1)
    dec = mk.Decoder(s, w, max_seq=32)
    i1, l1, h1 = _run_gpu(dec, prompt, 8)
    dec.reset()
    i2, l2, h2 = _run_gpu(dec, prompt, 8)
    assert np.array_equal(i1, i2) and np.array_equal(l1, l2) and np.array_equal(h1, h2)


@pytest.mark.parametrize("chunks", [1, 2, 7, 0, 64])
def test_split_kv_result_independent_of_chunk_count(chunks):
    s = W.shape("mid")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 40, seed=1)
    ref = mk.Decoder(s, w, max_seq=48)
    _, l_ref, h_ref = _run_gpu(ref, prompt, 0, attn_chunks=1)
    dec = mk.Decoder(s, w, max_seq=48)
    _, lg, hd = _run_gpu(dec, prompt, 0, attn_chunks=chunks)
    assert np.abs(lg - l_ref).max() <= 1e-4 * max(1.0, np.abs(l_ref).max())
    assert np.abs(hd - h_ref).max() <= 1e-4 * max(1.0, np.abs(h_ref).max())


def test_calls_continue_from_the_cursor():
    # one call of 10 forwards == a prompt call followed by a greedy-only call
    s = W.shape("tiny")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 4, seed=1)
    one = mk.Decoder(s, w, max_seq=16)
    ia, la, _ = _run_gpu(one, prompt, 6)
    two = mk.Decoder(s, w, max_seq=16)
    ib1, lb1, _ = _run_gpu(two, prompt, 0)
    ib2, lb2, _ = _run_gpu(two, [], 6)
    assert np.array_equal(ia, np.concatenate([ib1, ib2]))
    assert np.array_equal(la, np.concatenate([lb1, lb2]))
    assert two.position == 10


def test_host_buffer_entry_point_matches_device_one():
    s = W.shape("tiny")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 5, seed=1)
    a = mk.Decoder(s, w, max_seq=16)
    b = mk.Decoder(s, w, max_seq=16)
    ia = a.decode(prompt, 5).cpu().numpy()
    ib = b.decode_host(prompt, 5)
    assert np.array_equal(ia, ib)


def test_phase_trace_stamps_are_ordered_and_change_nothing():
    from persistent_transformer_megakernel_gb300 import trace as T
    s = W.shape("mid")
    w = W.make_weights(s, seed=0)
    dec = mk.Decoder(s, w, max_seq=32)
    ref = dec.decode([1, 2, 3], 3).cpu().numpy()
    dec.reset()
    buf = T.buffer(dec, 6)
    ids = dec.decode([1, 2, 3], 3, trace=buf).cpu().numpy()
    torch.cuda.synchronize()
    assert np.array_equal(ids, ref)                       # the stamps change no result
    summ = T.summarize(buf, s["n_layers"])                # raises on a missing or unordered stamp
    assert all(summ["kinds"][k]["in_phase_us"] > 0 for k in T.KINDS)
    assert len(summ["forward_us"]) == 6 and min(summ["forward_us"]) > 0
    t = buf.cpu().numpy().reshape(-1, dec.info()["grid"], 4)
    assert (t[1:, :, 0] >= t[:-1, :, 3]).all()            # every CTA takes the phases in order


def test_errors_are_reported_not_raised_as_faults():
    s = W.shape("tiny")
    w = W.make_weights(s, seed=0)
    dec = mk.Decoder(s, w, max_seq=8)
    with pytest.raises(mk.MKError) as e:
        dec.decode([3, s["vocab_in"] + 5], 0)                     # id beyond the table
    assert e.value.code == -4
    dec.reset()
    with pytest.raises(mk.MKError) as e:
        dec.decode([-1], 0)                                       # sentinel without a buffer
    assert e.value.code == -4
    dec.reset()
    with pytest.raises(mk.MKError) as e:
        dec.decode([1, 2, 3], 6)                                  # 9 forwards > max_seq 8
    assert e.value.code == -3
    dec.reset()
    # a CTA that never arrives at the grid barrier closing forward 1 (hook
    # value 2): the others give up after the wait budget and the call returns
    # a timeout
    with pytest.raises(mk.MKError) as e:
        dec.decode([1, 2], 1, spin_ns=20_000_000, fault_skip_barrier=2)
    assert e.value.code == -5
    dec.reset()
    # forward counts whose sum does not fit an int32 are rejected before any
    # launch (KV full) and leave the cursor where it was
    import ctypes as C
    d_in = torch.tensor([1], dtype=torch.int32, device="cuda:0")
    d_out = torch.empty(8, dtype=torch.int32, device="cuda:0")
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    big = 2 ** 31 - 1
    assert dec.lib.mk_decode(dec.h, C.c_void_p(d_in.data_ptr()), 1, big, C.c_void_p(d_out.data_ptr()),
                             None, st) == -3
    h_in = np.array([1], dtype=np.int32)
    h_out = np.empty(8, dtype=np.int32)
    assert dec.lib.mk_decode_host(dec.h, h_in.ctypes.data_as(C.c_void_p), 1, big,
                                  h_out.ctypes.data_as(C.c_void_p), None, st) == -3
    assert dec.info()["position"] == 0
    ids = dec.decode([1, 2], 2)                                   # the handle still works
    assert ids.shape[0] == 4


def test_zeroed_options_struct_is_a_plain_decode():
    # a memset-zero mk_decode_opts (the natural C initialiser) must run a plain
    # decode: every field's zero means "off" or "the default"
    import ctypes as C
    from persistent_transformer_megakernel_gb300 import _binding as B
    s = W.shape("tiny")
    w = W.make_weights(s, seed=0)
    prompt = W.make_prompt(s["vocab_in"], 4, seed=1)
    want = mk.Decoder(s, w, max_seq=16).decode(prompt, 4).cpu().numpy()
    dec = mk.Decoder(s, w, max_seq=16)
    d_in = torch.as_tensor(prompt, dtype=torch.int32, device="cuda:0")
    d_out = torch.full((8,), -7, dtype=torch.int32, device="cuda:0")
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    o = B.mk_decode_opts()
    C.memset(C.byref(o), 0, C.sizeof(o))
    rc = dec.lib.mk_decode(dec.h, C.c_void_p(d_in.data_ptr()), 4, 4, C.c_void_p(d_out.data_ptr()), C.byref(o), st)
    assert rc == 0, mk.error_string(rc)
    assert np.array_equal(d_out.cpu().numpy(), want)
    # a negative hook value is rejected on the host
    o.fault_skip_barrier = -1
    dec.reset()
    assert dec.lib.mk_decode(dec.h, C.c_void_p(d_in.data_ptr()), 4, 0, C.c_void_p(d_out.data_ptr()),
                             C.byref(o), st) == -1
