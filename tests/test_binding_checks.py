"""The binding's size checks (host logic, no GPU): a tensor the kernel would
read or write past its end is refused before any call reaches the library."""
import pytest
import torch

from persistent_transformer_megakernel_gb300._binding import check_options

S = dict(n_layers=2, hidden=8, vocab=10)      # L, H, V
N = 5                                         # forwards of the call
G = 3                                         # CTAs (trace rows)


def _ok(**kw):
    check_options(S, N, on_device=False, **kw)


def _bad(**kw):
    with pytest.raises(ValueError):
        check_options(S, N, on_device=False, **kw)


def _t(*shape, dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype)


def test_buffers_of_the_documented_sizes_pass():
    _ok()
    _ok(out=_t(N, dtype=torch.int32), logits=_t(N, 10), hidden=_t(N, 3, 8),
        pos3=_t(3, N, dtype=torch.int32), embeds=_t(7, 8))
    _ok(out=_t(64, dtype=torch.int32), logits=_t(N + 1, 10))          # larger outputs are fine
    _ok(trace=_t(N, 11, G, 4, dtype=torch.int64), grid=G)
    _ok(talker=(_t(16, 20, 8, dtype=torch.bfloat16), _t(30, 8, dtype=torch.bfloat16),
                _t(N, 16, dtype=torch.int32), _t(N, dtype=torch.int32)))


def test_undersized_outputs_are_refused():
    _bad(out=_t(N - 1, dtype=torch.int32))
    _bad(logits=_t(N, 9))
    _bad(hidden=_t(N, 2, 8))                       # L + 1 = 3 states per forward
    _bad(trace=_t(N, 10, G, 4, dtype=torch.int64), grid=G)


def test_inputs_must_match_the_call():
    _bad(pos3=_t(3, N + 1, dtype=torch.int32))     # the row stride is the call's forward count
    _bad(pos3=_t(3, N - 1, dtype=torch.int32))
    _bad(embeds=_t(7, 9))                          # rows of hidden width
    _bad(embeds=_t(56))
    books, text = _t(16, 20, 8, dtype=torch.bfloat16), _t(30, 8, dtype=torch.bfloat16)
    _bad(talker=(books, text, _t(N, 15, dtype=torch.int32), _t(N, dtype=torch.int32)))   # codes per row
    _bad(talker=(books, text, _t(N, 16, dtype=torch.int32), _t(N - 1, dtype=torch.int32)))
    _bad(talker=(books, _t(30, 9, dtype=torch.bfloat16), _t(N, 16, dtype=torch.int32), _t(N, dtype=torch.int32)))


def test_dtype_and_layout_are_checked():
    _bad(out=_t(N, dtype=torch.int64))
    _bad(logits=_t(N, 10, dtype=torch.float64))
    _bad(pos3=_t(N, 3, dtype=torch.int32).t())     # right size, not contiguous
    _bad(trace=_t(N, 11, G, 4, dtype=torch.int32), grid=G)
    with pytest.raises(ValueError):                # host tensors where device ones are needed
        check_options(S, N, out=_t(N, dtype=torch.int32))


def test_embed_sum_tensors_are_checked():
    from persistent_transformer_megakernel_gb300._binding import check_embed_sum
    books, text = _t(16, 20, 8, dtype=torch.bfloat16), _t(30, 8, dtype=torch.bfloat16)
    codes, tids = _t(N, 16, dtype=torch.int32), _t(N, dtype=torch.int32)
    check_embed_sum(books, text, codes, tids, _t(N, 8), on_device=False)
    check_embed_sum(books, text, codes, tids, _t(N * 8 + 3), on_device=False)   # larger out is fine
    for bad in (_t(N - 1, 8), _t(N, 8, dtype=torch.float64), _t(8, N).t()):      # small, wrong dtype, strided
        with pytest.raises(ValueError):
            check_embed_sum(books, text, codes, tids, bad, on_device=False)
    with pytest.raises(ValueError):                                            # fp32 tables
        check_embed_sum(_t(16, 20, 8), text, codes, tids, _t(N, 8), on_device=False)
    with pytest.raises(ValueError):                                            # codes per row != books
        check_embed_sum(books, text, _t(N, 15, dtype=torch.int32), tids, _t(N, 8), on_device=False)
    with pytest.raises(ValueError):                                            # host tensors
        check_embed_sum(books, text, codes, tids, _t(N, 8))


def test_weights_are_checked_against_the_config():
    import numpy as np
    from persistent_transformer_megakernel_gb300._binding import check_weights
    s = dict(n_layers=1, hidden=8, n_q_heads=2, n_kv_heads=1, head_dim=4, intermediate=12, vocab=10, vocab_in=10)

    def layer():
        z = lambda *sh: np.zeros(sh, dtype=np.uint16)
        return dict(attn_norm=z(8), wq=z(8, 8), wk=z(4, 8), wv=z(4, 8), q_norm=z(4), k_norm=z(4), wo=z(8, 8),
                    mlp_norm=z(8), w_gate=z(12, 8), w_up=z(12, 8), w_down=z(8, 12))

    good = dict(embed=np.zeros((10, 8), np.uint16), final_norm=np.zeros(8, np.uint16), lm_head=None,
                layers=[layer()])
    check_weights(s, good)
    bad = dict(good, layers=[dict(layer(), wo=np.zeros((8, 4), np.uint16))])      # wrong width
    with pytest.raises(ValueError):
        check_weights(s, bad)
    with pytest.raises(ValueError):                                               # transposed view
        check_weights(s, dict(good, layers=[dict(layer(), w_down=np.zeros((12, 8), np.uint16))]))
    with pytest.raises(ValueError):                                               # fp32 numbers
        check_weights(s, dict(good, embed=np.zeros((10, 8), np.float32)))
    with pytest.raises(ValueError):                                               # torch fp32 tensor
        check_weights(s, dict(good, final_norm=torch.zeros(8)))
    t = torch.zeros(8, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):                                               # non-contiguous bf16
        check_weights(s, dict(good, layers=[dict(layer(), wq=t.t()[:, :8].t().contiguous().t())]))
    with pytest.raises(ValueError):                                               # missing layer
        check_weights(s, dict(good, layers=[]))
    with pytest.raises(ValueError):                                               # untied head of wrong size
        check_weights(s, dict(good, lm_head=np.zeros((9, 8), np.uint16)))
