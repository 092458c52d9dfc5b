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
