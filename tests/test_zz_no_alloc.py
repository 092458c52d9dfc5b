"""The allocation-free talker embedding sum, called through the C ABI.

Some callers of this library cannot allocate device memory while they run (a
host embedded in another framework's fixed memory pool, or a streaming thread
where cudaMalloc could block and synchronise the device).  For them
``mk_embed_sum_noalloc`` keeps its scratch in a static device array.  This test
checks it against ``mk_embed_sum`` on two calls in a row (the second call must
not see the first call's scratch), and its error paths.  It lives in a file of
its own that pytest collects last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W
from parity_util import assert_close

pytestmark = pytest.mark.gpu

mk = pytest.importorskip("persistent_transformer_megakernel_gb300")


def _call(fn, books, text, codes, tids, out):
    n_books, book_rows, H = books.shape
    return fn(C.c_void_p(books.data_ptr()), n_books, book_rows, C.c_void_p(text.data_ptr()), text.shape[0],
              H, C.c_void_p(codes.data_ptr()), C.c_void_p(tids.data_ptr()), codes.shape[0],
              C.c_void_p(out.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_embed_sum_matches_the_allocating_entry_point():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    lib = mk.load_library()
    H = 512
    tables = W.make_tts_tables(H, seed=3, codebook_size=256, text_vocab=1000)
    books = torch.from_numpy(tables["codebooks"].view(np.int16)).view(torch.bfloat16).cuda()
    text = torch.from_numpy(tables["text"].view(np.int16)).view(torch.bfloat16).cuda()
    for seed, n in ((2, 40), (5, 9)):          # two calls in a row with different inputs
        codes_np, tids_np = W.make_tts_codes(n, seed=seed, codebook_size=256, text_vocab=1000)
        codes = torch.as_tensor(codes_np).cuda().contiguous()
        tids = torch.as_tensor(tids_np).cuda().contiguous()
        ref = torch.zeros((n, H), dtype=torch.float32, device="cuda")
        got = torch.full((n, H), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(lib.mk_embed_sum, books, text, codes, tids, ref) == 0
        assert _call(lib.mk_embed_sum_noalloc, books, text, codes, tids, got) == 0
        torch.cuda.synchronize()
        assert_close(got.double().cpu().numpy(), ref.double().cpu().numpy(), "no-alloc embedding sum")

    # a bad id is reported, and the next call starts from clean scratch
    codes_np, tids_np = W.make_tts_codes(6, seed=7, codebook_size=256, text_vocab=1000)
    bad = codes_np.copy()
    bad[3, 5] = 256
    out = torch.zeros((6, H), dtype=torch.float32, device="cuda")
    assert _call(lib.mk_embed_sum_noalloc, books, text, torch.as_tensor(bad).cuda(),
                 torch.as_tensor(tids_np).cuda(), out) == -4
    assert _call(lib.mk_embed_sum_noalloc, books, text, torch.as_tensor(codes_np).cuda(),
                 torch.as_tensor(tids_np).cuda(), out) == 0
    # more rows than the static scratch holds
    big = torch.zeros((4097, 16), dtype=torch.int32, device="cuda")
    big_t = torch.zeros(4097, dtype=torch.int32, device="cuda")
    big_out = torch.zeros((4097, H), dtype=torch.float32, device="cuda")
    assert _call(lib.mk_embed_sum_noalloc, books, text, big, big_t, big_out) == -1
