"""Seeded synthetic workloads for batch-1 decode of a Qwen3-style decoder.

This module only draws numbers: model shapes, random bf16 weights, prompt ids,
TTS codebook ids and position streams.  It holds none of the decoder's
arithmetic, so the CPU oracle (``oracle/``) and the CUDA library
(``persistent_transformer_megakernel_gb300``) can both consume exactly the same
inputs without sharing any code.

The pages this build follows use trained Qwen3 / Qwen3-TTS checkpoints and real
speech text; neither exists offline, so every input here is synthetic:

* weights: ``N(0, 0.02)`` rounded to bf16 (round-to-nearest-even), RMSNorm
  gains ``1 + N(0, 0.02)``, drawn from ``torch.Generator`` seeded 0 in the
  fixed order ``embed, per layer [attn_norm, wq, wk, wv, q_norm, k_norm, wo,
  mlp_norm, w_gate, w_up, w_down], final_norm, lm_head (untied only)``;
* prompts: ids uniform in ``[0, vocab_in)`` from seed 1;
* TTS talker inputs: per step 16 codebook ids uniform in ``[0, 2048)`` and one
  text id uniform in ``[0, 151936)`` from seed 2; the 16 + 1 tables are drawn
  like weights from seed 3.

All bf16 tensors are returned as ``numpy.uint16`` bit patterns (row-major,
``[out_features][in_features]`` like ``torch.nn.Linear``).
"""
from __future__ import annotations

import numpy as np
import torch

# ---------------------------------------------------------------------------
# shapes
# ---------------------------------------------------------------------------

#: decoder shapes by workload name.  ``tied`` means the LM head reads the
#: input embedding table; ``mrope_sections`` (pairs per position stream) is
#: ``None`` for plain RoPE.
SHAPES = {
    # 2-layer decoder small enough for the oracle to finish in well under a second
    "tiny": dict(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                 intermediate=768, vocab=512, vocab_in=512, tied=False,
                 mrope_sections=None),
    # Qwen3-0.6B dimensions, tied head
    "qwen3_0p6b": dict(n_layers=28, hidden=1024, n_q_heads=16, n_kv_heads=8, head_dim=128,
                       intermediate=3072, vocab=151936, vocab_in=151936, tied=True,
                       mrope_sections=None),
    # Qwen3-TTS talker: 0.6B dims, untied 3072-entry audio-code head, MRoPE
    "tts_talker": dict(n_layers=28, hidden=1024, n_q_heads=16, n_kv_heads=8, head_dim=128,
                       intermediate=3072, vocab=3072, vocab_in=3072, tied=False,
                       mrope_sections=(24, 20, 20)),
    # Qwen3-1.7B dimensions, untied head
    "qwen3_1p7b": dict(n_layers=28, hidden=2048, n_q_heads=16, n_kv_heads=8, head_dim=128,
                       intermediate=6144, vocab=151936, vocab_in=151936, tied=False,
                       mrope_sections=None),
    # --- shapes used only by the parity tests (several tiles per CTA, ragged tails)
    # 0.6B-wide layers, few of them, a ragged vocab
    "mid": dict(n_layers=3, hidden=1024, n_q_heads=16, n_kv_heads=8, head_dim=128,
                intermediate=3072, vocab=5003, vocab_in=5003, tied=False,
                mrope_sections=None),
    # GQA group 4, head_dim 64, tied head, ragged vocab
    "gqa4": dict(n_layers=2, hidden=768, n_q_heads=8, n_kv_heads=2, head_dim=64,
                 intermediate=1536, vocab=3001, vocab_in=3001, tied=True,
                 mrope_sections=None),
    # talker-like MRoPE with head_dim 64 (sections of 32 pairs) and few layers
    "mrope_small": dict(n_layers=2, hidden=512, n_q_heads=8, n_kv_heads=4, head_dim=64,
                        intermediate=1536, vocab=1024, vocab_in=1024, tied=False,
                        mrope_sections=(12, 10, 10)),
    # the same with the interleaved MRoPE layout
    "mrope_small_interleaved": dict(n_layers=2, hidden=512, n_q_heads=8, n_kv_heads=4, head_dim=64,
                                    intermediate=1536, vocab=1024, vocab_in=1024, tied=False,
                                    mrope_sections=(12, 10, 10), mrope_interleaved=True),
    # multi-head attention (GQA group 1, the degenerate case), head_dim 128 and 64
    "mha": dict(n_layers=2, hidden=512, n_q_heads=4, n_kv_heads=4, head_dim=128,
                intermediate=1536, vocab=2003, vocab_in=2003, tied=False,
                mrope_sections=None),
    "mha64": dict(n_layers=2, hidden=512, n_q_heads=6, n_kv_heads=6, head_dim=64,
                  intermediate=1536, vocab=1024, vocab_in=1024, tied=True,
                  mrope_sections=None),
}

#: fixed scalars of every shape (Qwen3 defaults)
RMS_EPS = 1e-6
ROPE_THETA = 1e6

#: the workloads: shape, prompt length, greedy steps after the prompt
WORKLOADS = {
    "tiny": dict(shape="tiny", prompt=8, steps=16),
    "qwen3_0p6b": dict(shape="qwen3_0p6b", prompt=32, steps=512),
    "tts_talker": dict(shape="tts_talker", prompt=256, steps=0, sentinel=True),
    "qwen3_1p7b": dict(shape="qwen3_1p7b", prompt=32, steps=512),
    "long_ctx": dict(shape="qwen3_0p6b", prompt=4096, steps=1024),
}

TTS_CODEBOOKS = 16
TTS_CODEBOOK_SIZE = 2048
TTS_TEXT_VOCAB = 151936


def shape(name: str) -> dict:
    """A fresh copy of the named decoder shape with the fixed scalars added."""
    s = dict(SHAPES[name])
    s["rms_eps"] = RMS_EPS
    s["rope_theta"] = ROPE_THETA
    return s


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
              "mlp_norm", "w_gate", "w_up", "w_down")


def layer_shapes(s: dict) -> dict:
    """Per-layer tensor shapes, ``[out][in]`` for matrices."""
    H, d, I = s["hidden"], s["head_dim"], s["intermediate"]
    q, kv = s["n_q_heads"] * d, s["n_kv_heads"] * d
    return {
        "attn_norm": (H,), "wq": (q, H), "wk": (kv, H), "wv": (kv, H),
        "q_norm": (d,), "k_norm": (d,), "wo": (H, q), "mlp_norm": (H,),
        "w_gate": (I, H), "w_up": (I, H), "w_down": (H, I),
    }


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _matrix(g: torch.Generator, shp, std=0.02) -> np.ndarray:
    return _bf16_bits(torch.randn(shp, generator=g, dtype=torch.float32) * std)


def _gain(g: torch.Generator, n: int) -> np.ndarray:
    return _bf16_bits(1.0 + 0.02 * torch.randn((n,), generator=g, dtype=torch.float32))


def make_weights(s: dict, seed: int = 0) -> dict:
    """Random-init bf16 weights of shape ``s`` (bit patterns, see module doc)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    ls = layer_shapes(s)
    w = {"embed": _matrix(g, (s["vocab_in"], s["hidden"]))}
    layers = []
    for _ in range(s["n_layers"]):
        lw = {}
        for k in LAYER_KEYS:
            shp = ls[k]
            lw[k] = _gain(g, shp[0]) if len(shp) == 1 else _matrix(g, shp)
        layers.append(lw)
    w["layers"] = layers
    w["final_norm"] = _gain(g, s["hidden"])
    w["lm_head"] = None if s["tied"] else _matrix(g, (s["vocab"], s["hidden"]))
    return w


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------

def make_prompt(vocab_in: int, n: int, seed: int = 1) -> np.ndarray:
    """``n`` prompt ids uniform in ``[0, vocab_in)`` (int32)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(0, vocab_in, (n,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def make_tts_tables(hidden: int, seed: int = 3, codebook_size: int = TTS_CODEBOOK_SIZE,
                    text_vocab: int = TTS_TEXT_VOCAB) -> dict:
    """The 16 codebook tables and the text table of the talker input (bf16 bits)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    books = np.stack([_matrix(g, (codebook_size, hidden)) for _ in range(TTS_CODEBOOKS)])
    text = _matrix(g, (text_vocab, hidden))
    return {"codebooks": books, "text": text}


def make_tts_codes(n: int, seed: int = 2, codebook_size: int = TTS_CODEBOOK_SIZE,
                   text_vocab: int = TTS_TEXT_VOCAB) -> tuple:
    """Per step: 16 codebook ids ``[n][16]`` and one text id ``[n]`` (int32)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    codes = torch.randint(0, codebook_size, (n, TTS_CODEBOOKS), generator=g, dtype=torch.int64)
    text = torch.randint(0, text_vocab, (n,), generator=g, dtype=torch.int64)
    return codes.numpy().astype(np.int32), text.numpy().astype(np.int32)


def sentinel_ids(n: int, first_row: int = 0) -> np.ndarray:
    """Ids that select rows ``first_row .. first_row+n-1`` of a precomputed
    embedding buffer: row ``r`` is requested by id ``-(r + 1)``."""
    return (-(np.arange(first_row, first_row + n, dtype=np.int64) + 1)).astype(np.int32)


def make_pos3(start: int, n: int, distinct: bool) -> np.ndarray:
    """Three position-id streams ``[3][n]`` for slots ``start .. start+n-1``.

    Equal streams repeat the slot index; ``distinct`` streams are
    ``(p, p + 7, 2p + 3)`` so that every MRoPE section sees a different angle.
    """
    p = np.arange(start, start + n, dtype=np.int64)
    if distinct:
        out = np.stack([p, p + 7, 2 * p + 3])
    else:
        out = np.stack([p, p, p])
    return out.astype(np.int32)
