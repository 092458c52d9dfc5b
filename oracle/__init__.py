"""CPU oracle for batch-1 decode of a Qwen3-style decoder.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
definition that the CUDA megakernel is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
reference arm) may import it.  The CUDA library never imports, links or runs
anything here, and nothing here imports the CUDA library: the two share only
the seeded inputs drawn by ``workloads.py``.

Arithmetic is float64 throughout (numpy); bf16 enters only where the model
defines it: weights are bf16 bit patterns widened exactly, and the KV cache
stores keys and values rounded to bf16.

Sources (cited by page title and section in every function):

* page A -- "Porting a 1,200-line persistent CUDA megakernel to Qwen3-TTS:
  ~25 ms to first audio chunk" (dev.to), sections "The idea: one kernel that
  never exits", "Porting it to Qwen3-TTS-1.7B", "What I took away";
* page B -- "I made a single CUDA kernel speak: streaming Qwen3-TTS at 50ms
  latency on an RTX 5090" (theaicatchup.com), sections "Why Does a Single
  Kernel Even Matter for TTS?" and "So, What's the Catch with These
  Megakernels?".

The pages name the architecture (a Qwen3 text decoder; the TTS talker "mirrors
Qwen3-0.6B", with an untied head, sectioned MRoPE and summed 17-way input
embeddings) but print no formulas.  Where they are silent the oracle takes the
plain Qwen3 reading: RMSNorm ``x / sqrt(mean(x^2) + eps) * w``; QK-RMSNorm per
head before rotary; rotate-half rotary pairs ``(i, i + d/2)`` with
``omega_i = theta^(-2i/d)``; causal softmax attention scaled by ``1/sqrt(d)``
with grouped KV heads (q head ``j`` reads kv head ``j // (Hq/Hkv)``); SiLU-gated
MLP; greedy argmax with the lowest index winning ties.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
hand-worked values, invariants and brute force (see those files).
"""
from .decoder import (  # noqa: F401
    Decoder,
    DecoderShape,
    argmax_lowest,
    attention_decode,
    bf16_bits_to_f64,
    embed_sum17,
    pair_streams,
    prefix_forward,
    rms_norm,
    rope_angles,
    rope_apply,
    round_to_bf16,
    silu,
)
