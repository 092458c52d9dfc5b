"""float64 reference decoder (test infrastructure only; see the package doc).

Page A = "Porting a 1,200-line persistent CUDA megakernel to Qwen3-TTS: ~25 ms
to first audio chunk" (dev.to).  Page B = "I made a single CUDA kernel speak:
streaming Qwen3-TTS at 50ms latency on an RTX 5090" (theaicatchup.com).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# bf16 <-> float64
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns exactly: a bf16 value is the top 16 bits of the
    float32 with the same sign, exponent and leading 7 mantissa bits."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):      # NaN patterns stay NaN
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(F64)


_BF16_MAX = float.fromhex("0x1.fep127")  # (2 - 2^-7) * 2^127


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits (1 implicit + 7 stored) and float32's
    exponent range; below 2^-126 the spacing stays 2^-133 (subnormals).
    Used for the bf16 KV cache the decode path keeps (long-context workload:
    "bf16 KV cache")."""
    x = np.asarray(x, dtype=F64)
    _, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    e_eff = np.maximum(e, -125)              # 2^-126 = 0.5 * 2^-125
    q = np.rint(np.ldexp(x, 8 - e_eff))      # 8 significant bits; rint = ties-to-even
    y = np.ldexp(q, e_eff - 8)
    y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, x), y)
    return np.where(np.isfinite(x), y, x)


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------

def rms_norm(x, w, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: ``x / sqrt(mean(x^2) + eps) * w``
    (Qwen3's normalisation; the pages only name the model family, page A
    "Porting it to Qwen3-TTS-1.7B")."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)


def silu(z) -> np.ndarray:
    """SiLU ``z * sigmoid(z) = z / (1 + e^-z)``, the gate of Qwen3's MLP."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def pair_streams(head_dim: int, mrope_sections: Optional[Sequence[int]],
                 interleaved: bool = False) -> np.ndarray:
    """Which position stream drives each rotary pair ``i < d/2``.

    Plain RoPE: stream 0 for every pair.  MRoPE (page A, "Porting it to
    Qwen3-TTS-1.7B": the talker's rotary positions come in sections):
    contiguous runs of pair indices, ``sections[0]`` pairs on stream 0, the next
    ``sections[1]`` on stream 1, the rest on stream 2.

    Interleaved variant (the pages name only "sections"; this layout is a
    reading): the three streams take turns pair by pair -- pair ``i`` with
    ``i mod 3 = s`` for ``s`` in {1, 2} belongs to stream ``s`` while
    ``i < 3 * sections[s]``; every other pair belongs to stream 0.  Each stream
    still drives exactly ``sections[s]`` pairs."""
    half = head_dim // 2
    if mrope_sections is None:
        return np.zeros(half, dtype=np.int64)
    if sum(mrope_sections) != half:
        raise ValueError("MRoPE sections must cover head_dim/2 pairs")
    if not interleaved:
        return np.repeat(np.arange(len(mrope_sections)), mrope_sections)
    out = np.zeros(half, dtype=np.int64)
    for i in range(half):
        r = i % 3
        if r in (1, 2) and i < 3 * mrope_sections[r]:
            out[i] = r
    return out


def rope_angles(positions, head_dim: int, theta: float,
                mrope_sections: Optional[Sequence[int]] = None, interleaved: bool = False) -> np.ndarray:
    """Rotation angle of every pair: ``phi_i = pos_{s(i)} * theta^(-2i/d)``.

    ``positions`` is one position (plain RoPE) or three position-stream values.
    The frequencies are the host-built table the talker needs (page B, "So,
    What's the Catch with These Megakernels?": rotary frequencies come from
    tables built on the host), here in double precision."""
    half = head_dim // 2
    i = np.arange(half, dtype=F64)
    omega = np.power(F64(theta), -2.0 * i / head_dim)
    pos = np.atleast_1d(np.asarray(positions, dtype=F64))
    s = pair_streams(head_dim, mrope_sections, interleaved)
    if pos.size == 1:
        p = np.full(half, pos[0])
    else:
        p = pos[s]
    return p * omega


def rope_apply(v, phi) -> np.ndarray:
    """Rotate-half rotary embedding on the last axis: pair ``(a, b) =
    (v_i, v_{i+d/2})`` becomes ``(a cos phi_i - b sin phi_i,
    b cos phi_i + a sin phi_i)``."""
    v = np.asarray(v, dtype=F64)
    half = v.shape[-1] // 2
    a, b = v[..., :half], v[..., half:]
    c, s = np.cos(phi), np.sin(phi)
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention_decode(q, K, V, n_q_heads: int, n_kv_heads: int) -> np.ndarray:
    """One query position against cached keys/values (grouped-query attention).

    ``q`` is ``[Hq][d]``; ``K``, ``V`` are ``[Hkv][T][d]`` for the ``T`` attended
    slots.  Head ``j`` reads kv head ``j // (Hq / Hkv)``; weights are
    ``softmax_t(q_j . K_t / sqrt(d))`` with the maximum subtracted first; the
    output is ``sum_t a_t V_t``.  Returns ``[Hq][d]``."""
    q = np.asarray(q, dtype=F64)
    d = q.shape[-1]
    group = n_q_heads // n_kv_heads
    out = np.empty_like(q)
    for j in range(n_q_heads):
        g = j // group
        s = K[g] @ q[j] / np.sqrt(F64(d))
        a = np.exp(s - s.max())
        a /= a.sum()
        out[j] = a @ V[g]
    return out


def argmax_lowest(logits) -> int:
    """Greedy choice: the largest logit, the lowest index among equals.
    A NaN or infinite logit is an error."""
    x = np.asarray(logits, dtype=F64)
    if not np.all(np.isfinite(x)):
        raise FloatingPointError("non-finite logit")
    return int(np.argmax(x))  # numpy returns the first maximal index


def embed_sum17(codebooks_bits, text_bits, codes, text_ids) -> np.ndarray:
    """The talker's per-step input: the sum of 16 codebook embeddings and one
    text embedding (page B, "Why Does a Single Kernel Even Matter for TTS?":
    each talker input is that 17-way sum).  Summed in table order
    0..15 then text.  ``codes`` ``[n][16]``, ``text_ids`` ``[n]`` -> ``[n][H]``."""
    codes = np.asarray(codes)
    text_ids = np.asarray(text_ids)
    n, nb = codes.shape
    out = np.zeros((n, codebooks_bits.shape[-1]), dtype=F64)
    for r in range(n):
        acc = np.zeros(codebooks_bits.shape[-1], dtype=F64)
        for j in range(nb):
            acc = acc + bf16_bits_to_f64(codebooks_bits[j, codes[r, j]])
        acc = acc + bf16_bits_to_f64(text_bits[text_ids[r]])
        out[r] = acc
    return out


# ---------------------------------------------------------------------------
# model
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class DecoderShape:
    """Dimensions of a Qwen3-style decoder (page B, "Why Does a Single Kernel
    Even Matter for TTS?": the talker has Qwen3-0.6B's dimensions, layer count
    and heads; only vocab, RoPE frequencies and the untied head differ)."""
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    vocab_in: int
    tied: bool
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    mrope_sections: Optional[tuple] = None
    mrope_interleaved: bool = False

    @classmethod
    def from_dict(cls, s: dict) -> "DecoderShape":
        ms = s.get("mrope_sections")
        return cls(n_layers=s["n_layers"], hidden=s["hidden"], n_q_heads=s["n_q_heads"],
                   n_kv_heads=s["n_kv_heads"], head_dim=s["head_dim"],
                   intermediate=s["intermediate"], vocab=s["vocab"],
                   vocab_in=s["vocab_in"], tied=bool(s["tied"]),
                   rms_eps=float(s.get("rms_eps", 1e-6)),
                   rope_theta=float(s.get("rope_theta", 1e6)),
                   mrope_sections=None if ms is None else tuple(ms),
                   mrope_interleaved=bool(s.get("mrope_interleaved", False)))


class Weights:
    """bf16 weights widened once to float64."""

    def __init__(self, shp: DecoderShape, bits: dict):
        self.embed = bf16_bits_to_f64(bits["embed"])
        self.final_norm = bf16_bits_to_f64(bits["final_norm"])
        # untied vs tied head (page A, "Porting it to Qwen3-TTS-1.7B": the text
        # model ties input embedding and output head, the talker does not)
        if shp.tied:
            self.lm_head = self.embed
        else:
            self.lm_head = bf16_bits_to_f64(bits["lm_head"])
        self.layers = [{k: bf16_bits_to_f64(v) for k, v in lw.items()} for lw in bits["layers"]]


def _input_row(W: Weights, token: int, sentinel_rows) -> np.ndarray:
    """Input embedding of one forward.  A non-negative id reads the embedding
    table; a negative id ``-(r+1)`` reads row ``r`` of the caller's precomputed
    buffer (page B, "Why Does a Single Kernel Even Matter for TTS?": a
    non-negative token id is looked up, anything else is taken precomputed from
    a buffer)."""
    if token >= 0:
        return W.embed[token].copy()
    if sentinel_rows is None:
        raise ValueError("negative id without a precomputed embedding buffer")
    return np.asarray(sentinel_rows[-token - 1], dtype=F64).copy()


class Decoder:
    """Step-by-step decoder with a bf16 KV cache: one token per forward.

    ``hidden[f]`` of a forward is ``[L+1][H]``: the input embedding followed by
    the residual stream after each layer (the layer-by-layer states page A,
    "Porting it to Qwen3-TTS-1.7B", diffs against a reference forward)."""

    def __init__(self, shape, weight_bits: dict, max_seq: int, weights: Optional[Weights] = None):
        self.s = shape if isinstance(shape, DecoderShape) else DecoderShape.from_dict(shape)
        self.W = weights if weights is not None else Weights(self.s, weight_bits)
        s = self.s
        self.max_seq = max_seq
        self.K = np.zeros((s.n_layers, s.n_kv_heads, max_seq, s.head_dim), dtype=F64)
        self.V = np.zeros_like(self.K)
        self.pos = 0
        self.last_id = 0

    def reset(self):
        self.pos = 0
        self.last_id = 0

    def forward_embedding(self, x, pos3=None):
        """Run one forward at slot ``self.pos`` from input embedding ``x``.
        ``pos3`` (three position streams) drives MRoPE; by default every stream
        is the slot index.  Returns ``(logits [V], hidden [L+1][H])``."""
        s, W = self.s, self.W
        P = self.pos
        if P >= self.max_seq:
            raise IndexError("KV cache full")
        d, Hq, Hkv = s.head_dim, s.n_q_heads, s.n_kv_heads
        pos = (P,) if pos3 is None else tuple(int(v) for v in pos3)
        if s.mrope_sections is None:
            pos = pos[:1]
        phi = rope_angles(pos, d, s.rope_theta, s.mrope_sections, s.mrope_interleaved)
        x = np.asarray(x, dtype=F64).copy()
        hidden = [x.copy()]
        for l, lw in enumerate(W.layers):
            # attention block
            h = rms_norm(x, lw["attn_norm"], s.rms_eps)
            q = (lw["wq"] @ h).reshape(Hq, d)
            k = (lw["wk"] @ h).reshape(Hkv, d)
            v = (lw["wv"] @ h).reshape(Hkv, d)
            q = rms_norm(q, lw["q_norm"], s.rms_eps)      # QK-norm per head, then rotary
            k = rms_norm(k, lw["k_norm"], s.rms_eps)
            q = rope_apply(q, phi)
            k = rope_apply(k, phi)
            self.K[l, :, P] = round_to_bf16(k)            # append to the bf16 cache
            self.V[l, :, P] = round_to_bf16(v)
            o = attention_decode(q, self.K[l, :, :P + 1], self.V[l, :, :P + 1], Hq, Hkv)
            x = x + lw["wo"] @ o.reshape(-1)
            # MLP block
            h = rms_norm(x, lw["mlp_norm"], s.rms_eps)
            u = silu(lw["w_gate"] @ h) * (lw["w_up"] @ h)
            x = x + lw["w_down"] @ u
            hidden.append(x.copy())
        logits = W.lm_head @ rms_norm(x, W.final_norm, s.rms_eps)
        self.pos = P + 1
        return logits, np.stack(hidden)

    def generate(self, in_ids, n_steps: int, sentinel_rows=None, pos3=None):
        """``len(in_ids) + n_steps`` forwards from the current cursor.

        Forward ``i < n_in`` consumes ``in_ids[i]``; later forwards consume the
        greedy id of the forward before (the first one, with no input, the
        decoder's last id).  ``pos3`` is ``[3][n_in + n_steps]`` or ``None``.
        Returns ``(ids [n], logits [n][V], hidden [n][L+1][H])``."""
        in_ids = [int(t) for t in np.asarray(in_ids, dtype=np.int64).reshape(-1)]
        n = len(in_ids) + int(n_steps)
        ids, all_logits, all_hidden = [], [], []
        prev = self.last_id
        for i in range(n):
            tok = in_ids[i] if i < len(in_ids) else prev
            x = _input_row(self.W, tok, sentinel_rows)
            p3 = None if pos3 is None else np.asarray(pos3)[:, i]
            logits, hid = self.forward_embedding(x, p3)
            prev = argmax_lowest(logits)
            ids.append(prev)
            all_logits.append(logits)
            all_hidden.append(hid)
        self.last_id = prev
        return np.asarray(ids, dtype=np.int32), np.stack(all_logits), np.stack(all_hidden)


def prefix_forward(shape, weight_bits: dict, tokens, sentinel_rows=None, pos3=None,
                   logits_for=None, weights: Optional[Weights] = None):
    """All positions of a prompt at once with a causal mask (no KV cache).

    A second, separately written path of the same model: positions ``0..T-1``
    are processed as matrices, keys and values are rounded to bf16 exactly as
    the cache would hold them, and position ``t`` attends to ``0..t``.
    ``logits_for`` lists the positions whose logits are wanted (default: all).
    Returns ``(logits [len(logits_for)][V], hidden [T][L+1][H], K, V)`` where
    ``K``, ``V`` ``[L][Hkv][T][d]`` are the bf16-rounded keys and values."""
    s = shape if isinstance(shape, DecoderShape) else DecoderShape.from_dict(shape)
    W = weights if weights is not None else Weights(s, weight_bits)
    toks = [int(t) for t in np.asarray(tokens, dtype=np.int64).reshape(-1)]
    T = len(toks)
    d, Hq, Hkv = s.head_dim, s.n_q_heads, s.n_kv_heads
    group = Hq // Hkv
    X = np.stack([_input_row(W, t, sentinel_rows) for t in toks])
    if pos3 is None:
        streams = np.tile(np.arange(T), (3, 1))
    else:
        streams = np.asarray(pos3)[:, :T]
    if s.mrope_sections is None:
        Phi = np.stack([rope_angles((streams[0, t],), d, s.rope_theta) for t in range(T)])
    else:
        Phi = np.stack([rope_angles(streams[:, t], d, s.rope_theta, s.mrope_sections, s.mrope_interleaved)
                        for t in range(T)])
    Phi = Phi[:, None, :]                                   # broadcast over heads
    causal = np.triu(np.full((T, T), -np.inf), k=1)
    hidden = [X.copy()]
    Ks, Vs = [], []
    for lw in W.layers:
        Hn = rms_norm(X, lw["attn_norm"], s.rms_eps)
        Q = (Hn @ lw["wq"].T).reshape(T, Hq, d)
        Kx = (Hn @ lw["wk"].T).reshape(T, Hkv, d)
        Vx = (Hn @ lw["wv"].T).reshape(T, Hkv, d)
        Q = rope_apply(rms_norm(Q, lw["q_norm"], s.rms_eps), Phi)
        Kx = round_to_bf16(rope_apply(rms_norm(Kx, lw["k_norm"], s.rms_eps), Phi))
        Vx = round_to_bf16(Vx)
        Ks.append(Kx.transpose(1, 0, 2))
        Vs.append(Vx.transpose(1, 0, 2))
        O = np.empty((T, Hq, d), dtype=F64)
        for j in range(Hq):
            g = j // group
            S = Q[:, j, :] @ Kx[:, g, :].T / np.sqrt(F64(d)) + causal
            A = np.exp(S - S.max(axis=1, keepdims=True))
            A /= A.sum(axis=1, keepdims=True)
            O[:, j, :] = A @ Vx[:, g, :]
        X = X + O.reshape(T, Hq * d) @ lw["wo"].T
        Hn = rms_norm(X, lw["mlp_norm"], s.rms_eps)
        U = silu(Hn @ lw["w_gate"].T) * (Hn @ lw["w_up"].T)
        X = X + U @ lw["w_down"].T
        hidden.append(X.copy())
    rows = list(range(T)) if logits_for is None else list(logits_for)
    logits = rms_norm(X[rows], W.final_norm, s.rms_eps) @ W.lm_head.T
    return logits, np.stack(hidden, axis=1), np.stack(Ks), np.stack(Vs)
