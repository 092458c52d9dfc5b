"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in the oracle's source (a dropped term, a wrong
sign, index or operand order, an off-by-one, a wrong rounding), loads the
changed source as a fresh module in place of ``oracle.decoder``, and runs the
pins of ``test_oracle_blocks.py`` and ``test_oracle_model.py`` against it: at
least one pin must fail.  The planted mistakes live only in memory, on the CPU;
the file on disk is never changed.
"""
import contextlib
import inspect
import types

import pytest

import oracle
import oracle.decoder as D
import test_oracle_blocks
import test_oracle_model

SRC = inspect.getsource(D)

# a planted mistake may make numpy divide by zero or overflow: expected, not an error
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

# (name, [(text in the oracle, replacement), ...]); every text occurs exactly once
MUTATIONS = [
    # bf16
    ("widening shift", [("<< np.uint32(16)", "<< np.uint32(15)")]),
    ("rounding truncates", [("q = np.rint(np.ldexp(x, 8 - e_eff))", "q = np.trunc(np.ldexp(x, 8 - e_eff))")]),
    ("rounding keeps 7 bits", [("q = np.rint(np.ldexp(x, 8 - e_eff))", "q = np.rint(np.ldexp(x, 7 - e_eff))"),
                               ("y = np.ldexp(q, e_eff - 8)", "y = np.ldexp(q, e_eff - 7)")]),
    # RMSNorm
    ("rmsnorm eps outside the root", [("return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)",
                                       "return x / (np.sqrt(ms) + eps) * np.asarray(w, dtype=F64)")]),
    ("rmsnorm drops the gain", [("return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)",
                                 "return x / np.sqrt(ms + eps)")]),
    ("rmsnorm (1 + w) gain", [("return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)",
                               "return x / np.sqrt(ms + eps) * (1.0 + np.asarray(w, dtype=F64))")]),
    ("rmsnorm sum instead of mean", [("ms = np.mean(x * x, axis=-1, keepdims=True)",
                                      "ms = np.sum(x * x, axis=-1, keepdims=True)")]),
    # SiLU
    ("silu sign", [("return z / (1.0 + np.exp(-z))", "return z / (1.0 + np.exp(z))")]),
    ("silu as sigmoid", [("return z / (1.0 + np.exp(-z))", "return 1.0 / (1.0 + np.exp(-z))")]),
    # rotary
    ("rope frequency exponent", [("omega = np.power(F64(theta), -2.0 * i / head_dim)",
                                  "omega = np.power(F64(theta), -1.0 * i / head_dim)")]),
    ("rope frequency index", [("omega = np.power(F64(theta), -2.0 * i / head_dim)",
                               "omega = np.power(F64(theta), -2.0 * (i + 1) / head_dim)")]),
    ("rope direction", [("[a * c - b * s, b * c + a * s]", "[a * c + b * s, b * c - a * s]")]),
    ("rope adjacent pairs", [("a, b = v[..., :half], v[..., half:]", "a, b = v[..., 0::2], v[..., 1::2]")]),
    ("mrope stream order", [("return np.repeat(np.arange(len(mrope_sections)), mrope_sections)",
                             "return np.repeat(np.arange(len(mrope_sections))[::-1], mrope_sections)")]),
    ("interleaved mrope phase", [("        r = i % 3\n", "        r = (i + 1) % 3\n")]),
    # attention
    ("attention unscaled", [("s = K[g] @ q[j] / np.sqrt(F64(d))", "s = K[g] @ q[j]")]),
    ("attention scaled by d", [("s = K[g] @ q[j] / np.sqrt(F64(d))", "s = K[g] @ q[j] / F64(d)")]),
    ("attention group mapping", [("    for j in range(n_q_heads):\n        g = j // group",
                                  "    for j in range(n_q_heads):\n        g = j % n_kv_heads")]),
    ("attention normalised by count", [("        a /= a.sum()\n", "        a /= len(a)\n")]),
    # head and greedy choice
    ("argmax highest index on ties", [("return int(np.argmax(x))", "return int(len(x) - 1 - np.argmax(x[::-1]))")]),
    ("tied flag inverted", [("        if shp.tied:\n", "        if not shp.tied:\n")]),
    # inputs
    ("sentinel row off by one", [("return np.asarray(sentinel_rows[-token - 1], dtype=F64).copy()",
                                  "return np.asarray(sentinel_rows[-token], dtype=F64).copy()")]),
    ("17-way sum drops the text row", [("        acc = acc + bf16_bits_to_f64(text_bits[text_ids[r]])\n", "")]),
    # step path
    ("step: rotary before QK-norm",
     [("            q = rms_norm(q, lw[\"q_norm\"], s.rms_eps)      # QK-norm per head, then rotary\n"
       "            k = rms_norm(k, lw[\"k_norm\"], s.rms_eps)\n"
       "            q = rope_apply(q, phi)\n"
       "            k = rope_apply(k, phi)\n",
       "            q = rope_apply(q, phi)\n"
       "            k = rope_apply(k, phi)\n"
       "            q = rms_norm(q, lw[\"q_norm\"], s.rms_eps)\n"
       "            k = rms_norm(k, lw[\"k_norm\"], s.rms_eps)\n")]),
    ("step: key cached unrounded", [("self.K[l, :, P] = round_to_bf16(k)", "self.K[l, :, P] = k")]),
    ("step: value cached unrounded", [("self.V[l, :, P] = round_to_bf16(v)", "self.V[l, :, P] = v")]),
    ("step: attention residual dropped", [("x = x + lw[\"wo\"] @ o.reshape(-1)", "x = lw[\"wo\"] @ o.reshape(-1)")]),
    ("step: MLP residual dropped", [("x = x + lw[\"w_down\"] @ u", "x = lw[\"w_down\"] @ u")]),
    ("step: gate and up swapped", [("u = silu(lw[\"w_gate\"] @ h) * (lw[\"w_up\"] @ h)",
                                    "u = silu(lw[\"w_up\"] @ h) * (lw[\"w_gate\"] @ h)")]),
    ("step: post-attention norm gain", [("h = rms_norm(x, lw[\"mlp_norm\"], s.rms_eps)",
                                         "h = rms_norm(x, lw[\"attn_norm\"], s.rms_eps)")]),
    ("step: final norm dropped", [("logits = W.lm_head @ rms_norm(x, W.final_norm, s.rms_eps)",
                                   "logits = W.lm_head @ x")]),
    ("step: newest slot not attended", [("self.K[l, :, :P + 1], self.V[l, :, :P + 1]",
                                         "self.K[l, :, :max(P, 1)], self.V[l, :, :max(P, 1)]")]),
    ("step: greedy feedback from the cursor's id", [("tok = in_ids[i] if i < len(in_ids) else prev",
                                                     "tok = in_ids[i] if i < len(in_ids) else self.last_id")]),
    # all-positions path
    ("prefix: mask admits the next position", [("causal = np.triu(np.full((T, T), -np.inf), k=1)",
                                                "causal = np.triu(np.full((T, T), -np.inf), k=2)")]),
    ("prefix: group mapping", [("            g = j // group\n            S = Q",
                                "            g = j % Hkv\n            S = Q")]),
    ("prefix: value cached unrounded", [("        Vx = round_to_bf16(Vx)\n", "")]),
    # the same mistake in both paths (their agreement cannot catch it)
    ("both: post-attention norm gain", [("h = rms_norm(x, lw[\"mlp_norm\"], s.rms_eps)",
                                         "h = rms_norm(x, lw[\"attn_norm\"], s.rms_eps)"),
                                        ("Hn = rms_norm(X, lw[\"mlp_norm\"], s.rms_eps)",
                                         "Hn = rms_norm(X, lw[\"attn_norm\"], s.rms_eps)")]),
    ("both: rotary before QK-norm",
     [("            q = rms_norm(q, lw[\"q_norm\"], s.rms_eps)      # QK-norm per head, then rotary\n"
       "            k = rms_norm(k, lw[\"k_norm\"], s.rms_eps)\n"
       "            q = rope_apply(q, phi)\n"
       "            k = rope_apply(k, phi)\n",
       "            q = rope_apply(q, phi)\n"
       "            k = rope_apply(k, phi)\n"
       "            q = rms_norm(q, lw[\"q_norm\"], s.rms_eps)\n"
       "            k = rms_norm(k, lw[\"k_norm\"], s.rms_eps)\n"),
      ("Q = rope_apply(rms_norm(Q, lw[\"q_norm\"], s.rms_eps), Phi)",
       "Q = rms_norm(rope_apply(Q, Phi), lw[\"q_norm\"], s.rms_eps)"),
      ("Kx = round_to_bf16(rope_apply(rms_norm(Kx, lw[\"k_norm\"], s.rms_eps), Phi))",
       "Kx = round_to_bf16(rms_norm(rope_apply(Kx, Phi), lw[\"k_norm\"], s.rms_eps))")]),
    ("both: query gain on keys", [("k = rms_norm(k, lw[\"k_norm\"], s.rms_eps)",
                                   "k = rms_norm(k, lw[\"q_norm\"], s.rms_eps)"),
                                  ("rms_norm(Kx, lw[\"k_norm\"], s.rms_eps)",
                                   "rms_norm(Kx, lw[\"q_norm\"], s.rms_eps)")]),
    ("both: values cached unrounded", [("self.V[l, :, P] = round_to_bf16(v)", "self.V[l, :, P] = v"),
                                       ("        Vx = round_to_bf16(Vx)\n", "")]),
    ("both: keys cached unrounded", [("self.K[l, :, P] = round_to_bf16(k)", "self.K[l, :, P] = k"),
                                     ("Kx = round_to_bf16(rope_apply(rms_norm(Kx, lw[\"k_norm\"], s.rms_eps), Phi))",
                                      "Kx = rope_apply(rms_norm(Kx, lw[\"k_norm\"], s.rms_eps), Phi)")]),
    ("both: key and value projections swapped",
     [("k = (lw[\"wk\"] @ h).reshape(Hkv, d)", "k = (lw[\"wv\"] @ h).reshape(Hkv, d)"),
      ("v = (lw[\"wv\"] @ h).reshape(Hkv, d)", "v = (lw[\"wk\"] @ h).reshape(Hkv, d)"),
      ("Kx = (Hn @ lw[\"wk\"].T).reshape(T, Hkv, d)", "Kx = (Hn @ lw[\"wv\"].T).reshape(T, Hkv, d)"),
      ("Vx = (Hn @ lw[\"wv\"].T).reshape(T, Hkv, d)", "Vx = (Hn @ lw[\"wk\"].T).reshape(T, Hkv, d)")]),
    ("both: SiLU on the up projection", [("u = silu(lw[\"w_gate\"] @ h) * (lw[\"w_up\"] @ h)",
                                          "u = silu(lw[\"w_up\"] @ h) * (lw[\"w_gate\"] @ h)"),
                                         ("U = silu(Hn @ lw[\"w_gate\"].T) * (Hn @ lw[\"w_up\"].T)",
                                          "U = silu(Hn @ lw[\"w_up\"].T) * (Hn @ lw[\"w_gate\"].T)")]),
    ("both: eps dropped from the layer and final norms",
     [("h = rms_norm(x, lw[\"attn_norm\"], s.rms_eps)", "h = rms_norm(x, lw[\"attn_norm\"], 0.0)"),
      ("h = rms_norm(x, lw[\"mlp_norm\"], s.rms_eps)", "h = rms_norm(x, lw[\"mlp_norm\"], 0.0)"),
      ("logits = W.lm_head @ rms_norm(x, W.final_norm, s.rms_eps)",
       "logits = W.lm_head @ rms_norm(x, W.final_norm, 0.0)"),
      ("Hn = rms_norm(X, lw[\"attn_norm\"], s.rms_eps)", "Hn = rms_norm(X, lw[\"attn_norm\"], 0.0)"),
      ("Hn = rms_norm(X, lw[\"mlp_norm\"], s.rms_eps)", "Hn = rms_norm(X, lw[\"mlp_norm\"], 0.0)"),
      ("logits = rms_norm(X[rows], W.final_norm, s.rms_eps) @ W.lm_head.T",
       "logits = rms_norm(X[rows], W.final_norm, 0.0) @ W.lm_head.T")]),
    ("both: eps dropped from QK-norm",
     [("q = rms_norm(q, lw[\"q_norm\"], s.rms_eps)", "q = rms_norm(q, lw[\"q_norm\"], 0.0)"),
      ("k = rms_norm(k, lw[\"k_norm\"], s.rms_eps)", "k = rms_norm(k, lw[\"k_norm\"], 0.0)"),
      ("rms_norm(Q, lw[\"q_norm\"], s.rms_eps)", "rms_norm(Q, lw[\"q_norm\"], 0.0)"),
      ("rms_norm(Kx, lw[\"k_norm\"], s.rms_eps)", "rms_norm(Kx, lw[\"k_norm\"], 0.0)")]),
    ("both: final norm dropped", [("logits = W.lm_head @ rms_norm(x, W.final_norm, s.rms_eps)", "logits = W.lm_head @ x"),
                                  ("logits = rms_norm(X[rows], W.final_norm, s.rms_eps) @ W.lm_head.T",
                                   "logits = X[rows] @ W.lm_head.T")]),
]


def _pins():
    fns = []
    for mod in (test_oracle_blocks, test_oracle_model):
        for name, fn in inspect.getmembers(mod, inspect.isfunction):
            if name.startswith("test_") and fn.__module__ == mod.__name__ \
                    and not inspect.signature(fn).parameters:
                fns.append((mod.__name__ + "." + name, fn))
    return fns


@contextlib.contextmanager
def _planted(edits):
    src = SRC
    for old, new in edits:
        assert src.count(old) == 1, "mutation text must occur exactly once: %r" % old[:60]
        src = src.replace(old, new)
    mod = types.ModuleType(D.__name__)
    mod.__file__ = D.__file__
    exec(compile(src, D.__file__, "exec"), mod.__dict__)
    names = [n for n in vars(oracle) if not n.startswith("_") and n in mod.__dict__]
    saved = {n: getattr(oracle, n) for n in names}
    saved_mod = oracle.decoder
    try:
        for n in names:
            setattr(oracle, n, getattr(mod, n))
        oracle.decoder = mod
        yield
    finally:
        for n, v in saved.items():
            setattr(oracle, n, v)
        oracle.decoder = saved_mod


def test_pins_pass_on_the_unchanged_oracle_source():
    # the reloaded source with no edit is the oracle itself: every pin passes
    with _planted([]):
        for name, fn in _pins():
            fn()


@pytest.mark.parametrize("name,edits", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(name, edits):
    caught = None
    with _planted(edits):
        for pin, fn in _pins():
            try:
                fn()
            except Exception:  # an assertion or the error the mistake raises
                caught = pin
                break
    assert caught is not None, "no pin fails with the planted mistake: " + name
