"""Shared helpers of the parity tests: run the oracle and the CUDA path on the
same seeded inputs and compare with the stated tolerances.

Tolerances (logits and per-layer hidden states): max-abs <= 3e-2 and
relative L2 <= 1e-2; greedy ids bit-exact wherever the oracle's top-2 logit
gap exceeds 1e-2.
"""
import numpy as np

ATOL = 3e-2
REL_L2 = 1e-2
TIE_GAP = 1e-2


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_close(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite values"
    err = float(np.abs(got - want).max())
    rl = rel_l2(got, want)
    assert err <= ATOL and rl <= REL_L2, "%s: max-abs %.3g rel-L2 %.3g" % (what, err, rl)
    return err, rl


def clear_steps(logits_ref):
    """Forwards whose oracle top-2 gap exceeds the tie threshold."""
    top2 = np.sort(np.asarray(logits_ref), axis=1)[:, -2:]
    return (top2[:, 1] - top2[:, 0]) > TIE_GAP


def assert_ids(got, want, logits_ref, what="ids"):
    got = np.asarray(got)
    want = np.asarray(want)
    clear = clear_steps(logits_ref)
    bad = np.nonzero(clear & (got != want))[0]
    assert bad.size == 0, "%s differ at clear forwards %s" % (what, bad[:10])
    # where the oracle is near a tie, the GPU id must still be one of its top two
    near = np.nonzero(~clear)[0]
    for f in near:
        top = np.argsort(logits_ref[f])[-2:]
        assert got[f] in top, "%s: forward %d picked %d, oracle top-2 %s" % (what, f, got[f], top)


def first_near_tie(logits_ref):
    clear = clear_steps(logits_ref)
    idx = np.nonzero(~clear)[0]
    return int(idx[0]) if idx.size else len(clear)
