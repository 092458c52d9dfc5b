"""The phase-stamp reader (host arithmetic only) on synthetic stamps with known
durations."""
import numpy as np
import pytest

from persistent_transformer_megakernel_gb300 import trace as T


def _stamps(n_fwd=2, L=2, G=4):
    # CTA c enters phase gp at 10 us * gp + 0.1 us * c, waits 1 us for its
    # inputs (2 us in attention), computes 3 us, leaves 0.5 us later; CTAs 2
    # and 3 have no attention unit (stamp 1 never written: 0)
    nph = 5 * L + 1
    t = np.zeros((n_fwd, nph, G, 4), dtype=np.int64)
    for f in range(n_fwd):
        for ph in range(nph):
            gp = f * nph + ph
            attn = ph < 5 * L and ph % 5 == 1
            for c in range(G):
                s0 = 1_000_000 + 10_000 * gp + 100 * c
                wait = 2_000 if attn else 1_000
                t[f, ph, c] = [s0, s0 + wait, s0 + wait + 3_000, s0 + wait + 3_500]
                if attn and c >= 2:
                    t[f, ph, c, 1] = 0
    return t


def test_medians_per_kind_and_forward_time():
    L = 2
    s = T.summarize(_stamps(L=L), L)
    k = s["kinds"]
    for name in ("qkv", "o_proj", "gate_up", "down", "lm_head"):
        assert k[name]["wait_us"] == pytest.approx(1.0)
        assert k[name]["work_us"] == pytest.approx(3.0)
        assert k[name]["exit_us"] == pytest.approx(0.5)
        assert k[name]["in_phase_us"] == pytest.approx(4.5)
    # attention: stamp 1 only from the CTAs with a unit; the others still count for the rest
    assert k["attention"]["wait_us"] == pytest.approx(2.0)
    assert k["attention"]["work_us"] == pytest.approx(3.0)
    assert k["attention"]["in_phase_us"] == pytest.approx(5.5)
    # span: the slowest CTA's leave minus the previous phase's.  Phases start 10 us
    # apart; attention's 1 us longer wait adds 1 us to its span and takes it from O's
    for name in ("qkv", "gate_up", "down", "lm_head"):
        assert k[name]["span_us"] == pytest.approx(10.0)
    assert k["attention"]["span_us"] == pytest.approx(11.0)
    assert k["o_proj"]["span_us"] == pytest.approx(9.0)
    # a forward: first entry of its first phase to the last leave of its head phase
    nph = 5 * L + 1
    assert s["forward_us"] == pytest.approx([10.0 * (nph - 1) + 0.3 + 4.5] * 2)
    assert s["n_fwd"] == 2 and s["grid"] == 4
    assert "attention" in T.format_summary(s)


def test_missing_or_misshapen_stamps_are_refused():
    L = 2
    t = _stamps(L=L)
    with pytest.raises(ValueError):
        T.summarize(t, L + 1)                 # phase count does not match the layers
    bad = t.copy()
    bad[1, 3, 0, 0] = 0                        # a phase never entered (call aborted, or no buffer)
    with pytest.raises(ValueError):
        T.summarize(bad, L)
    with pytest.raises(ValueError):
        T.summarize(t[..., :3], L)
