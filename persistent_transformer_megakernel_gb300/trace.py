"""Reading the decode kernel's phase stamps (``mk_decode_opts.trace``).

With a trace buffer the kernel's thread 0 of every CTA writes four
``%globaltimer`` stamps (nanoseconds) per phase of every forward, at
``trace[f][phase][cta][k]``:

* ``k = 0``: the CTA enters the phase;
* ``k = 1``: its inputs are in registers (GEMV phases: the polled activation
  slice; attention: the group's queries normed and rotated and the new key and
  value appended).  CTAs without an attention unit in a forward never write it;
* ``k = 2``: its tiles and epilogue are done (outputs published);
* ``k = 3``: it leaves the phase (the LM head phase: after the grid barrier
  that closes the forward).

Phases per forward: ``5 * n_layers`` layer phases (QKV, attention, O, gate/up,
down for each layer) and the LM head.  This module allocates the buffer and
turns the stamps into per-phase times: how long a CTA waits for its inputs,
computes, and takes to leave, and the span of each phase on the critical path
(how far the slowest CTA advanced).  It is host-side arithmetic only.
"""
from __future__ import annotations

import numpy as np

#: the layer phases in order, then the head
KINDS = ("qkv", "attention", "o_proj", "gate_up", "down", "lm_head")


def buffer(dec, n_fwd: int):
    """A zeroed device buffer for ``n_fwd`` traced forwards of ``dec`` (a
    ``Decoder``): int64 ``[n_fwd][5 L + 1][grid][4]``, passed as ``trace=``."""
    import torch
    grid = dec.info()["grid"]
    nph = 5 * dec.shape["n_layers"] + 1
    return torch.zeros((n_fwd, nph, grid, 4), dtype=torch.int64, device=dec.device)


def _kind_of_phase(nph: int) -> np.ndarray:
    k = np.arange(nph) % 5
    k[nph - 1] = 5
    return k


def summarize(trace, n_layers: int) -> dict:
    """Per-kind medians (microseconds) over forwards, layers and CTAs, and the
    forward times.  ``trace`` is the buffer after the call (tensor or array).

    For each kind: ``wait_us`` (enter -> inputs in registers), ``work_us``
    (inputs -> tiles and epilogue done), ``exit_us`` (done -> leave),
    ``in_phase_us`` (enter -> leave) and ``span_us`` (the latest leave of the
    phase minus the latest leave of the phase before, the first phase of the
    call excluded).  ``forward_us``: per forward, the latest leave of its head
    phase minus the earliest entry of its first phase."""
    t = trace.cpu().numpy() if hasattr(trace, "cpu") else np.asarray(trace)
    t = t.astype(np.int64)
    if t.ndim != 4 or t.shape[3] != 4:
        raise ValueError("trace must be [n_fwd][5 L + 1][grid][4]")
    n_fwd, nph, grid, _ = t.shape
    if nph != 5 * n_layers + 1:
        raise ValueError("trace has %d phases per forward, expected %d" % (nph, 5 * n_layers + 1))
    s = t.astype(np.float64)
    s0, s1, s2, s3 = s[..., 0], s[..., 1], s[..., 2], s[..., 3]
    if np.any(s0 <= 0) or np.any(s2 < s0) or np.any(s3 < s2):
        raise ValueError("stamps missing or out of order (was the buffer passed to the call?)")
    has1 = (s1 >= s0) & (s1 <= s2)                 # stamp 1 written in this call
    wait = np.where(has1, s1 - s0, np.nan)
    work = np.where(has1, s2 - s1, np.nan)
    exit_ = s3 - s2
    inside = s3 - s0
    last_leave = s3.max(axis=2).reshape(-1)        # [n_fwd * nph]
    span = np.full(n_fwd * nph, np.nan)
    span[1:] = np.diff(last_leave)
    span = span.reshape(n_fwd, nph)
    kind = _kind_of_phase(nph)
    out = {}
    for ki, name in enumerate(KINDS):
        sel = kind == ki
        out[name] = {
            "wait_us": float(np.nanmedian(wait[:, sel])) / 1e3 if np.any(~np.isnan(wait[:, sel])) else None,
            "work_us": float(np.nanmedian(work[:, sel])) / 1e3 if np.any(~np.isnan(work[:, sel])) else None,
            "exit_us": float(np.median(exit_[:, sel])) / 1e3,
            "in_phase_us": float(np.median(inside[:, sel])) / 1e3,
            "span_us": float(np.nanmedian(span[:, sel])) / 1e3 if np.any(~np.isnan(span[:, sel])) else None,
        }
    fwd = (s3[:, nph - 1, :].max(axis=1) - s0[:, 0, :].min(axis=1)) / 1e3
    return {"kinds": out, "forward_us": fwd.tolist(), "forward_us_median": float(np.median(fwd)),
            "n_fwd": int(n_fwd), "grid": int(grid)}


def format_summary(summ: dict) -> str:
    """A small text table of ``summarize``'s result."""
    def f(v):
        return "   -   " if v is None else "%7.2f" % v
    lines = ["%-10s %7s %7s %7s %9s %7s" % ("phase", "wait", "work", "exit", "in-phase", "span")]
    for name in KINDS:
        k = summ["kinds"][name]
        lines.append("%-10s %s %s %s %s   %s" % (name, f(k["wait_us"]), f(k["work_us"]), f(k["exit_us"]),
                                                 f(k["in_phase_us"]), f(k["span_us"])))
    lines.append("forward: median %.1f us over %d forwards, %d CTAs (times in us, medians)"
                 % (summ["forward_us_median"], summ["n_fwd"], summ["grid"]))
    return "\n".join(lines)
