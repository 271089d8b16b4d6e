"""Float64 brute-force CTC posteriors by enumerating every alignment.

Independent of the oracle: no prefix recursion, no merging rule -- each
length-T alignment is collapsed (merge repeats, drop blanks) and its
probability exp(sum_t lp[t, a_t]) is added to its label sequence.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

NEG32 = float(np.finfo(np.float32).min)


def collapse(path, blank, space=None):
    """Merge repeats, drop blanks.  A word-boundary label ``space`` is never
    merged with itself: every frame of it is a token of its own."""
    out = []
    prev = None
    for a in path:
        if a != blank and (a != prev or a == space):
            out.append(a)
        prev = a
    return tuple(out)


def posteriors(frames, blank, cap=None, space=None, bonus=None):
    """{prefix: log P(prefix)} over all alignments of ``frames`` ([T, V], log-probs).

    Labels whose log-prob is <= -FLT_MAX are impossible and not enumerated.
    With ``cap``, alignments collapsing to more than ``cap`` labels are dropped.
    ``space``: the word-boundary label of ``collapse``.  ``bonus`` ({label:
    value}): each label of a prefix adds its bonus to the prefix's log score.
    """
    frames = np.asarray(frames, dtype=np.float64)
    T, V = frames.shape
    allowed = [[c for c in range(V) if frames[t, c] > NEG32] for t in range(T)]
    acc = {}
    for path in itertools.product(*allowed):
        lab = collapse(path, blank, space)
        if cap is not None and len(lab) > cap:
            continue
        lp = sum(frames[t, a] for t, a in enumerate(path))
        acc[lab] = acc.get(lab, 0.0) + math.exp(lp)
    bon = bonus or {}
    return {k: math.log(v) + sum(float(bon.get(c, 0.0)) for c in k) for k, v in acc.items() if v > 0.0}


def virtual_blank(V, blank):
    f = np.full(V, NEG32, dtype=np.float64)
    f[blank] = 0.0
    return f


def skip_augmented(frames, blank, thr, kept=None):
    """Kept frames of section 3.5 with a certain-blank frame before and after each
    kept frame that follows skipped ones (the collapsed-blank correction).
    ``kept`` (frame indices in order) overrides the threshold selection."""
    frames = np.asarray(frames, dtype=np.float32)
    T, V = frames.shape
    if kept is not None:
        kept = list(kept)
    elif thr >= 1.0:
        kept = list(range(T))
    elif thr <= 0.0:
        kept = []
    else:
        lt = np.float32(math.log(thr))
        kept = [t for t in range(T) if np.float32(max(frames[t, blank], NEG32)) < lt]
    out = []
    prev = -1
    for t in kept:
        gap = t > prev + 1
        if gap:
            out.append(virtual_blank(V, blank))
        out.append(frames[t].astype(np.float64))
        if gap:
            out.append(virtual_blank(V, blank))
        prev = t
    return np.array(out).reshape(-1, V), kept
