"""Seeded random sweep of the oracle against the float64 enumeration of every
alignment ("GPU CTC Prefix Beam Search Decoder", sections 3.1-3.5): tiny
vocabularies and lengths with every option combined -- the blank id, a cap,
frame skipping by threshold, a speech mask, a word-boundary label, label
bonuses -- decoded
with a beam wide enough to hold every reachable prefix, so the N best must be
the exact posteriors."""
import math

import numpy as np
import pytest

import oracle as O
from bruteforce import NEG32, posteriors, skip_augmented

NEG = np.float32(NEG32)


def draw(seed):
    rng = np.random.default_rng(5000 + seed)
    V = int(rng.integers(2, 5))
    T = int(rng.integers(1, 6 if V <= 3 else 5))
    blank = int(rng.integers(0, V)) if rng.random() < 0.4 else 0
    x = rng.normal(0.0, float(rng.choice([0.7, 1.5, 3.0])), size=(T, V))
    x[:, blank] += float(rng.choice([0.0, 1.5, 3.0]))
    x -= x.max(-1, keepdims=True)
    lp = (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32)
    opt = {}
    if rng.random() < 0.3:
        opt["cap"] = int(rng.integers(1, T + 1))
    if rng.random() < 0.3:
        opt["thr"] = float(rng.choice([0.5, 0.7, 0.9]))
    labels = [c for c in range(V) if c != blank]
    if rng.random() < 0.3 and labels:
        opt["space"] = int(rng.choice(labels))
    if rng.random() < 0.3 and labels:
        opt["bonus"] = {int(c): float(np.float32(rng.uniform(-2, 2))) for c in labels if rng.random() < 0.7}
    if rng.random() < 0.3:
        opt["mask"] = (rng.random(T) < 0.7).astype(np.uint8)
    return lp, blank, opt


@pytest.mark.parametrize("seed", range(400))
def test_unpruned_decode_equals_enumeration(seed):
    lp, blank, opt = draw(seed)
    T, V = lp.shape
    frames, kept = lp, list(range(T))
    if "thr" in opt or "mask" in opt:  # the kept frames: below the threshold and marked as speech
        kept = skip_augmented(lp, blank, opt.get("thr", 1.0))[1]
        if "mask" in opt:
            kept = [t for t in kept if opt["mask"][t]]
        frames, kept = skip_augmented(lp, blank, 1.0, kept=kept)
    exact = posteriors(frames, blank, cap=opt.get("cap"), space=opt.get("space"), bonus=opt.get("bonus"))
    if not kept:  # every frame skipped: the empty prefix with score 0
        exact = {(): 0.0}
    beam = min(128, max(V, sum((V - 1) ** k for k in range(len(kept) + 1))))
    tok, ln, sc = O.decode(lp[None], None, beam=beam, blank=blank, cap=opt.get("cap", T), thr=opt.get("thr", 1.0),
                           space=opt.get("space", -1), mask=None if "mask" not in opt else opt["mask"][None],
                           boost=None if "bonus" not in opt else [opt["bonus"]])
    got = {}
    for n in range(ln.shape[1]):
        if sc[0, n] > NEG:
            pre = tuple(int(v) for v in tok[0, n, :ln[0, n]])
            assert pre not in got, "duplicate prefix"
            assert blank not in pre
            got[pre] = float(sc[0, n])
    assert set(got) == set(exact), (seed, opt)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre])), (seed, opt, pre, s, exact[pre])
    scores = [float(v) for v in sc[0] if v > NEG]
    assert scores == sorted(scores, reverse=True)
    if "bonus" not in opt and "cap" not in opt:  # the posteriors of all prefixes sum to one
        assert math.isclose(sum(math.exp(v) for v in exact.values()), 1.0, rel_tol=1e-6)  # float32 inputs
