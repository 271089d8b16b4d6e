"""Hand-derived decodes whose result is decided by the tie-break rule.

The rule: candidates rank by score (descending), then source slot
(ascending), then token id (ascending), where the blank slot's token is
blank_id.  Step 0 orders its slots as the labels by (log-prob descending, id
ascending), then the empty prefix ("GPU CTC Prefix Beam Search Decoder",
sections 3.3 and 3.4.4-3.4.6).  The N-best output is a stable sort by score,
so hypotheses with equal scores keep their slot order.

Every frame below is built so that several candidates have bit-equal float32
scores (equal log-probabilities added to the same score), and the expected
N-best lists were worked out by hand from the rule, not taken from any
decoder.  Scores are checked two ways: equalities that hold bit for bit by
construction, and values against float64 sums of the kept paths'
probabilities.

`check(decode)` runs every case through `decode(lp [1, T, V] float32, beam,
nbest, blank) -> (tokens, lengths, scores)` and returns {case: passed}.
"""
from __future__ import annotations

import numpy as np

SCORE_ABS = 1e-5  # float64 expectation vs the float32 decode


def _f(x):
    return np.float32(np.log(x))


def _case_step0_order():
    # One frame.  Labels 1 and 3 tie with the blank (0.15); label 2 is best.
    # beam 4 seeds three labels: 2 (best), then 1 and 3 (equal log-probs, id
    # ascending); the empty prefix takes the last slot.  All but [2] score
    # log 0.15, so the stable output keeps [1], [3], [] in slot order.
    x, y, z = _f(0.15), _f(0.4), _f(0.05)
    lp = np.array([[[x, x, y, x, z]]], np.float32)
    want = [[2], [1], [3], []]
    scores = [float(y), float(x), float(x), float(x)]
    return dict(lp=lp, beam=4, nbest=4, blank=0, want=want, scores=scores, equal=[(1, 2), (2, 3)])


def _case_source_order():
    # Two uniform frames over V = 3 (blank 0), beam 3.  Step 0: [1], [2] (equal
    # log-probs, id ascending), then the empty prefix.  Frame 1: the blank slots
    # of [1] and [2] both absorb a fold from the empty prefix and tie at
    # Z = lse(2l, lse(2l, 2l)); [1,2], [2,1] and the empty prefix's blank slot
    # tie at 2l and rank by source slot, so [1,2] (source 0) takes the third
    # slot.
    l = _f(1.0 / 3.0)
    lp = np.full((1, 2, 3), l, np.float32)
    z = float(np.log(3.0 * (1.0 / 3.0) ** 2))
    two_l = float(np.float32(l) + np.float32(l))
    return dict(lp=lp, beam=3, nbest=3, blank=0, want=[[1], [2], [1, 2]], scores=[z, z, two_l],
                equal=[(0, 1)])


def _case_token_order():
    # Two uniform frames over V = 4 with blank id 1, beam 2.  Step 0: [0] (the
    # lowest id of three equal labels), then the empty prefix.  Frame 1: [0]'s
    # blank slot leads; [0,2], [0,3] tie with the empty prefix's blank slot and
    # [2], [3] at 2l; source 0 comes first, and within it token 2 before 3.
    l = _f(0.25)
    lp = np.full((1, 2, 4), l, np.float32)
    z = float(np.log(3.0 * 0.25 ** 2))
    two_l = float(np.float32(l) + np.float32(l))
    return dict(lp=lp, beam=2, nbest=2, blank=1, want=[[0], [0, 2]], scores=[z, two_l], equal=[])


def _case_blank_token(blank):
    # Three frames over V = 4, beam 2.  Frames 0 and 1 are blank-dominant
    # (blank 0.97, every label 0.01), so after step 1 the slots are: the empty
    # prefix (0.97^2), then [c0] (c0 = the lowest non-blank id).  Frame 2 is
    # uniform (0.25): [c0]'s blank slot, which absorbs the fold of the empty
    # prefix + c0, leads; the empty prefix's blank slot and its extensions by
    # every label but c0 then tie exactly, all from source 0, so the smallest
    # token wins -- and the blank slot's token is blank_id.
    pb, pl = 0.97, 0.01
    row = np.full(4, _f(pl), np.float32)
    row[blank] = _f(pb)
    lp = np.stack([row, row, np.full(4, _f(0.25), np.float32)])[None]
    labels = [c for c in range(4) if c != blank]
    c0 = labels[0]
    tie = min([blank] + labels[1:])
    second = [] if tie == blank else [tie]
    # float64 path sums after frame 1: [c0] holds pb*pl (blank after c0) +
    # pnb1, pnb1 = pl*pl (c0 held) + pl*pb (the folded empty prefix + c0).  At
    # frame 2 its blank slot collects all of [c0], its stay (pnb1) and the
    # folded empty prefix + c0 (pb*pb), each times 0.25.
    pnb1 = pl * pl + pl * pb
    first = float(np.log(0.25 * ((pb * pl + pnb1) + pnb1 + pb * pb)))
    sec = float(np.log(0.25 * pb * pb))
    return dict(lp=lp, beam=2, nbest=2, blank=blank, want=[[c0], second], scores=[first, sec], equal=[])


def cases():
    out = {"step-0 slot order": _case_step0_order(), "source-slot order": _case_source_order(),
           "token order": _case_token_order()}
    for blank in range(4):
        out[f"blank slot ranks as token {blank}"] = _case_blank_token(blank)
    return out


def outcome(case, tok, ln, sc) -> bool:
    want = case["want"]
    nb = case["nbest"]
    if tok.shape[:2] != (1, nb):
        return False
    for n, seq in enumerate(want):
        if int(ln[0, n]) != len(seq):
            return False
        if [int(v) for v in tok[0, n, :len(seq)]] != seq:
            return False
        if np.any(tok[0, n, len(seq):] != -1):
            return False
    s = sc[0].astype(np.float64)
    if np.max(np.abs(s[:len(want)] - np.asarray(case["scores"]))) > SCORE_ABS:
        return False
    return all(sc[0, i].view(np.int32) == sc[0, j].view(np.int32) for i, j in case["equal"])


def check(decode) -> dict:
    res = {}
    for name, c in cases().items():
        try:
            tok, ln, sc = decode(c["lp"], c["beam"], c["nbest"], c["blank"])
            res[f"tie: {name}"] = outcome(c, tok, ln, sc)
        except (ValueError, AssertionError):
            res[f"tie: {name}"] = False
    return res
