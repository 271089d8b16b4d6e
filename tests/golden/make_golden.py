"""Write tests/golden/cases.json: small decodes by the oracle, each one a case
the pages describe ("GPU CTC Prefix Beam Search Decoder", cited per case).

    python tests/golden/make_golden.py

Test infrastructure: calls only ``oracle/`` (inputs are seeded numpy draws
written into the file).  The stored values are checked three ways by
tests/test_golden.py: the oracle must reproduce them bit for bit, the
unpruned cases must equal the float64 enumeration of every alignment, and
the CUDA path must reproduce them bit for bit.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402


def log_softmax(x):
    x = np.asarray(x, np.float64)
    x = x - x.max(-1, keepdims=True)
    return (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32)


def draw(seed, B, T, V, blank=0, blank_boost=0.0, scale=1.5):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, scale, size=(B, T, V))
    x[:, :, blank] += blank_boost
    return log_softmax(x)


def one_hot_frames(seq, V, hi=0.0, lo=-6.0):
    """Frames whose label seq[t] has logit hi and every other label lo."""
    x = np.full((1, len(seq), V), lo)
    for t, c in enumerate(seq):
        x[0, t, c] = hi
    return log_softmax(x)


CASES = [
    dict(name="two_labels_pruned", cite="section 3.4.4-3.4.6 (top-beam selection prunes)",
         lp=("draw", 11, 1, 6, 3), beam=2, nbest=2),
    dict(name="unpruned_exact", cite="section 3 (prefix beam search; exact when nothing is pruned)",
         lp=("draw", 12, 2, 4, 3), beam=32, nbest=6, exact=True),
    dict(name="doubled_label", cite="section 3.2 (c == last extends only from pb: a, blank, a is 'aa')",
         lp=("onehot", [1, 0, 1], 2), beam=4, nbest=3, exact=True),
    dict(name="held_label", cite="section 3.2 (a label held over frames is one token)",
         lp=("onehot", [1, 1, 1, 2, 2], 3), beam=4, nbest=3),
    dict(name="threshold_skip", cite="section 3.5 (frames whose blank probability exceeds the threshold are skipped)",
         lp=("draw_blank", 13, 2, 8, 4, 2.5), beam=4, nbest=4, thr=0.6),
    dict(name="length_cap", cite="sections 11 and 13 (max_seq_len caps the hypothesis length)",
         lp=("draw", 14, 1, 6, 3), beam=6, nbest=6, cap=1, exact=True),
    dict(name="word_boundary", cite="sections 3.4.1-3.4.2 (space_id: every space frame is a token)",
         lp=("draw", 15, 1, 4, 4), beam=128, nbest=5, space=3, exact=True),
    dict(name="label_boost", cite="section 15's extension point with the per-utterance label boosting of 'GPU-Accelerated WFST "
              "Beam Search Decoder for CTC-based Speech Recognition'",
         lp=("draw", 16, 1, 4, 4), beam=128, nbest=5, boost=[{2: 1.5, 3: -0.75}], exact=True),
    dict(name="speech_mask", cite="section 8 (is_speech_mask: frames marked 0 bypass the decoder)",
         lp=("draw", 17, 2, 7, 3), beam=4, nbest=4, mask=[[1, 1, 0, 1, 0, 0, 1], [0, 1, 1, 1, 1, 0, 1]]),
    dict(name="beam_one", cite="section 3.3 (beam 1 seeds the best label, no empty slot)",
         lp=("draw", 18, 1, 5, 4), beam=1, nbest=1),
    dict(name="empty_and_short_rows", cite="section 13 (a row that never decodes gives the empty prefix, score 0)",
         lp=("draw", 19, 3, 4, 3), beam=3, nbest=3, lens=[0, 1, 4]),
    dict(name="blank_not_zero", cite="section 11 (blank_id is a parameter)",
         lp=("draw_blank_id", 20, 1, 5, 3, 2), beam=4, nbest=4, blank=2),
]


def inputs(spec):
    kind = spec[0]
    if kind == "draw":
        _, seed, B, T, V = spec
        return draw(seed, B, T, V)
    if kind == "draw_blank":
        _, seed, B, T, V, bb = spec
        return draw(seed, B, T, V, blank_boost=bb)
    if kind == "draw_blank_id":
        _, seed, B, T, V, blank = spec
        return draw(seed, B, T, V, blank=blank, blank_boost=1.0)
    if kind == "onehot":
        _, seq, V = spec
        return one_hot_frames(seq, V)
    raise ValueError(kind)


def run(case, lp):
    B, T, _ = lp.shape
    lens = None if "lens" not in case else np.asarray(case["lens"], np.int32)
    mask = None if "mask" not in case else np.asarray(case["mask"], np.uint8)
    return O.decode(lp, lens, beam=case["beam"], nbest=case["nbest"], blank=case.get("blank", 0),
                    cap=case.get("cap", T), thr=case.get("thr", 1.0), out_len=T, mask=mask,
                    space=case.get("space", -1), boost=case.get("boost"))


def main():
    out = []
    for c in CASES:
        lp = inputs(c["lp"])
        tok, ln, sc = run(c, lp)
        rec = {k: v for k, v in c.items() if k != "lp"}
        if "boost" in rec:
            rec["boost"] = [{str(k): float(v) for k, v in row.items()} for row in rec["boost"]]
        rec["input_recipe"] = list(c["lp"])
        rec["log_prob"] = [[[float(v) for v in fr] for fr in row] for row in lp]
        rec["tokens"] = tok.tolist()
        rec["lengths"] = ln.tolist()
        rec["scores"] = [[float(v) for v in row] for row in sc]
        out.append(rec)
    with open(os.path.join(HERE, "cases.json"), "w") as f:
        json.dump({"about": "oracle decodes of small cases; written by tests/golden/make_golden.py",
                   "cases": out}, f, indent=1)
        f.write("\n")
    print(f"{len(out)} cases")


if __name__ == "__main__":
    main()
