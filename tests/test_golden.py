"""Stored decodes of small cases (tests/golden/cases.json, written by
tests/golden/make_golden.py from the oracle; each case cites the section of
"GPU CTC Prefix Beam Search Decoder" it exercises).

* CPU: the stored inputs are the seeded draws their recipe names, and the
  oracle reproduces every stored output bit for bit (an oracle change that
  alters them must be justified by the pages).
* CPU: the cases that prune nothing equal the float64 enumeration of every
  alignment (tests/bruteforce.py): the same N best prefixes, scores within
  2e-5 relative.
* GPU: the CUDA path reproduces every stored output bit for bit.
"""
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden as G  # noqa: E402
from bruteforce import posteriors  # noqa: E402

with open(os.path.join(HERE, "golden", "cases.json")) as f:
    CASES = json.load(f)["cases"]
NAMES = [c["name"] for c in CASES]
NEG = float(np.finfo(np.float32).min)


def case(name):
    return next(c for c in CASES if c["name"] == name)


def stored(c):
    lp = np.asarray(c["log_prob"], np.float32)
    boost = None if "boost" not in c else [{int(k): v for k, v in row.items()} for row in c["boost"]]
    return lp, boost


def expected(c):
    return (np.asarray(c["tokens"], np.int32), np.asarray(c["lengths"], np.int32),
            np.asarray(c["scores"], np.float32))


def test_every_case_cites_the_pages():
    assert len(CASES) >= 10
    for c in CASES:
        assert c["cite"].startswith("section"), c["name"]


@pytest.mark.parametrize("name", NAMES)
def test_stored_inputs_are_the_recipes_draws(name):
    c = case(name)
    lp, _ = stored(c)
    np.testing.assert_array_equal(lp, G.inputs(tuple(c["input_recipe"])))


@pytest.mark.parametrize("name", NAMES)
def test_oracle_reproduces_stored_outputs(name):
    c = case(name)
    lp, boost = stored(c)
    tok, ln, sc = G.run(dict(c, boost=boost) if boost else c, lp)
    et, el, es = expected(c)
    np.testing.assert_array_equal(tok, et)
    np.testing.assert_array_equal(ln, el)
    np.testing.assert_array_equal(sc.view(np.uint32), es.view(np.uint32))


@pytest.mark.parametrize("name", [c["name"] for c in CASES if c.get("exact")])
def test_unpruned_cases_equal_enumeration(name):
    c = case(name)
    lp, boost = stored(c)
    et, el, es = expected(c)
    B, T, _ = lp.shape
    lens = c.get("lens", [T] * B)
    for b in range(B):
        exact = posteriors(lp[b, :lens[b]], c.get("blank", 0), cap=c.get("cap"), space=c.get("space"),
                           bonus=None if boost is None else boost[b])
        assert len(exact) <= c["beam"]  # every prefix fits the beam: nothing is pruned
        ranked = sorted(exact.items(), key=lambda kv: -kv[1])
        live = [i for i in range(c["nbest"]) if es[b, i] > NEG]
        assert len(live) == min(c["nbest"], len(exact))
        for i in live:
            pre = tuple(int(x) for x in et[b, i, :el[b, i]])
            assert pre in exact, (b, i, pre)
            assert abs(float(es[b, i]) - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre])), (b, i)
            # rank i by the exact scores, up to float32-level ties
            assert abs(exact[pre] - ranked[i][1]) <= 1e-4 * max(1.0, abs(ranked[i][1])), (b, i)


@pytest.mark.gpu
@pytest.mark.parametrize("name", NAMES)
def test_cuda_path_reproduces_stored_outputs(name):
    import torch
    from ctc_prefix_beam_gb300 import build
    from ctc_prefix_beam_gb300 import decoder as D
    build.build()
    c = case(name)
    lp, boost = stored(c)
    B, T, V = lp.shape
    kw = dict(beam=c["beam"], nbest=c["nbest"], blank_id=c.get("blank", 0), max_seq_len=c.get("cap", T),
              blank_threshold=c.get("thr", 1.0))
    if "space" in c:
        kw["space_id"] = c["space"]
    if boost:
        kw["max_boost"] = max(len(r) for r in boost)
    cfg = D.Config(**kw)
    x = torch.from_numpy(lp).cuda()
    if "mask" in c:  # the speech mask is a streaming input: every frame in one chunk
        st = D.StreamState(cfg, B, V)
        st.step_chunk(x, is_speech=torch.tensor(c["mask"], dtype=torch.uint8).cuda())
        got = st.read(out_len=T)
    else:
        lens = None if "lens" not in c else torch.tensor(c["lens"], dtype=torch.int32).cuda()
        got = D.decode_offline(cfg, x, lens, out_len=T, boost=boost)
    torch.cuda.synchronize()
    tok, ln, sc = (v.cpu().numpy() for v in got)
    et, el, es = expected(c)
    np.testing.assert_array_equal(tok, et)
    np.testing.assert_array_equal(ln, el)
    np.testing.assert_array_equal(sc.view(np.uint32), es.view(np.uint32))
