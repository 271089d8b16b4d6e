"""The oracle's tie-break, pinned by hand-derived decodes (tests/tie_cases.py).

Each case makes several candidates score bit-equal in float32 and states the
N-best that the rule "score descending, then source slot ascending, then token
id ascending; the blank slot's token is blank_id", with step 0's slot order
(labels by log-prob descending then id ascending, then the empty prefix), gives
("GPU CTC Prefix Beam Search Decoder", sections 3.3 and 3.4.4-3.4.6).  The
same cases run on the CUDA path in tests/test_gpu_ties.py."""
import pytest

import oracle as O
import tie_cases


def oracle_decode(lp, beam, nbest, blank):
    return O.decode(lp, None, beam=beam, nbest=nbest, blank=blank)


@pytest.mark.parametrize("name", sorted(tie_cases.cases()))
def test_oracle_breaks_ties_by_the_rule(name):
    c = tie_cases.cases()[name]
    tok, ln, sc = oracle_decode(c["lp"], c["beam"], c["nbest"], c["blank"])
    got = [[int(v) for v in tok[0, n, :ln[0, n]]] for n in range(c["nbest"])]
    assert got[:len(c["want"])] == c["want"]
    assert tie_cases.outcome(c, tok, ln, sc), (got, sc[0].tolist(), c["scores"])

