"""The oracle's pins catch plausible mistakes.  Each case plants one mistake
in a copy of oracle/ctcpb_oracle.cpp (a dropped term, a wrong path, a wrong
coefficient, an off-by-one, a reversed tie-break), compiles it into a temporary library, and runs
the independent pins on it: F = log(1 + e^-d) and its coefficients against
float64 and mpmath, lse against float64, and the unpruned
decode against the float64 enumeration of every alignment, plain and with a
cap, frame skipping, a word-boundary label and label bonuses ("GPU CTC Prefix
Beam Search Decoder", sections 3.1-3.5), and the hand-derived tie cases of
tests/tie_cases.py (sections 3.3, 3.4.4-3.4.6).  The real oracle passes every pin;
every mutant must fail at least one."""
import subprocess

import numpy as np
import pytest

import oracle as O
import tie_cases
from bruteforce import NEG32, posteriors, skip_augmented

NEG = np.float32(NEG32)


def log_softmax(x):
    x = np.asarray(x, np.float64)
    m = x.max(-1, keepdims=True)
    return (x - m - np.log(np.exp(x - m).sum(-1, keepdims=True))).astype(np.float32)


def frames(seed, T, V, blank_boost=0.0):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 1.5, size=(T, V))
    x[:, 0] += blank_boost
    return log_softmax(x)


def n_prefixes(V, T):
    return sum((V - 1) ** k for k in range(T + 1))


def unpruned_matches(lp, exact, **kw):
    """The decode with a beam holding every prefix equals the enumeration."""
    V = lp.shape[1]
    beam = min(128, max(V, n_prefixes(V, lp.shape[0])))
    tok, ln, sc = O.decode(lp[None], None, beam=beam, **kw)
    got = {}
    for n in range(ln.shape[1]):
        if sc[0, n] > NEG:
            got[tuple(int(v) for v in tok[0, n, :ln[0, n]])] = float(sc[0, n])
    if set(got) != set(exact):
        return False
    return all(abs(s - exact[p]) <= 2e-5 * max(1.0, abs(exact[p])) for p, s in got.items())


def pins_hold():
    """Every independent pin, as one boolean per pin."""
    res = {}
    # F = log(1 + e^-d) within 2 ulp of float64 on every segment, its
    # coefficients against mpmath's Taylor coefficients, lse within 4 ulp
    ds = np.concatenate([np.linspace(0.0, 23.99, 4001), [1e-6, 23.9999]]).astype(np.float32)
    f = O.F(ds).astype(np.float64)
    ref = np.log1p(np.exp(-ds.astype(np.float64)))
    res["F"] = bool(np.all(np.abs(f - ref) <= 2 * np.spacing(ref.astype(np.float32)).astype(np.float64)))
    from test_oracle_math import exact_coefficients
    res["F coefficients"] = bool(np.array_equal(O.F_coefficients(), exact_coefficients()))
    rng = np.random.default_rng(3)
    a = rng.uniform(-30, 0, 300).astype(np.float32)
    b = rng.uniform(-30, 0, 300).astype(np.float32)
    got = O.lse(a, b).astype(np.float64)
    ref = np.logaddexp(a.astype(np.float64), b.astype(np.float64))
    res["lse"] = bool(np.all(np.abs(got - ref) <= 4 * np.spacing(np.abs(ref).astype(np.float32))))
    # the decode against the enumeration of every alignment
    for i, (V, T, bb) in enumerate([(3, 5, 0.0), (4, 4, 1.0), (2, 6, 0.0), (3, 6, 2.0)]):
        lp = frames(10 + i, T, V, bb)
        res[f"plain V{V} T{T}"] = unpruned_matches(lp, posteriors(lp, 0))
    lp = frames(20, 5, 3)
    for cap in (1, 2):
        res[f"cap {cap}"] = unpruned_matches(lp, posteriors(lp, 0, cap=cap), cap=cap)
    for seed in range(6):  # skipped frames, a skipped lead-in among them
        lp = frames(30 + seed, 8, 3, blank_boost=2.5)
        lp[0] = log_softmax([9.0, 0.0, 0.0])
        aug, kept = skip_augmented(lp, 0, 0.9)
        if len(kept) <= 6:
            res[f"skip {seed}"] = unpruned_matches(lp, posteriors(aug, 0), thr=0.9)
    lp = frames(40, 4, 4)
    res["word boundary"] = unpruned_matches(lp, posteriors(lp, 0, space=2), space=2)
    lp = frames(41, 4, 3)
    bonus = {1: 1.25, 2: -0.5}
    res["bonus"] = unpruned_matches(lp, posteriors(lp, 0, bonus=bonus), boost=[bonus])
    # the tie-break rule and step 0's slot order, on hand-derived decodes
    res.update(tie_cases.check(lambda lp, beam, nbest, blank: O.decode(lp, None, beam=beam, nbest=nbest,
                                                                       blank=blank)))
    return res


MUTATIONS = {
    "repeat path takes lse(pb, pnb)": (
        "float ext = (!empty && c == last && c != space) ? add(v, pb[k]) : add(v, A[k]);",
        "float ext = add(v, A[k]);"),
    "stay path dropped": (
        "float bpnb = (!empty && !gap && last != space) ? add(rd(lpt + last), pnb[k]) : NEG;",
        "float bpnb = NEG;"),
    "fold takes lse(pb, pnb) on a repeat": (
        "float ext = rep ? add(v, pb[i]) : add(v, A[i]);",
        "float ext = add(v, A[i]);"),
    "fold dropped": ("bpnb = lse(bpnb, ext);", "(void)ext;"),
    "blank slot from pb only": ("float bpb = add(lpb, A[k]);", "float bpb = add(lpb, pb[k]);"),
    "no collapse before a step after a gap": (
        "if (gap) {\n          pb[k] = lse(pb[k], pnb[k]);", "if (false) {\n          pb[k] = lse(pb[k], pnb[k]);"),
    "no collapse of the winners after a gap": (
        "if (gap) {\n          h.pb = c.score;", "if (false) {\n          h.pb = c.score;"),
    "skipped lead-in seeds the non-blank slot": (
        "Hyp h{{ranked[k].second}, gap0 ? v : NEG, gap0 ? NEG : v};", "Hyp h{{ranked[k].second}, NEG, v};"),
    "cap off by one": ("if ((int)h.pre.size() >= a.cap) continue;", "if ((int)h.pre.size() > a.cap) continue;"),
    "space label repeats like any label": (
        "float ext = (!empty && c == last && c != space) ? add(v, pb[k]) : add(v, A[k]);",
        "float ext = (!empty && c == last) ? add(v, pb[k]) : add(v, A[k]);"),
    "F: Taylor polynomial about the segment start": ("const float u = d - ((float)k * 0.25f + 0.125f);",
                                                     "const float u = d - ((float)k * 0.25f);"),
    "F: the degree-5 term dropped": ("float p = c[5];", "float p = 0.0f * c[5];"),
    "F: wrong derivative recurrence": ("Q[i] -= i * P[i];", "Q[i] += i * P[i];"),
    "F: wrong factorial": ("fact *= n;", "fact *= n + 1;"),
    "lse: the smaller argument as the base": ("float m = std::fmax(a, b);", "float m = std::fmin(a, b);"),
    "ties: source slot descending": ("if (x.src != y.src) return x.src < y.src;",
                                     "if (x.src != y.src) return x.src > y.src;"),
    "ties: token descending": ("return x.tok < y.tok;", "return x.tok > y.tok;"),
    "ties: source slot and token both descending": (
        "if (x.src != y.src) return x.src < y.src;\n  return x.tok < y.tok;",
        "if (x.src != y.src) return x.src > y.src;\n  return x.tok > y.tok;"),
    "ties: the blank slot ranks after every label": [
        ("if (sc > NEG) cands.push_back(Cand{sc, k, a.blank, bpb, bpnb});",
         "if (sc > NEG) cands.push_back(Cand{sc, k, a.V, bpb, bpnb});"),
        ("if (c.tok != a.blank) h.pre.push_back(c.tok);",
         "if (c.tok != a.blank && c.tok != a.V) h.pre.push_back(c.tok);")],
    "step 0: the empty prefix in the first slot": (
        "if (lpb > NEG) beams.push_back(Hyp{{}, lpb, NEG});",
        "if (lpb > NEG) beams.insert(beams.begin(), Hyp{{}, lpb, NEG});"),
    "step 0: equal labels by id descending": ("return a.second < b.second;", "return a.second > b.second;"),
    "output: equal scores in reverse slot order": (
        "[&](int x, int y) { return sc[x] > sc[y]; }",
        "[&](int x, int y) { return sc[x] > sc[y] || (sc[x] == sc[y] && x > y); }"),
}


def build_variant(tmp_path, edits):
    src = open(O._SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    path = tmp_path / "mutant.cpp"
    path.write_text(src)
    lib = str(tmp_path / "libmutant.so")
    cmd = O.build_cmd()
    cmd[cmd.index(O._LIB)] = lib
    cmd[cmd.index(O._SRC)] = str(path)
    subprocess.run(cmd, check=True)
    return lib


def use_library(monkeypatch, path):
    monkeypatch.setattr(O, "_lib", None)
    monkeypatch.setattr(O, "build", lambda force=False: path)


def test_the_oracle_passes_every_pin():
    res = pins_hold()
    assert all(res.values()), [k for k, v in res.items() if not v]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(name, tmp_path, monkeypatch):
    edits = MUTATIONS[name]
    use_library(monkeypatch, build_variant(tmp_path, edits if isinstance(edits, list) else [edits]))
    try:
        res = pins_hold()
    except (AssertionError, ValueError, FloatingPointError):
        return  # the mutant broke an invariant outright
    failed = [k for k, v in res.items() if not v]
    assert failed, f"no pin caught: {name}"
