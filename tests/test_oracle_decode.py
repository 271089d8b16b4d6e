"""Pins of the oracle decoder against things other than itself.

* brute force: with a beam wide enough to hold every reachable prefix, every
  output score equals log of the float64 sum over all alignments collapsing to
  that prefix ("GPU CTC Prefix Beam Search Decoder", sections 3.1-3.4), also
  under a token cap and under frame skipping (section 3.5 / 3.4.5 collapse,
  which equals a certain-blank frame inserted before and after each kept frame
  that follows skipped ones);
* pruning: a pruned beam can only lose alignment mass, so every score is at
  most the exact posterior of its prefix;
* closed forms: the V=2 posteriors written out by hand; one-hot frames decode
  to the collapsed argmax path with score 0; unpruned posteriors sum to 1;
* invariants: distinct prefixes, no blank token, length <= cap, sorted scores;
* frame selection and per-frame ranked labels against numpy routines.
"""
import math

import numpy as np
import pytest

from bruteforce import NEG32, collapse, posteriors, skip_augmented

NEG = np.float32(NEG32)


def log_softmax(x):
    x = np.asarray(x, np.float64)
    m = x.max(-1, keepdims=True)
    return (x - m - np.log(np.exp(x - m).sum(-1, keepdims=True))).astype(np.float32)


def random_frames(rng, T, V, scale, blank, blank_boost=0.0):
    x = rng.normal(0.0, scale, size=(T, V))
    x[:, blank] += blank_boost
    return log_softmax(x)


def n_prefixes(V, T, cap=None):
    """Number of label sequences of length <= min(T, cap) over V-1 labels."""
    L = T if cap is None else min(T, cap)
    return sum((V - 1) ** k for k in range(L + 1))


def decoded(oracle, lp, **kw):
    tok, ln, sc = oracle.decode(lp[None], None, **kw)
    out = {}
    for n in range(ln.shape[1]):
        if sc[0, n] > NEG:
            pre = tuple(int(v) for v in tok[0, n, :ln[0, n]])
            assert pre not in out, "duplicate prefix in the beam"
            out[pre] = float(sc[0, n])
    return out, tok, ln, sc


CASES = [  # (V, T, scale, blank, blank_boost)
    (2, 1, 1.0, 0, 0.0), (2, 6, 1.0, 0, 0.0), (2, 7, 3.0, 1, 1.0),
    (3, 1, 1.0, 0, 0.0), (3, 4, 2.0, 0, 0.0), (3, 5, 0.5, 2, 0.0), (3, 6, 1.0, 1, 2.0),
    (4, 3, 1.0, 0, 0.0), (4, 4, 2.0, 3, -1.0), (4, 4, 0.2, 0, 0.0), (5, 3, 1.5, 0, 0.0),
]


@pytest.mark.parametrize("V,T,scale,blank,boost", CASES)
def test_unpruned_equals_brute_force(oracle, V, T, scale, blank, boost):
    rng = np.random.default_rng(1000 + 7 * V + T)
    lp = random_frames(rng, T, V, scale, blank, boost)
    exact = posteriors(lp, blank)
    beam = max(V, n_prefixes(V, T))
    got, *_ = decoded(oracle, lp, beam=beam, blank=blank)
    assert set(got) == set(exact)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre])), (pre, s, exact[pre])


@pytest.mark.parametrize("V,T,cap", [(3, 6, 1), (3, 6, 2), (4, 5, 2), (2, 7, 2), (3, 5, 3)])
def test_cap_equals_restricted_brute_force(oracle, V, T, cap):
    rng = np.random.default_rng(V * 100 + T * 10 + cap)
    lp = random_frames(rng, T, V, 1.5, 0)
    exact = posteriors(lp, 0, cap=cap)
    beam = max(V, n_prefixes(V, T, cap))
    got, tok, ln, sc = decoded(oracle, lp, beam=beam, cap=cap)
    assert set(got) == set(exact)
    assert (ln <= cap).all()
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre]))


@pytest.mark.parametrize("seed", range(6))
def test_skipping_equals_virtual_blank_brute_force(oracle, seed):
    rng = np.random.default_rng(50 + seed)
    V, T = 3, 9
    x = rng.normal(0.0, 1.0, size=(T, V))
    # make a random subset of frames blank-dominant so they are skipped
    dom = rng.random(T) < 0.45
    x[dom, 0] += 9.0
    lp = log_softmax(x)
    thr = 0.99
    aug, kept = skip_augmented(lp, 0, thr)
    assert 0 < len(kept) < T
    exact = posteriors(aug, 0)
    beam = max(V, n_prefixes(V, len(kept)))
    got, *_ = decoded(oracle, lp, beam=beam, thr=thr)
    assert set(got) == set(exact)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre]))


def test_leading_skip_seeds_blank_slot(oracle):
    """A skipped lead-in puts every seeded label's mass in its blank slot: a
    label repeated on the next kept frame then decodes as a doubled token."""
    V = 3
    lp = log_softmax(np.array([[12.0, 0, 0], [0, 5.0, 0], [0, 5.0, 0]]))
    aug, kept = skip_augmented(lp, 0, 0.99)
    assert kept == [1, 2]
    exact = posteriors(aug, 0)
    got, *_ = decoded(oracle, lp, beam=8, thr=0.99)
    assert set(got) == set(exact)
    best = max(got, key=got.get)
    assert best == (1, 1)


@pytest.mark.parametrize("V,T,beam,seed", [(4, 7, 2, 0), (4, 7, 3, 1), (5, 6, 4, 2), (3, 9, 2, 3),
                                           (4, 8, 5, 4), (6, 5, 3, 5)])
def test_pruned_scores_bounded_by_exact(oracle, V, T, beam, seed):
    rng = np.random.default_rng(seed)
    lp = random_frames(rng, T, V, 1.5, 0, 1.0)
    exact = posteriors(lp, 0)
    got, tok, ln, sc = decoded(oracle, lp, beam=beam)
    assert 1 <= len(got) <= beam
    for pre, s in got.items():
        assert pre in exact
        assert s <= exact[pre] + 2e-5 * max(1.0, abs(exact[pre]))


def test_two_symbol_hand_computed(oracle):
    """V=2 (blank=0, label a=1), T=3, posteriors written out by hand."""
    p = np.array([[0.6, 0.4], [0.3, 0.7], [0.8, 0.2]])
    lp = np.log(p).astype(np.float32)
    b = p[:, 0].astype(np.float64)
    a = p[:, 1].astype(np.float64)
    P_empty = b[0] * b[1] * b[2]
    # "a": aaa, aab, abb, baa, bba, bab? (b a b) -> a; aba -> aa (excluded); abb; bba
    P_a = (a[0] * a[1] * a[2] + a[0] * a[1] * b[2] + a[0] * b[1] * b[2] + b[0] * a[1] * a[2]
           + b[0] * b[1] * a[2] + b[0] * a[1] * b[2])
    P_aa = a[0] * b[1] * a[2]
    got, *_ = decoded(oracle, lp, beam=4)
    assert set(got) == {(), (1,), (1, 1)}
    assert abs(got[()] - math.log(P_empty)) < 1e-6
    assert abs(got[(1,)] - math.log(P_a)) < 1e-6
    assert abs(got[(1, 1)] - math.log(P_aa)) < 1e-6
    assert abs(P_empty + P_a + P_aa - 1.0) < 1e-12


@pytest.mark.parametrize("blank", [0, 4])
def test_one_hot_path(oracle, blank):
    rng = np.random.default_rng(9)
    V, T = 5, 40
    path = rng.integers(0, V, size=T)
    lp = np.full((T, V), NEG, np.float32)
    lp[np.arange(T), path] = 0.0
    got, tok, ln, sc = decoded(oracle, lp, beam=3, blank=blank)
    best = tuple(int(v) for v in tok[0, 0, :ln[0, 0]])
    assert best == collapse(path.tolist(), blank)
    assert sc[0, 0] == 0.0
    assert (sc[0, 1:] == NEG).all() and (ln[0, 1:] == 0).all()


@pytest.mark.parametrize("V,T", [(3, 10), (4, 5), (2, 15)])
def test_unpruned_mass_sums_to_one(oracle, V, T):
    rng = np.random.default_rng(V + T)
    lp = random_frames(rng, T, V, 2.0, 0)
    beam = max(V, n_prefixes(V, T))
    if beam > 4096:
        pytest.skip("too many prefixes")
    got, *_ = decoded(oracle, lp, beam=beam)
    total = sum(math.exp(s) for s in got.values())
    assert abs(total - 1.0) < 1e-4


def test_invariants_tiny_workload(oracle):
    from ctc_prefix_beam_gb300 import synth
    w = synth.WORKLOADS["tiny"]
    lp, lens = synth.gen_batch(w)
    for cap in (None, 5):
        tok, ln, sc = oracle.decode(lp, lens, beam=w.beam, cap=cap)
        for b in range(lp.shape[0]):
            seen = set()
            for n in range(w.nbest):
                if sc[b, n] <= NEG:
                    assert ln[b, n] == 0 and (tok[b, n] == -1).all()
                    continue
                row = tok[b, n]
                pre = tuple(row[: min(ln[b, n], row.size)])
                assert w.blank_id not in pre
                assert pre not in seen
                seen.add(pre)
                if cap is not None:
                    assert ln[b, n] <= cap
            assert (np.diff(sc[b]) <= 0).all()


def test_rows_without_frames(oracle):
    lp = np.zeros((3, 4, 5), np.float32)
    lp[...] = np.log(0.2)
    lens = np.array([0, 4, 0], np.int32)
    tok, ln, sc = oracle.decode(lp, lens, beam=3, thr=1.0)
    for b in (0, 2):
        assert sc[b, 0] == 0.0 and ln[b, 0] == 0
        assert (sc[b, 1:] == NEG).all()
    # a threshold <= 0 keeps no frame
    tok, ln, sc = oracle.decode(lp, lens, beam=3, thr=0.0)
    assert (sc[:, 0] == 0.0).all() and (sc[:, 1:] == NEG).all()


def test_truncated_output_reports_full_length(oracle):
    rng = np.random.default_rng(5)
    lp = random_frames(rng, 30, 6, 3.0, 0)
    tok_full, ln_full, sc_full = oracle.decode(lp[None], None, beam=4)
    tok, ln, sc = oracle.decode(lp[None], None, beam=4, out_len=3)
    assert np.array_equal(ln, ln_full)
    assert np.array_equal(sc, sc_full)
    assert np.array_equal(tok, tok_full[:, :, :3])


@pytest.mark.parametrize("thr", [0.98, 0.5, 1.0, 0.0, 2.0])
def test_frame_selection_matches_numpy(oracle, thr):
    rng = np.random.default_rng(11)
    B, T, V = 4, 37, 6
    lp = random_frames(rng, B * T, V, 2.0, 0, 2.0).reshape(B, T, V)
    lp[1, 3, 0] = -np.inf
    lens = np.array([37, 20, 0, 5], np.int32)
    sel, nsel = oracle.select_frames(lp, lens, 0, thr)
    for b in range(B):
        col = lp[b, : lens[b], 0]
        if thr >= 1:
            want = np.arange(lens[b])
        elif thr <= 0:
            want = np.arange(0)
        else:
            want = np.nonzero(np.maximum(col, NEG) < np.float32(math.log(thr)))[0]
        assert nsel[b] == len(want)
        assert np.array_equal(sel[b, : nsel[b]], want)


def test_frame_lists_match_lexsort(oracle):
    rng = np.random.default_rng(12)
    R, V, C = 64, 300, 22
    rows = rng.normal(-5, 2, size=(R, V)).astype(np.float32)
    # ties, dead entries, -0.0 and NaN
    rows[3, 10:40] = -1.0
    rows[4, :] = -2.0
    rows[5, 50:] = -np.inf
    rows[6, 7] = np.nan
    rows[7, 0:V:2] = -0.0
    rows[7, 1:V:2] = 0.0
    rows[8, 1:] = NEG
    out = oracle.frame_lists(rows, 0, C)
    for r in range(R):
        v = np.maximum(np.nan_to_num(rows[r], nan=-np.inf), NEG) + np.float32(0.0)
        ids = np.arange(1, V)
        live = ids[v[1:] > NEG]
        order = live[np.lexsort((live, -v[live].astype(np.float64)))]
        n = min(C, order.size)
        assert out["cnt"][r] == n
        assert np.array_equal(out["ids"][r, :n], order[:n])
        assert np.array_equal(out["lps"][r, :n], v[order[:n]])
        assert out["lpb"][r] == v[0]
        if order.size > C:
            assert out["front_id"][r] == order[C] and out["front_lp"][r] == v[order[C]]
        else:
            assert out["front_id"][r] == -1 and out["front_lp"][r] == NEG


# ---- speech mask ("GPU CTC Prefix Beam Search Decoder", sections 8, 14, 15:
# frames the caller marks as non-speech bypass the decoder like skipped frames)

@pytest.mark.parametrize("seed", range(6))
def test_mask_equals_virtual_blank_brute_force(oracle, seed):
    rng = np.random.default_rng(90 + seed)
    V, T = 3, 9
    lp = random_frames(rng, T, V, 1.2, 0, 0.5)
    mask = (rng.random(T) < 0.6).astype(np.uint8)
    mask[rng.integers(0, T)] = 1
    kept = [t for t in range(T) if mask[t]]
    aug, _ = skip_augmented(lp, 0, 1.0, kept=kept)
    exact = posteriors(aug, 0)
    beam = max(V, n_prefixes(V, len(kept)))
    got, *_ = decoded(oracle, lp, beam=beam, mask=mask[None])
    assert set(got) == set(exact)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre]))


def test_mask_of_ones_is_no_mask_and_zeros_decode_nothing(oracle):
    rng = np.random.default_rng(7)
    B, T, V = 3, 40, 12
    lp = np.stack([random_frames(rng, T, V, 2.0, 0, 1.5) for _ in range(B)])
    lens = np.array([40, 17, 1], np.int32)
    ref = oracle.decode(lp, lens, beam=5)
    ones = oracle.decode(lp, lens, beam=5, mask=np.ones((B, T), np.uint8))
    for a, b in zip(ref, ones):
        assert np.array_equal(a, b)
    tok, ln, sc = oracle.decode(lp, lens, beam=5, mask=np.zeros((B, T), np.uint8))
    assert (ln[:, 0] == 0).all() and (sc[:, 0] == 0.0).all()


def test_mask_and_threshold_select_their_intersection(oracle):
    rng = np.random.default_rng(11)
    B, T, V = 4, 60, 10
    x = rng.normal(0.0, 1.0, size=(B, T, V))
    x[:, :, 0] += np.where(rng.random((B, T)) < 0.5, 9.0, 0.0)
    lp = log_softmax(x)
    thr = 0.99
    mask = (rng.random((B, T)) < 0.7).astype(np.uint8)
    sel, nsel = oracle.select_frames(lp, np.full(B, T, np.int32), 0, thr)
    both = np.zeros((B, T), np.uint8)
    for b in range(B):
        for t in sel[b, :nsel[b]]:
            both[b, t] = mask[b, t]
    a = oracle.decode(lp, None, beam=6, thr=thr, mask=mask)
    c = oracle.decode(lp, None, beam=6, mask=both)
    for u, v in zip(a, c):
        assert np.array_equal(u, v)


# ---- word-boundary label ("GPU CTC Prefix Beam Search Decoder", sections
# 3.4.1/3.4.2: the space extension always takes lp[space] + lse(pb, pnb), and
# a space-ending beam has no stay path): every space frame is its own token

@pytest.mark.parametrize("seed", range(5))
def test_space_unpruned_equals_brute_force(oracle, seed):
    rng = np.random.default_rng(120 + seed)
    V, T, space = 3, 8, 2
    lp = random_frames(rng, T, V, 1.0, 0, 0.3)
    exact = posteriors(lp, 0, space=space)
    beam = n_prefixes(V, T)
    got, *_ = decoded(oracle, lp, beam=beam, space=space)
    assert set(got) == set(exact)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre]))
    # the collapse really differs from the plain one on these frames
    assert set(exact) != set(posteriors(lp, 0))


@pytest.mark.parametrize("seed", range(3))
def test_space_with_skipping_equals_brute_force(oracle, seed):
    rng = np.random.default_rng(140 + seed)
    V, T, space = 3, 9, 1
    x = rng.normal(0.0, 1.0, size=(T, V))
    x[rng.random(T) < 0.4, 0] += 9.0
    lp = log_softmax(x)
    thr = 0.99
    aug, kept = skip_augmented(lp, 0, thr)
    exact = posteriors(aug, 0, space=space)
    beam = max(V, n_prefixes(V, len(kept)))
    got, *_ = decoded(oracle, lp, beam=beam, thr=thr, space=space)
    assert set(got) == set(exact)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre]))


def test_space_equal_to_blank_has_no_effect(oracle):
    rng = np.random.default_rng(5)
    lp = np.stack([random_frames(rng, 30, 8, 2.0, 0, 1.0) for _ in range(3)])
    a = oracle.decode(lp, None, beam=6)
    b = oracle.decode(lp, None, beam=6, space=0)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ---- token boosting (the per-utterance word-boosting table of "GPU-Accelerated
# WFST Beam Search Decoder for CTC-based Speech Recognition", applied to CTC
# labels): a label emitted by an extension adds its bonus, so without pruning
# a prefix scores log P(l) + the sum of its labels' bonuses

def random_bonus(rng, V, blank, n):
    labels = [c for c in range(V) if c != blank]
    pick = rng.choice(labels, size=min(n, len(labels)), replace=False)
    return {int(c): float(np.float32(rng.normal(0.0, 2.0))) for c in pick}


@pytest.mark.parametrize("seed", range(6))
def test_boost_unpruned_equals_brute_force(oracle, seed):
    rng = np.random.default_rng(300 + seed)
    V, T, blank = (3, 6, 0) if seed % 2 == 0 else (4, 4, 2)
    lp = random_frames(rng, T, V, 1.5, blank, 0.5)
    bonus = random_bonus(rng, V, blank, 2)
    exact = posteriors(lp, blank, bonus=bonus)
    beam = max(V, n_prefixes(V, T))
    got, *_ = decoded(oracle, lp, beam=beam, blank=blank, boost=[bonus])
    assert set(got) == set(exact)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre])), (pre, s, exact[pre])
    # the bonuses really move the scores
    plain = posteriors(lp, blank)
    assert any(abs(exact[p] - plain[p]) > 1e-3 for p in exact)


@pytest.mark.parametrize("seed", range(3))
def test_boost_with_cap_space_and_skipping_equals_brute_force(oracle, seed):
    rng = np.random.default_rng(330 + seed)
    V, T, space, cap = 3, 9, 2, 3
    x = rng.normal(0.0, 1.0, size=(T, V))
    x[rng.random(T) < 0.4, 0] += 9.0
    lp = log_softmax(x)
    thr = 0.99
    bonus = {1: 1.25, 2: -0.75}
    aug, kept = skip_augmented(lp, 0, thr)
    exact = posteriors(aug, 0, cap=cap, space=space, bonus=bonus)
    beam = max(V, n_prefixes(V, len(kept), cap))
    got, *_ = decoded(oracle, lp, beam=beam, thr=thr, space=space, cap=cap, boost=[bonus])
    assert set(got) == set(exact)
    for pre, s in got.items():
        assert abs(s - exact[pre]) <= 2e-5 * max(1.0, abs(exact[pre])), (pre, s, exact[pre])


def test_zero_bonus_is_bit_identical(oracle):
    rng = np.random.default_rng(9)
    lp = np.stack([random_frames(rng, 40, 12, 2.0, 0, 1.0) for _ in range(3)])
    a = oracle.decode(lp, None, beam=5)
    b = oracle.decode(lp, None, beam=5, boost=[{c: 0.0 for c in range(1, 12)}] * 3)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


@pytest.mark.parametrize("seed", range(4))
def test_boost_pruned_scores_at_most_exact(oracle, seed):
    """A pruned beam keeps a subset of each prefix's alignments, each carrying
    that prefix's bonuses, so its score is at most the exact boosted one."""
    rng = np.random.default_rng(360 + seed)
    V, T = 4, 7
    lp = random_frames(rng, T, V, 1.5, 0, 0.5)
    bonus = random_bonus(rng, V, 0, 3)
    exact = posteriors(lp, 0, bonus=bonus)
    got, *_ = decoded(oracle, lp, beam=3, boost=[bonus])
    for pre, s in got.items():
        assert s <= exact[pre] + 2e-5 * max(1.0, abs(exact[pre]))


def test_large_bonus_wins_the_beam(oracle):
    """A label the acoustics rank second on every frame becomes the 1-best's
    only label once its bonus outweighs the gap."""
    T, V = 6, 5
    x = np.full((T, V), -4.0)
    x[:, 0] = 0.0
    x[2, 1] = 2.0
    x[2, 3] = 1.0
    lp = log_softmax(x)
    tok, ln, _ = oracle.decode(lp[None], None, beam=4)
    assert tok[0, 0, :ln[0, 0]].tolist() == [1]
    tok, ln, _ = oracle.decode(lp[None], None, beam=4, boost=[{3: 2.0}])
    assert tok[0, 0, :ln[0, 0]].tolist() == [3]
