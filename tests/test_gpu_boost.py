"""Label boosting on the GPU against the oracle, through the C ABI.

Boosting adapts the per-utterance word-boosting table of "GPU-Accelerated
WFST Beam Search Decoder for CTC-based Speech Recognition" to CTC labels: an
emitted label scores lp + bonus in the ranking, the extensions and the merge
folds.  Bars as in the other parity tests: tokens and lengths bit-exact,
scores bit-identical (hence within 1e-4).
"""
import numpy as np
import pytest
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import assert_same, cfg_of, oracle_offline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    O.lib()
    assert torch.cuda.is_available()


def random_boosts(rng, B, V, blank, n, lo=-3.0, hi=5.0, frames=None):
    """n boosted labels per row, half of them labels the row's frames favour
    (so the bonuses change the decode), bonuses uniform in [lo, hi)."""
    out = []
    for b in range(B):
        labels = [c for c in range(V) if c != blank]
        pick = set()
        if frames is not None:
            best = np.argsort(-frames[b].max(0))
            pick.update(int(c) for c in best[:2 * n] if c != blank and len(pick) < n // 2)
        pick.update(int(c) for c in rng.choice(labels, size=min(n, len(labels)), replace=False))
        pick = sorted(pick)[:n]
        out.append({c: float(np.float32(rng.uniform(lo, hi))) for c in pick})
    return out


def gpu_boosted(cfg, lp, lens, boost, out_len=None):
    dev = torch.device("cuda")
    x = torch.from_numpy(np.ascontiguousarray(lp)).to(dev)
    ln = None if lens is None else torch.from_numpy(np.ascontiguousarray(lens, np.int32)).to(dev)
    B, T, V = lp.shape
    ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device=dev)
    tok, l, s = D.decode_offline(cfg, x, ln, out_len=out_len, workspace=ws, boost=boost)
    torch.cuda.synchronize()
    return (tok.cpu().numpy(), l.cpu().numpy(), s.cpu().numpy()), ws


CASES = [
    ("bpe", dict(B=6, T=160), dict(), 24),                                    # beam 10: block kernel, 32 threads
    ("bpe", dict(B=4, T=120), dict(beam=40, nbest=40), 64),                   # 128 threads
    ("char", dict(B=3, T=150), dict(), 8),                                    # paged, beam 128
    ("char", dict(B=3, T=150), dict(paged=False, beam=24, nbest=24), 28),     # every letter boosted
    ("skip", dict(B=6, T=300), dict(), 16),                                   # frame skipping
    ("bpe", dict(B=4, T=100), dict(paged=True, page_size=4, max_seq_len=40), 12),
]


@pytest.mark.parametrize("name,shape,over,nb", CASES)
def test_boosted_decode_matches_oracle(name, shape, over, nb):
    w = synth.workload(name, **shape)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w, max_boost=max(nb, 1), **over)
    rng = np.random.default_rng(len(name) * 100 + nb)
    boost = random_boosts(rng, lp.shape[0], lp.shape[2], cfg.blank_id, nb, frames=lp)
    g, ws = gpu_boosted(cfg, lp, lens, boost)
    o = oracle_offline(cfg, lp, lens, boost=boost)
    assert_same(g, o, f"{name}{shape}{over}")
    assert D.read_status(ws) == 0
    assert D.read_counters(ws)["steps"] > 0
    # the bonuses change the result
    plain = oracle_offline(cfg, lp, lens)
    assert not all(np.array_equal(u, v) for u, v in zip(o, plain))


def test_boost_with_word_boundary_matches_oracle():
    w = synth.workload("char", B=3, T=150)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w, paged=False, beam=16, nbest=16, space_id=27, max_boost=4)
    boost = [{27: 1.5, 5: 2.0}, {27: -1.0}, {3: 0.5, 9: 3.0, 27: 0.75}]
    g, _ = gpu_boosted(cfg, lp, lens, boost)
    assert_same(g, oracle_offline(cfg, lp, lens, boost=boost), "space + boost")


def test_zero_bonuses_equal_the_plain_decode():
    w = synth.workload("bpe", B=4, T=120)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w, beam=12, nbest=12, max_boost=16)
    boost = [{c: 0.0 for c in range(1 + b, 200, 13)} for b in range(4)]
    g, _ = gpu_boosted(cfg, lp, lens, boost)
    assert_same(g, oracle_offline(cfg_of(w, beam=12, nbest=12), lp, lens), "zero bonuses")


def test_rejected_entries_are_ignored_and_flagged():
    w = synth.workload("bpe", B=3, T=100)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w, beam=10, nbest=10, max_boost=3)
    # row 0: a repeated label (the first bonus stays), the blank, a label past V;
    # row 1: a non-finite bonus and one above 1e6; row 2: more than max_boost labels
    tokens = [5, 9, 5, 0, 5000, 7, 8, 11, 1, 2, 3, 4]
    bonus = [2.0, 1.0, -7.0, 3.0, 3.0, float("inf"), 2e6, 1.5, 0.5, 0.5, 0.5, 0.5]
    row_ptr = [0, 5, 8, 12]
    tables = (torch.tensor(row_ptr, dtype=torch.int32), torch.tensor(tokens, dtype=torch.int32),
              torch.tensor(bonus, dtype=torch.float32))
    g, ws = gpu_boosted(cfg, lp, lens, tables)
    kept = [{5: 2.0, 9: 1.0}, {11: 1.5}, {1: 0.5, 2: 0.5, 3: 0.5}]
    assert_same(g, oracle_offline(cfg, lp, lens, boost=kept), "rejected entries")
    assert D.read_status(ws) & 0x10


@pytest.mark.parametrize("paged", [False, True])
def test_streaming_boost_equals_offline(paged):
    w = synth.workload("bpe", B=3, T=150)
    lp, _ = synth.gen_batch(w)
    cfg = cfg_of(w, beam=12, nbest=12, paged=paged, max_seq_len=150, max_boost=20)
    rng = np.random.default_rng(4)
    boost = random_boosts(rng, 3, lp.shape[2], 0, 20, frames=lp)
    ref = oracle_offline(cfg, lp, None, out_len=150, boost=boost)
    for chunks in ([150], [16] * 9 + [6], [7, 70, 73]):
        st = D.StreamState(cfg, 3, lp.shape[2])
        st.set_boost(boost)
        t0 = 0
        for c in chunks:
            st.step_chunk(torch.from_numpy(np.ascontiguousarray(lp[:, t0:t0 + c])).cuda())
            t0 += c
        out = st.read(out_len=150)
        torch.cuda.synchronize()
        assert_same(tuple(v.cpu().numpy() for v in out), ref, f"chunks {chunks[:3]}")
        assert st.status() == 0


@pytest.mark.parametrize("name,over", [("bpe", dict(beam=10)), ("char", dict(paged=True, beam=40, nbest=5))])
def test_boosted_host_buffer_decode_matches_oracle(name, over):
    w = synth.workload(name, B=4, T=180)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w, max_boost=16, **over)
    rng = np.random.default_rng(11)
    boost = random_boosts(rng, lp.shape[0], lp.shape[2], cfg.blank_id, 16, frames=lp)
    x = torch.from_numpy(np.ascontiguousarray(lp)).pin_memory()
    ln = torch.from_numpy(np.ascontiguousarray(lens, np.int32)).pin_memory()
    out = D.decode_offline_host(cfg, x, ln, boost=boost)
    assert_same(tuple(o.numpy() for o in out), oracle_offline(cfg, lp, lens, boost=boost), f"host {name}")


def test_streaming_boost_with_speech_mask_equals_offline():
    """Label boosts and a speech mask together (masked streaming on the boosted
    kernels) against the oracle decoding the same frames with the same mask."""
    w = synth.workload("bpe", B=3, T=150)
    lp, _ = synth.gen_batch(w)
    cfg = cfg_of(w, beam=10, nbest=10, max_seq_len=150, max_boost=12)
    rng = np.random.default_rng(21)
    boost = random_boosts(rng, 3, lp.shape[2], 0, 12, frames=lp)
    mask = (rng.random((3, 150)) > 0.3).astype(np.uint8)
    ref = O.decode(lp, None, beam=10, nbest=10, cap=150, out_len=150, mask=mask, boost=boost)
    st = D.StreamState(cfg, 3, lp.shape[2])
    st.set_boost(boost)
    t0 = 0
    for c in (16, 40, 94):
        st.step_chunk(torch.from_numpy(np.ascontiguousarray(lp[:, t0:t0 + c])).cuda(),
                      is_speech=torch.from_numpy(np.ascontiguousarray(mask[:, t0:t0 + c])).cuda())
        t0 += c
    out = st.read(out_len=150)
    torch.cuda.synchronize()
    assert_same(tuple(v.cpu().numpy() for v in out), ref, "boost + mask")
    assert st.status() == 0
