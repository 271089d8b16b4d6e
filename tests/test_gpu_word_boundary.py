"""The word-boundary ("space") label ("GPU CTC Prefix Beam Search Decoder",
sections 3.4.1/3.4.2: its extension always takes lp[space] + lse(pb, pnb), so
every space frame is a token of its own, and a space-ending beam has no stay
path) against the oracle, on every step-kernel path."""
import numpy as np
import pytest
import torch

from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import assert_same, cfg_of, gpu_offline, oracle_offline

pytestmark = pytest.mark.gpu


def log_softmax(x):
    x = np.asarray(x, np.float64)
    m = x.max(-1, keepdims=True)
    return (x - m - np.log(np.exp(x - m).sum(-1, keepdims=True))).astype(np.float32)


def spaced_batch(B, T, V, space, seed, blank=0, skip_frac=0.0):
    """Frames where the space label often wins; ``skip_frac`` of them are
    blank-dominant enough for a 0.999 threshold to skip."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 1.0, size=(B, T, V))
    x[:, :, blank] += np.where(rng.random((B, T)) < skip_frac, 18.0, 2.0)
    runs = rng.random((B, T)) < 0.3
    x[:, :, space] += np.where(runs, 4.0, 0.0)
    return log_softmax(x)


@pytest.mark.parametrize("name,over,space", [("bpe", dict(B=6, T=120), 3), ("skip", dict(B=8, T=200), 5),
                                             ("char", dict(B=3, T=80), 27), ("tiny", dict(B=4, T=50), 1)])
def test_word_boundary_matches_oracle(name, over, space):
    w = synth.workload(name, **over)
    lp, lens = synth.gen_batch(w)
    lp2 = spaced_batch(w.B, w.T, w.V, space, seed=space, skip_frac=0.3 if w.blank_threshold < 1.0 else 0.0)
    lp = np.where(np.isnan(lp), lp, lp2).astype(np.float32)  # keep the NaN padding of the workload
    cfg = cfg_of(w, space_id=space)
    g = gpu_offline(cfg, lp, lens)
    assert_same(g, oracle_offline(cfg, lp, lens), f"{name}{over} space {space}")
    # the label really decodes as separate tokens somewhere
    toks = g[0][g[0] >= 0]
    assert (toks == space).any()


@pytest.mark.parametrize("case", [dict(beam=4, V=5, space=2), dict(beam=32, V=9, space=8),
                                  dict(beam=40, V=7, space=1), dict(beam=6, V=6, space=3, paged=True),
                                  dict(beam=8, V=12, space=0, blank_id=4)])
def test_word_boundary_edge_cases(case):
    case = dict(case)
    V, space = case.pop("V"), case.pop("space")
    lp = spaced_batch(5, 60, V, space, seed=V, blank=case.get("blank_id", 0))
    lens = np.array([60, 0, 1, 37, 59], np.int32)
    cfg = D.Config(space_id=space, **case)
    assert_same(gpu_offline(cfg, lp, lens), oracle_offline(cfg, lp, lens), str(case))


def test_word_boundary_streaming_equals_offline():
    w = synth.workload("bpe", B=5, T=100)
    lp = spaced_batch(w.B, w.T, w.V, 7, seed=1)
    cfg = D.Config(beam=10, space_id=7, max_seq_len=w.T)
    dev = torch.device("cuda")
    st = D.StreamState(cfg, w.B, w.V, device=dev)
    x = torch.from_numpy(lp).to(dev)
    for t0 in range(0, w.T, 24):
        st.step_chunk(x[:, t0:t0 + 24])
    got = tuple(o.cpu().numpy() for o in st.read(out_len=w.T))
    assert st.status() == 0
    assert_same(got, oracle_offline(cfg, lp, np.full(w.B, w.T, np.int32)), "streaming")
