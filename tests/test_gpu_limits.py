"""Decodes at the limits the C ABI accepts, against the oracle: the largest
vocabulary (2^20 labels, the 20-bit label field of the rank keys; its rows
are too large to stage in shared memory, so the plain per-warp ranking runs),
utterances of 12,000 frames (hypotheses of thousands of labels, written to
the token store in many windows) and the largest page size."""
import numpy as np
import pytest
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D
from gpu_util import assert_same, gpu_offline, oracle_offline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    O.lib()
    assert torch.cuda.is_available()


def frames(seed, B, T, V, blank_boost=2.0, peak=0.0):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 1.5, size=(B, T, V)).astype(np.float64)
    x[:, :, 0] += blank_boost
    if peak:  # one label per frame raised, so long rows emit many labels
        lab = rng.integers(1, V, size=(B, T))
        np.put_along_axis(x, lab[:, :, None], np.take_along_axis(x, lab[:, :, None], 2) + peak, 2)
    x -= x.max(-1, keepdims=True)
    return (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32)


@pytest.mark.parametrize("beam,B,T", [(4, 2, 5), (17, 1, 3)])
def test_largest_vocabulary(beam, B, T):
    V = 1 << 20
    lp = frames(beam, B, T, V, blank_boost=4.0)
    cfg = D.Config(beam=beam, nbest=min(beam, 4))
    assert_same(gpu_offline(cfg, lp, None), oracle_offline(cfg, lp, None), f"V=2^20 beam {beam}")


def test_vocabulary_past_the_label_field_is_rejected():
    with pytest.raises(D.CtcpbError) as e:
        D.workspace_size(D.Config(beam=4), 1, 4, (1 << 20) + 1)
    assert e.value.code == D.EINVAL


@pytest.mark.parametrize("kw", [dict(beam=8, nbest=3), dict(beam=24, nbest=3, paged=True, page_size=64)],
                         ids=["flat warp kernel", "paged block kernel"])
def test_long_utterances(kw):
    B, T, V = 2, 12000, 29
    lp = frames(11, B, T, V, blank_boost=1.0, peak=3.0)
    lens = np.array([T, T - 777], np.int32)
    cfg = D.Config(**kw)
    got = gpu_offline(cfg, lp, lens)
    ref = oracle_offline(cfg, lp, lens)
    assert int(ref[1].max()) > 2000  # thousands of labels per hypothesis
    assert_same(got, ref, f"T={T} {kw}")


def test_largest_page_size():
    B, T, V = 3, 300, 40
    lp = frames(12, B, T, V, peak=2.0)
    cfg = D.Config(beam=8, nbest=8, paged=True, page_size=1024)
    assert_same(gpu_offline(cfg, lp, None), oracle_offline(cfg, lp, None), "page 1024")
