"""Streaming across the warp step kernel's label history ("GPU CTC Prefix Beam
Search Decoder", sections 3.4.5 and 8): the kernel records each step's
(source slot, label) in a 128-step ring and writes the token rows when the
ring fills, before an exact merge check and at the end of every call.
Chunkings that cross the ring's boundary at many offsets, reads between
calls, short outputs and exact merge checks in streamed rows must all give
the oracle's tokens and scores."""
import numpy as np
import pytest
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D
from gpu_util import assert_same

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    O.lib()
    assert torch.cuda.is_available()


def frames(seed, B, T, V, p_blank=0.6):
    """Log-softmax of N(0, 1.5) logits, the blank raised by 5 on a random 60%
    of the frames."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 1.5, size=(B, T, V))
    x[:, :, 0] += np.where(rng.random((B, T)) < p_blank, 5.0, 0.0)
    x -= x.max(-1, keepdims=True)
    return (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32)


def oracle_prefix(cfg, lp, t, out_len):
    return O.decode(np.ascontiguousarray(lp[:, :t]), None, beam=cfg.beam, nbest=cfg.c().nbest, blank=0,
                    cap=cfg.max_seq_len, out_len=out_len)


@pytest.mark.parametrize("beam,V,chunks", [(10, 100, (1,)),
                                           (10, 100, (5, 16, 64)),
                                           (4, 29, (127, 1, 128)),
                                           (16, 1000, (129, 3)),
                                           (7, 29, (31, 97)),
                                           (1, 29, (64,))])
def test_chunkings_across_the_ring_boundary(beam, V, chunks):
    B, T = 3, 600
    lp = frames(beam * 1000 + V, B, T, V)
    cfg = D.Config(beam=beam, nbest=min(beam, 5), max_seq_len=T)
    st = D.StreamState(cfg, B, V)
    x = torch.from_numpy(lp).cuda()
    sizes, t = [], 0
    while t < T:
        c = min(chunks[len(sizes) % len(chunks)], T - t)
        sizes.append(c)
        t += c
    read_at = set(np.linspace(1, len(sizes) - 1, 6).astype(int).tolist())
    t = 0
    for i, c in enumerate(sizes):
        st.step_chunk(x[:, t:t + c])
        t += c
        if i in read_at:  # a read between calls: the frames so far, nothing changed
            got = st.read(out_len=T)
            torch.cuda.synchronize()
            assert_same(tuple(v.cpu().numpy() for v in got), oracle_prefix(cfg, lp, t, T), f"after {t} frames")
    got = st.read(out_len=T)
    torch.cuda.synchronize()
    assert_same(tuple(v.cpu().numpy() for v in got), oracle_prefix(cfg, lp, T, T), "all frames")
    assert st.status() == 0
    assert D.read_counters(st.buf)["steps"] == B * T


@pytest.mark.parametrize("out_len", [0, 3, 40])
def test_short_outputs_of_streamed_rows(out_len):
    """Outputs shorter than the hypotheses: the labels past out_len are cut,
    the lengths are full."""
    B, T, V = 2, 200, 29
    lp = frames(5, B, T, V, p_blank=0.3)
    cfg = D.Config(beam=8, nbest=8, max_seq_len=T)
    st = D.StreamState(cfg, B, V)
    x = torch.from_numpy(lp).cuda()
    for t0 in range(0, T, 50):
        st.step_chunk(x[:, t0:t0 + 50])
    got = st.read(out_len=out_len)
    torch.cuda.synchronize()
    assert_same(tuple(v.cpu().numpy() for v in got), oracle_prefix(cfg, lp, T, out_len), f"out_len {out_len}")


def streamed_merge_case(seed):
    """Small vocabularies and long rows make the warp kernel confirm prefix-hash
    merge proposals against the stored labels (the ring is written to the rows
    first), here in the middle of 16-frame streaming calls.  Returns how many
    merges the check confirmed."""
    B, T, V = 4, 900, 5
    lp = frames(70 + seed, B, T, V, p_blank=0.5)
    cfg = D.Config(beam=16, nbest=16, max_seq_len=T)
    st = D.StreamState(cfg, B, V)
    x = torch.from_numpy(lp).cuda()
    for t0 in range(0, T, 16):
        st.step_chunk(x[:, t0:t0 + 16])
    got = st.read(out_len=T)
    torch.cuda.synchronize()
    assert_same(tuple(v.cpu().numpy() for v in got), oracle_prefix(cfg, lp, T, T), f"seed {seed}")
    assert st.status() == 0
    return D.read_counters(st.buf)["hash_merges"]


def test_exact_merge_checks_in_streamed_rows():
    """Parity on every seed, and the inputs do exercise the exact check."""
    assert sum(streamed_merge_case(seed) for seed in range(4)) > 0
