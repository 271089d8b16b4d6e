"""Speech-masked streaming ("GPU CTC Prefix Beam Search Decoder", section 8's
is_speech_mask; sections 14-15: frames marked as non-speech bypass the
decoder) against the oracle decoding the same frames offline with the same
mask."""
import numpy as np
import pytest
import torch

from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import assert_same, cfg_of, oracle_offline

import oracle as O

pytestmark = pytest.mark.gpu


def stream_masked(cfg, lp, mask, chunk, nframes=None):
    B, T, V = lp.shape
    dev = torch.device("cuda")
    st = D.StreamState(cfg, B, V, device=dev)
    x = torch.from_numpy(np.ascontiguousarray(lp)).to(dev)
    m = torch.from_numpy(np.ascontiguousarray(mask, np.uint8)).to(dev)
    for t0 in range(0, T, chunk):
        nf = None if nframes is None else torch.from_numpy(nframes[t0 // chunk]).to(dev)
        st.step_chunk(x[:, t0:t0 + chunk], nf, is_speech=m[:, t0:t0 + chunk])
    out_len = cfg.max_seq_len
    tok, ln, sc = st.read(out_len=out_len)
    torch.cuda.synchronize()
    assert st.status() == 0
    return tok.cpu().numpy(), ln.cpu().numpy(), sc.cpu().numpy()


def oracle_masked(cfg, lp, mask):
    T = lp.shape[1]
    return O.decode(lp, None, beam=cfg.beam, nbest=cfg.nbest, blank=cfg.blank_id, cap=cfg.max_seq_len,
                    out_len=cfg.max_seq_len, mask=mask)


@pytest.mark.parametrize("name,over,chunk,p", [("bpe", dict(B=6, T=150), 16, 0.6),
                                               ("bpe", dict(B=6, T=150), 70, 0.85),
                                               ("skip", dict(B=10, T=120), 33, 0.5),
                                               ("char", dict(B=3, T=90), 16, 0.7),
                                               ("tiny", dict(B=4, T=50), 1, 0.6)])
def test_masked_streaming_matches_oracle(name, over, chunk, p):
    w = synth.workload(name, **over)
    lp, _ = synth.gen_batch(w, pad="zero")
    rng = np.random.default_rng(len(name) + chunk)
    mask = (rng.random((w.B, w.T)) < p).astype(np.uint8)
    mask[0, :] = 0                      # a stream that never speaks
    mask[1, : w.T // 2] = 0             # a long silent lead-in
    cfg = cfg_of(w, max_seq_len=w.T, blank_threshold=1.0)
    assert_same(stream_masked(cfg, lp, mask, chunk), oracle_masked(cfg, lp, mask), f"{name}{over} chunk {chunk}")


def test_mask_of_ones_equals_unmasked_streaming():
    w = synth.workload("bpe", B=5, T=100)
    lp, _ = synth.gen_batch(w, pad="zero")
    cfg = cfg_of(w, max_seq_len=w.T)
    a = stream_masked(cfg, lp, np.ones((w.B, w.T), np.uint8), 24)
    dev = torch.device("cuda")
    st = D.StreamState(cfg, w.B, w.V, device=dev)
    x = torch.from_numpy(lp).to(dev)
    for t0 in range(0, w.T, 24):
        st.step_chunk(x[:, t0:t0 + 24])
    b = tuple(o.cpu().numpy() for o in st.read(out_len=w.T))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_masked_partial_chunks():
    """Streams with ragged chunk lengths (n_frames) and masks."""
    w = synth.workload("bpe", B=4, T=96)
    lp, _ = synth.gen_batch(w, pad="zero")
    rng = np.random.default_rng(3)
    mask = (rng.random((w.B, w.T)) < 0.7).astype(np.uint8)
    chunk = 32
    # stream b delivers n_b frames per chunk: its frames are packed at rows 0..n_b-1
    counts = [np.array([32, 20, 5, 0], np.int32), np.array([32, 12, 27, 32], np.int32),
              np.array([32, 32, 32, 32], np.int32)]
    B, T, V = lp.shape
    pos = np.zeros(B, np.int64)
    dev = torch.device("cuda")
    cfg = cfg_of(w, max_seq_len=w.T)
    st = D.StreamState(cfg, B, V, device=dev)
    for nfs in counts:
        ch = np.zeros((B, chunk, V), np.float32)
        mk = np.zeros((B, chunk), np.uint8)
        for b in range(B):
            n = int(nfs[b])
            ch[b, :n] = lp[b, pos[b]:pos[b] + n]
            mk[b, :n] = mask[b, pos[b]:pos[b] + n]
            pos[b] += n
        st.step_chunk(torch.from_numpy(ch).to(dev), torch.from_numpy(nfs).to(dev),
                      is_speech=torch.from_numpy(mk).to(dev))
    tok, ln, sc = (o.cpu().numpy() for o in st.read(out_len=w.T))
    assert st.status() == 0
    for b in range(B):
        n = int(pos[b])
        o = O.decode(lp[b:b + 1, :n], None, beam=cfg.beam, nbest=cfg.nbest, cap=w.T, out_len=w.T,
                     mask=mask[b:b + 1, :n])
        assert_same((tok[b:b + 1], ln[b:b + 1], sc[b:b + 1]), o, f"stream {b}")


@pytest.mark.parametrize("name,over,paged", [("bpe", dict(B=4, T=70), False),
                                             ("char", dict(B=3, T=60), True),
                                             ("tiny", dict(B=4, T=50), False)])
def test_single_frame_steps_match_oracle(name, over, paged):
    """The one-frame call (section 9's ctc_beam_search_step), fed column views
    of a [B, T, V] tensor (row stride T*V), mixed with chunk calls, some
    frames flagged as non-speech per stream: the same result as the oracle
    decoding every frame with that mask."""
    w = synth.workload(name, **over)
    lp, _ = synth.gen_batch(w, pad="zero")
    rng = np.random.default_rng(4242 + w.B)
    mask = (rng.random((w.B, w.T)) < 0.7).astype(np.uint8)
    mask[:, 0] = 1
    cfg = cfg_of(w, max_seq_len=w.T, blank_threshold=1.0)
    if paged:
        cfg.paged, cfg.page_size = True, 16
    dev = torch.device("cuda")
    x = torch.from_numpy(np.ascontiguousarray(lp)).to(dev)
    m = torch.from_numpy(mask).to(dev)
    st = D.StreamState(cfg, w.B, w.V, device=dev)
    t = 0
    while t < w.T:
        if t % 3 == 2:                      # a chunk of up to 7 frames
            c = min(7, w.T - t)
            st.step_chunk(x[:, t:t + c], is_speech=m[:, t:t + c])
            t += c
            continue
        col = x[:, t]
        assert col.stride(0) == w.T * w.V
        st.step(col, is_speech=None if mask[:, t].all() else m[:, t].contiguous())
        t += 1
    got = st.read(out_len=cfg.max_seq_len)
    torch.cuda.synchronize()
    assert st.status() == 0
    assert_same(tuple(v.cpu().numpy() for v in got), oracle_masked(cfg, lp, mask), f"{name}{over}")


def test_single_frame_steps_equal_one_chunk():
    """Every frame by the one-frame call, no mask, equals one chunk call over
    the same frames (bit-identical outputs)."""
    w = synth.workload("bpe", B=3, T=40)
    lp, _ = synth.gen_batch(w, pad="zero")
    cfg = cfg_of(w, max_seq_len=w.T, blank_threshold=1.0)
    x = torch.from_numpy(np.ascontiguousarray(lp)).cuda()
    a = D.StreamState(cfg, w.B, w.V)
    for t in range(w.T):
        a.step(x[:, t])
    b = D.StreamState(cfg, w.B, w.V)
    b.step_chunk(x)
    ra, rb = a.read(out_len=w.T), b.read(out_len=w.T)
    torch.cuda.synchronize()
    for u, v in zip(ra, rb):
        assert torch.equal(u, v)
