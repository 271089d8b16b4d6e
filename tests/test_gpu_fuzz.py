"""Randomised parity sweep: seeded configurations across the decoder's options
(beam, vocabulary, lengths, paged storage, page size, list length, cap, frame
skipping, word-boundary label, label boosting), each decoded on the GPU and
by the oracle; tokens, lengths and scores bit-identical."""
import numpy as np
import pytest
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D
from gpu_util import assert_same, oracle_offline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    O.lib()
    assert torch.cuda.is_available()


def draw(seed):
    """One random configuration and its input (small enough for the oracle)."""
    rng = np.random.default_rng(10_000 + seed)
    V = int(rng.choice([3, 5, 12, 29, 64, 257, 1000, 2048]))
    beam = int(rng.choice([1, 2, 4, 7, 10, 16, 17, 24, 40, 64]))
    B = int(rng.integers(1, 6))
    T = int(rng.integers(1, 140))
    blank = int(rng.integers(0, V)) if rng.random() < 0.3 else 0
    cfg = dict(beam=beam, nbest=int(rng.integers(1, beam + 1)), blank_id=blank)
    if rng.random() < 0.3:
        cfg.update(paged=True, page_size=int(rng.choice([1, 3, 16, 64])))
    if rng.random() < 0.3:
        cfg["max_seq_len"] = int(rng.integers(1, 40))
    if rng.random() < 0.3:
        cfg["list_len"] = int(rng.integers(1, 80))
    if rng.random() < 0.3:
        cfg["blank_threshold"] = float(rng.choice([0.5, 0.9, 0.99, 0.999]))
    if rng.random() < 0.25 and V > 2:
        sp = int(rng.integers(0, V))
        cfg["space_id"] = sp
    boost = None
    if rng.random() < 0.3 and V > 2:
        nb = int(rng.integers(1, min(V - 1, 20) + 1))
        labels = [c for c in range(V) if c != blank]
        pick = rng.choice(labels, size=min(nb, len(labels)), replace=False)
        boost = [{int(c): float(np.float32(rng.uniform(-3, 5))) for c in pick} for _ in range(B)]
        cfg["max_boost"] = nb
    x = rng.normal(0.0, float(rng.choice([0.5, 1.5, 3.0])), size=(B, T, V))
    x[:, :, blank] += float(rng.choice([0.0, 2.0, 6.0]))
    lp = (x - np.log(np.exp(x - x.max(-1, keepdims=True)).sum(-1, keepdims=True)) - x.max(-1, keepdims=True))
    lp = lp.astype(np.float32)
    lens = rng.integers(0, T + 1, size=B).astype(np.int32) if rng.random() < 0.5 else None
    return D.Config(**cfg), lp, lens, boost


@pytest.mark.parametrize("seed", range(160))
def test_random_configuration_matches_oracle(seed):
    cfg, lp, lens, boost = draw(seed)
    dev = torch.device("cuda")
    x = torch.from_numpy(lp).to(dev)
    ln = None if lens is None else torch.from_numpy(lens).to(dev)
    B, T, V = lp.shape
    ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device=dev)
    tok, l, sc = D.decode_offline(cfg, x, ln, workspace=ws, boost=boost)
    torch.cuda.synchronize()
    g = (tok.cpu().numpy(), l.cpu().numpy(), sc.cpu().numpy())
    assert_same(g, oracle_offline(cfg, lp, lens, boost=boost), f"seed {seed}: {cfg}")
    assert D.read_status(ws) == 0


@pytest.mark.parametrize("seed", range(60))
def test_random_streaming_matches_oracle(seed):
    """The same configurations streamed in random chunkings, half of them
    with a random speech mask, against the oracle decoding every frame (the
    masked ones skipped) offline."""
    cfg, lp, _, boost = draw(seed)
    cfg.blank_threshold = 1.0  # streaming never skips by threshold
    B, T, V = lp.shape
    rng = np.random.default_rng(20_000 + seed)
    mask = (rng.random((B, T)) > 0.3).astype(np.uint8) if rng.random() < 0.5 else None
    st = D.StreamState(cfg, B, V)
    if boost is not None:
        st.set_boost(boost)
    t0 = 0
    while t0 < T:
        c = int(min(T - t0, rng.integers(1, 90)))
        chunk = torch.from_numpy(np.ascontiguousarray(lp[:, t0:t0 + c])).cuda()
        if mask is None:
            st.step_chunk(chunk)
        else:
            st.step_chunk(chunk, is_speech=torch.from_numpy(np.ascontiguousarray(mask[:, t0:t0 + c])).cuda())
        t0 += c
    out = st.read(out_len=T)
    torch.cuda.synchronize()
    cap = cfg.max_seq_len if cfg.max_seq_len > 0 else 4096
    ref = O.decode(lp, None, beam=cfg.beam, nbest=cfg.c().nbest, blank=cfg.blank_id, cap=cap, out_len=T,
                   mask=mask, space=cfg.space_id, boost=boost)
    assert_same(tuple(v.cpu().numpy() for v in out), ref, f"seed {seed}: {cfg}")
    assert st.status() == 0


@pytest.mark.parametrize("seed", range(60))
def test_random_host_buffer_decode_matches_oracle(seed):
    """The same configurations through the host-buffer call (chunked copies,
    streaming tiles, threshold skipping per tile)."""
    cfg, lp, lens, boost = draw(seed)
    x = torch.from_numpy(lp).pin_memory()
    ln = None if lens is None else torch.from_numpy(lens).pin_memory()
    out = D.decode_offline_host(cfg, x, ln, boost=boost)
    assert_same(tuple(o.numpy() for o in out), oracle_offline(cfg, lp, lens, boost=boost), f"seed {seed}: {cfg}")


def draw_long(seed):
    """A long-utterance configuration: rows of 150-800 frames (token-store
    writes in many rounds, several 64-step windows), beams up to 128."""
    rng = np.random.default_rng(999_000 + seed)
    V = int(rng.choice([29, 100, 1024, 5000]))
    beam = int(rng.choice([4, 10, 16, 20, 32, 48, 64, 128]))
    T = int(rng.integers(150, 800))
    if beam * V * T > 120_000_000:
        T = max(60, 120_000_000 // (beam * V))
    B = int(rng.integers(1, 4))
    cfg = dict(beam=beam, nbest=min(beam, int(rng.integers(1, 12))))
    if rng.random() < 0.4:
        cfg.update(paged=True, page_size=int(rng.choice([1, 2, 8, 16])))
    if rng.random() < 0.25:
        cfg["max_seq_len"] = int(rng.integers(5, 300))
    if rng.random() < 0.25:
        cfg["space_id"] = int(rng.integers(1, V))
    boost = None
    if rng.random() < 0.4:
        nb = min(int(rng.integers(1, 30)), V - 1)
        boost = [{int(c): float(np.float32(rng.uniform(-3, 5))) for c in rng.choice(np.arange(1, V), nb, replace=False)}
                 for _ in range(B)]
        cfg["max_boost"] = nb
    x = rng.normal(0, float(rng.choice([1.0, 2.0])), size=(B, T, V))
    x[:, :, 0] += np.where(rng.random((B, T)) < 0.7, 6.0, 0.0)
    lp = x - x.max(-1, keepdims=True)
    lp = (lp - np.log(np.exp(lp).sum(-1, keepdims=True))).astype(np.float32)
    return rng, D.Config(**cfg), lp, boost


@pytest.mark.parametrize("seed", range(24))
def test_random_long_utterances_match_oracle(seed):
    """Even seeds decode offline (with lengths, maybe a threshold); odd seeds
    stream in random chunks, maybe masked."""
    rng, cfg, lp, boost = draw_long(seed)
    B, T, V = lp.shape
    if seed % 2 == 0:
        lens = rng.integers(T // 3, T + 1, size=B).astype(np.int32)
        if rng.random() < 0.3:
            cfg.blank_threshold = float(rng.choice([0.9, 0.99, 0.999]))
        ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device="cuda")
        out = D.decode_offline(cfg, torch.from_numpy(lp).cuda(), torch.from_numpy(lens).cuda(), workspace=ws,
                               boost=boost)
        torch.cuda.synchronize()
        assert_same(tuple(o.cpu().numpy() for o in out), oracle_offline(cfg, lp, lens, boost=boost), f"seed {seed}")
        assert D.read_status(ws) == 0
        return
    mask = (rng.random((B, T)) > 0.25).astype(np.uint8) if rng.random() < 0.5 else None
    st = D.StreamState(cfg, B, V)
    if boost is not None:
        st.set_boost(boost)
    t = 0
    while t < T:
        c = int(min(T - t, rng.integers(1, 130)))
        ch = torch.from_numpy(np.ascontiguousarray(lp[:, t:t + c])).cuda()
        if mask is None:
            st.step_chunk(ch)
        else:
            st.step_chunk(ch, is_speech=torch.from_numpy(np.ascontiguousarray(mask[:, t:t + c])).cuda())
        t += c
    out = st.read(out_len=T)
    torch.cuda.synchronize()
    cap = cfg.max_seq_len if cfg.max_seq_len > 0 else 4096
    ref = O.decode(lp, None, beam=cfg.beam, nbest=cfg.c().nbest, blank=0, cap=cap, out_len=T, mask=mask,
                   space=cfg.space_id, boost=boost)
    assert_same(tuple(v.cpu().numpy() for v in out), ref, f"seed {seed}")
    assert st.status() == 0


def draw_slow(seed):
    """A warp-kernel configuration (beam <= 16, flat storage) with near-flat,
    tied or quantised frames, so that many steps are unproven, exhaustive or
    scan the frame."""
    rng = np.random.default_rng(50_000 + seed)
    V = int(rng.choice([8, 16, 40, 100, 256, 1000, 3000]))
    beam = int(rng.integers(2, 17))
    B, T = int(rng.integers(1, 5)), int(rng.integers(2, 80))
    L = int(rng.choice([0, 0, 1, 3, 8, 22, 40, 66]))
    cfg = D.Config(beam=beam, nbest=int(rng.integers(1, beam + 1)), list_len=L,
                   max_seq_len=int(rng.integers(2, 30)) if rng.random() < 0.2 else 0,
                   space_id=int(rng.integers(1, V)) if rng.random() < 0.2 else -1)
    x = rng.normal(0.0, float(rng.choice([0.02, 0.1, 0.5, 1.0])), size=(B, T, V))
    x[:, :, 0] += float(rng.choice([0.0, 0.5, 2.0]))
    lp = x - x.max(-1, keepdims=True)
    lp = (lp - np.log(np.exp(lp).sum(-1, keepdims=True))).astype(np.float32)
    if rng.random() < 0.5:  # tied frames: every non-blank label one log-prob
        fr = rng.random(T) < 0.4
        lp[:, fr, 1:] = lp[:, fr, 1:].mean(-1, keepdims=True)
    if rng.random() < 0.3:  # quantised log-probs: many exact ties
        lp = np.round(lp, 1).astype(np.float32)
    lens = rng.integers(0, T + 1, size=B).astype(np.int32)
    return cfg, lp, lens


@pytest.mark.parametrize("seed", range(60))
def test_random_slow_selections_match_oracle(seed):
    cfg, lp, lens = draw_slow(seed)
    B, T, V = lp.shape
    dev = torch.device("cuda")
    ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device=dev)
    out = D.decode_offline(cfg, torch.from_numpy(lp).to(dev), torch.from_numpy(lens).to(dev), workspace=ws)
    torch.cuda.synchronize()
    assert_same(tuple(o.cpu().numpy() for o in out), oracle_offline(cfg, lp, lens), f"seed {seed}: {cfg}")
    assert D.read_status(ws) == 0
