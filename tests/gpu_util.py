"""Shared helpers of the GPU parity tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D

NEG = np.float32(np.finfo(np.float32).min)
SCORE_TOL = 1e-4  # absolute score tolerance of the decoder's contract


def cfg_of(w, **kw):
    base = dict(beam=w.beam, nbest=w.nbest, blank_id=w.blank_id, max_seq_len=w.max_seq_len,
                blank_threshold=w.blank_threshold, paged=bool(w.paged), page_size=w.page_size)
    base.update(kw)
    return D.Config(**base)


def gpu_offline(cfg, lp: np.ndarray, lens: np.ndarray | None, out_len=None):
    dev = torch.device("cuda")
    x = torch.from_numpy(np.ascontiguousarray(lp)).to(dev)
    ln = None if lens is None else torch.from_numpy(np.ascontiguousarray(lens, np.int32)).to(dev)
    tok, l, s = D.decode_offline(cfg, x, ln, out_len=out_len)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), l.cpu().numpy(), s.cpu().numpy()


def oracle_offline(cfg, lp, lens, out_len=None, rows=None, boost=None):
    T = lp.shape[1]
    cap = cfg.max_seq_len if cfg.max_seq_len > 0 else T
    cap = min(cap, max(T, 1))
    if out_len is None:
        out_len = min(cfg.max_seq_len, T) if cfg.max_seq_len > 0 else T
    nb = cfg.beam if cfg.nbest is None else cfg.nbest
    if rows is not None:
        lp = lp[rows]
        lens = None if lens is None else lens[rows]
        boost = None if boost is None else [boost[r] for r in rows]
    return O.decode(lp, lens, beam=cfg.beam, nbest=nb, blank=cfg.blank_id, cap=cap,
                    thr=cfg.blank_threshold, out_len=out_len, space=cfg.space_id, boost=boost)


def assert_same(g, o, what="", exact_scores=True):
    gt, gl, gs = g
    ot, ol, os_ = o
    assert gl.shape == ol.shape, what
    bad = np.argwhere(gl != ol)
    assert bad.size == 0, f"{what}: lengths differ at {bad[:5].tolist()}"
    assert np.array_equal(gt, ot), f"{what}: tokens differ at {np.argwhere(gt != ot)[:5].tolist()}"
    d = np.abs(gs.astype(np.float64) - os_.astype(np.float64))
    assert d.max() <= SCORE_TOL, f"{what}: max score diff {d.max()}"
    if exact_scores:
        assert np.array_equal(gs.view(np.int32), os_.view(np.int32)), f"{what}: scores not bit-identical"
