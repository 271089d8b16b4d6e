"""ctcpb_decode_offline_host (host input and outputs, chunked copies overlapped
with the decode) against ctcpb_decode_offline and the oracle, element by
element: tokens, lengths and scores bit-identical."""
import numpy as np
import pytest
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import NEG, assert_same, cfg_of, gpu_offline, oracle_offline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    O.lib()
    assert torch.cuda.is_available()


def host_decode(cfg, lp, lens, pinned=True, out_len=None):
    x = torch.from_numpy(np.ascontiguousarray(lp))
    ln = None if lens is None else torch.from_numpy(np.ascontiguousarray(lens, np.int32))
    if pinned:
        x = x.pin_memory()
        ln = None if ln is None else ln.pin_memory()
    out = D.decode_offline_host(cfg, x, ln, out_len=out_len)
    return tuple(o.numpy() for o in out)


CASES = [
    ("bpe", dict(B=6, T=200), {}),                                  # warp kernel, fused tiles
    ("bpe", dict(B=5, T=150), dict(beam=24, nbest=24)),             # block kernel
    ("char", dict(B=3, T=150), {}),                                 # paged, V % 4 != 0: plain pre-pass
    ("char", dict(B=3, T=130), dict(paged=False, beam=20, nbest=5)),
    ("skip", dict(B=8, T=300), {}),                                 # threshold 0.999
    ("skip", dict(B=6, T=200), dict(blank_threshold=0.5)),
    ("skip", dict(B=4, T=100), dict(blank_threshold=0.0)),          # no frame kept
    ("tiny", {}, {}),                                               # T = 50 < one chunk
]


@pytest.mark.parametrize("name,shape,over", CASES)
def test_host_decode_equals_device_decode_and_oracle(name, shape, over):
    w = synth.workload(name, **shape)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w, **over)
    h = host_decode(cfg, lp, lens)
    assert_same(h, gpu_offline(cfg, lp, lens), f"{name}{shape}{over} vs device")
    assert_same(h, oracle_offline(cfg, lp, lens), f"{name}{shape}{over} vs oracle")


def test_pageable_buffers_no_lengths_and_short_output():
    w = synth.workload("bpe", B=4, T=140)
    lp, _ = synth.gen_batch(w)
    cfg = cfg_of(w, beam=10, nbest=3)
    h = host_decode(cfg, lp, None, pinned=False, out_len=7)
    assert_same(h, oracle_offline(cfg, lp, None, out_len=7), "pageable")


def test_lengths_zero_one_and_full():
    w = synth.workload("bpe", B=5, T=130)
    lp, _ = synth.gen_batch(w)
    lens = np.array([0, 1, 64, 65, 130], np.int32)  # chunk edges at 64 and 128
    cfg = cfg_of(w)
    assert_same(host_decode(cfg, lp, lens), oracle_offline(cfg, lp, lens), "lengths")


def test_strided_host_rows():
    w = synth.workload("bpe", B=3, T=100)
    lp, lens = synth.gen_batch(w)
    B, T, V = lp.shape
    big = np.full((B, T, V + 12), np.nan, np.float32)
    big[:, :, :V] = lp
    x = torch.from_numpy(big).pin_memory()[:, :, :V]  # stride_t = V + 12
    cfg = cfg_of(w)
    out = D.decode_offline_host(cfg, x, torch.from_numpy(lens).pin_memory())
    assert_same(tuple(o.numpy() for o in out), oracle_offline(cfg, lp, lens), "strided")


def test_repeated_calls_share_the_workspace():
    w = synth.workload("bpe", B=4, T=260)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w)
    B, T, V = lp.shape
    ws = torch.empty(D.host_workspace_size(cfg, B, T, V, T), dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(lp).pin_memory()
    ln = torch.from_numpy(lens).pin_memory()
    ref = oracle_offline(cfg, lp, lens)
    outs = [D.decode_offline_host(cfg, x, ln, workspace=ws, synchronize=False) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert_same(tuple(t.numpy() for t in o), ref, "repeat")


@pytest.mark.parametrize("name", ["bpe", "skip"])
def test_full_size_host_decode_every_row(name):
    """The benchmark's end-to-end configuration: the full workload through the
    host-buffer call, every row against the oracle."""
    w = synth.WORKLOADS[name]
    lp, lens = synth.gen_batch(w, pad="nan")
    cfg = cfg_of(w)
    h = host_decode(cfg, lp, lens)
    o = oracle_offline(cfg, lp, lens)
    assert_same(h, o, f"{name}: all {w.B} rows")


@pytest.mark.parametrize("B,T,V,over", [(1, 1, 2, dict(beam=1, nbest=1)),
                                        (3, 65, 7, dict(beam=3, nbest=3, paged=True, page_size=2,
                                                        blank_threshold=0.9)),
                                        (2, 0, 5, dict(beam=2, nbest=2))])
def test_host_decode_edge_shapes(B, T, V, over):
    rng = np.random.default_rng(B * 100 + T + V)
    x = rng.normal(0.0, 2.0, size=(B, T, V))
    if T:
        x[:, :, 0] += 1.5
    lp = (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32) if T else np.zeros((B, 0, V), np.float32)
    cfg = D.Config(**over)
    h = host_decode(cfg, lp, None)
    if T == 0:  # no decoded frame: the empty prefix with score 0, then dead slots
        nb = cfg.nbest
        exp_sc = np.full((B, nb), NEG, np.float32)
        exp_sc[:, 0] = 0.0
        assert_same(h, (np.zeros((B, nb, 0), np.int32), np.zeros((B, nb), np.int32), exp_sc), "T=0")
        return
    assert_same(h, oracle_offline(cfg, lp, None), f"B={B} T={T} V={V} {over}")
