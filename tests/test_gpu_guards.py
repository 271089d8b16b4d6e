"""Guard regions around every caller-owned buffer: the workspace or state and
the three outputs are views into larger buffers whose margins are filled with
a pattern before the calls and must be unchanged after them.  Run across the
kernels and storage modes (fused warp kernel, block kernel, paged storage,
label boosting, frame skipping, streaming with a speech mask, the host-buffer
call), so a write outside a buffer shows up without a sanitizer; the decodes
also match the oracle."""
import numpy as np
import pytest
import torch

from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import assert_same, oracle_offline

import oracle as O

pytestmark = pytest.mark.gpu

G = 1 << 16  # guard bytes on each side, a multiple of the 256-byte alignment
PAT = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    O.lib()
    assert torch.cuda.is_available()


class Guarded:
    """A byte buffer of n bytes between two patterned margins."""

    def __init__(self, n, device="cuda"):
        self.n = int(n)
        kw = dict(pin_memory=True) if device == "cpu" else dict(device=device)
        self.buf = torch.full((self.n + 2 * G,), PAT, dtype=torch.uint8, **kw)
        self.view = self.buf[G:G + self.n]

    def typed(self, dtype, shape):
        return self.view.view(dtype).view(shape)

    def intact(self):
        return bool((self.buf[:G] == PAT).all()) and bool((self.buf[G + self.n:] == PAT).all())


def guarded_outputs(B, nbest, out_len, device="cuda"):
    tok = Guarded(4 * B * nbest * max(out_len, 1), device)
    ln = Guarded(4 * B * nbest, device)
    sc = Guarded(4 * B * nbest, device)
    views = (tok.typed(torch.int32, (-1,))[:B * nbest * out_len].view(B, nbest, out_len),
             ln.typed(torch.int32, (B, nbest)), sc.typed(torch.float32, (B, nbest)))
    return [tok, ln, sc], views


def frames(seed, B, T, V, blank_boost=2.0):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 1.5, size=(B, T, V))
    x[:, :, 0] += np.where(rng.random((B, T)) < 0.6, blank_boost, 0.0)
    x -= x.max(-1, keepdims=True)
    return (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32)


OFFLINE = [
    ("fused warp kernel", dict(beam=10, nbest=10), (6, 150, 500)),
    ("block kernel, beam 40", dict(beam=40, nbest=7), (3, 120, 300)),
    ("block kernel, beam 128, paged", dict(beam=128, nbest=16, paged=True, page_size=16, max_seq_len=60), (2, 150, 29)),
    ("warp kernel, threshold skipping", dict(beam=16, nbest=16, blank_threshold=0.6), (5, 160, 256)),
    ("warp kernel, boosted", dict(beam=8, nbest=4, max_boost=6), (4, 100, 200)),
    ("block kernel, boosted, word boundary", dict(beam=24, nbest=5, max_boost=3, space_id=5), (3, 90, 64)),
]


@pytest.mark.parametrize("name,kw,shape", OFFLINE, ids=[o[0] for o in OFFLINE])
def test_offline_writes_stay_inside_the_buffers(name, kw, shape):
    B, T, V = shape
    lp = frames(len(name), B, T, V)
    lens = np.random.default_rng(B * T).integers(T // 2, T + 1, size=B).astype(np.int32)
    cfg = D.Config(**kw)
    boost = None
    if kw.get("max_boost"):
        rng = np.random.default_rng(V)
        boost = [{int(c): float(np.float32(rng.uniform(-2, 3))) for c in rng.choice(np.arange(1, V), kw["max_boost"],
                                                                                   replace=False)} for _ in range(B)]
    out_len = min(cfg.max_seq_len, T) if cfg.max_seq_len > 0 else T
    ws = Guarded(D.workspace_size(cfg, B, T, V))
    outs, views = guarded_outputs(B, cfg.c().nbest, out_len)
    D.decode_offline(cfg, torch.from_numpy(lp).cuda(), torch.from_numpy(lens).cuda(), workspace=ws.view,
                     out_len=out_len, outputs=views, boost=boost)
    torch.cuda.synchronize()
    assert ws.intact(), "workspace margins"
    assert all(g.intact() for g in outs), "output margins"
    assert D.read_status(ws.view) & ~D.DEV_BOOST == 0
    assert_same(tuple(v.cpu().numpy() for v in views), oracle_offline(cfg, lp, lens, out_len=out_len, boost=boost),
                name)


@pytest.mark.parametrize("kw", [dict(beam=10, nbest=3), dict(beam=48, nbest=4), dict(beam=20, nbest=2, paged=True)],
                         ids=["warp", "block", "paged"])
def test_streaming_writes_stay_inside_the_state(kw):
    B, T, V = 4, 200, 128
    lp = frames(7, B, T, V)
    mask = (np.random.default_rng(8).random((B, T)) < 0.8).astype(np.uint8)
    cfg = D.Config(max_seq_len=T, **kw)
    st = D.StreamState(cfg, B, V)
    g = Guarded(st.nbytes)
    st.buf = g.view
    st.init()
    x = torch.from_numpy(lp).cuda()
    m = torch.from_numpy(mask).cuda()
    for t0 in range(0, T, 37):
        st.step_chunk(x[:, t0:t0 + 37], is_speech=m[:, t0:t0 + 37])
    outs, views = guarded_outputs(B, cfg.c().nbest, T)
    st.read(out_len=T, outputs=views)
    torch.cuda.synchronize()
    assert g.intact(), "state margins"
    assert all(o.intact() for o in outs), "output margins"
    assert st.status() == 0
    ref = O.decode(lp, None, beam=cfg.beam, nbest=cfg.c().nbest, blank=0, cap=T, out_len=T, mask=mask)
    assert_same(tuple(v.cpu().numpy() for v in views), ref, f"stream {kw}")


def test_host_buffer_call_writes_stay_inside_the_buffers():
    w = synth.workload("bpe", B=6, T=300)
    lp, lens = synth.gen_batch(w, pad="zero")
    cfg = D.Config(beam=10, nbest=5)
    B, T, V = lp.shape
    ws = Guarded(D.host_workspace_size(cfg, B, T, V, T))
    outs, views = guarded_outputs(B, 5, T, device="cpu")
    D.decode_offline_host(cfg, torch.from_numpy(lp).pin_memory(), torch.from_numpy(lens).pin_memory(),
                          workspace=ws.view, out_len=T, outputs=views)
    assert ws.intact(), "device workspace margins"
    assert all(o.intact() for o in outs), "host output margins"
    assert_same(tuple(v.numpy() for v in views), oracle_offline(cfg, lp, lens, out_len=T), "host buffers")
