"""The one-launch pre-pass + steps path (a cooperative kernel whose ranking
blocks publish records that the step warps consume as they arrive) against
the two-kernel path and the oracle."""
import numpy as np
import pytest
import torch

from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import assert_same, cfg_of, oracle_offline

pytestmark = pytest.mark.gpu


def _run(cfg, lp, lens, split):
    dev = torch.device("cuda")
    x = torch.from_numpy(np.ascontiguousarray(lp)).to(dev)
    ln = torch.from_numpy(np.ascontiguousarray(lens, np.int32)).to(dev)
    B, T, V = lp.shape
    ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device=dev)
    out_len = T
    outs = (torch.empty((B, cfg.nbest, out_len), dtype=torch.int32, device=dev),
            torch.empty((B, cfg.nbest), dtype=torch.int32, device=dev),
            torch.empty((B, cfg.nbest), dtype=torch.float32, device=dev))
    if split == "stages":  # every stage in a call of its own: the reset and the selection apart too
        for stage in (D.STAGE_INIT, D.STAGE_SELECT, D.STAGE_RANK, D.STAGE_STEPS, D.STAGE_OUTPUT):
            D.decode_offline(cfg, x, ln, workspace=ws, outputs=outs, out_len=out_len, stages=stage)
    elif split:  # the pre-pass and the steps in two calls: two kernels
        D.decode_offline(cfg, x, ln, workspace=ws, outputs=outs, out_len=out_len,
                         stages=D.STAGE_INIT | D.STAGE_SELECT | D.STAGE_RANK)
        D.decode_offline(cfg, x, ln, workspace=ws, outputs=outs, out_len=out_len,
                         stages=D.STAGE_STEPS | D.STAGE_OUTPUT)
    else:
        D.decode_offline(cfg, x, ln, workspace=ws, outputs=outs, out_len=out_len)
    torch.cuda.synchronize()
    assert D.read_status(ws) == 0
    return tuple(o.cpu().numpy() for o in outs), D.read_counters(ws)


@pytest.mark.parametrize("name,over", [("bpe", dict(B=8, T=200)), ("skip", dict(B=24, T=300)),
                                       ("bpe", dict(B=40, T=64))])
def test_fused_equals_two_kernels_and_oracle(name, over):
    w = synth.workload(name, **over)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w)
    fused, cf = _run(cfg, lp, lens, split=False)
    split, cs = _run(cfg, lp, lens, split=True)
    staged, cg = _run(cfg, lp, lens, split="stages")
    assert cf["fused"] == 1 and cs["fused"] == 0 and cg["fused"] == 0
    for a, b, c in zip(fused, split, staged):
        assert np.array_equal(a, b) and np.array_equal(a, c)
    assert cf["steps"] == cs["steps"] == cg["steps"]
    assert_same(fused, oracle_offline(cfg, lp, lens), f"{name}{over}")


def test_fused_streaming_tiles_match_offline():
    w = synth.workload("bpe", B=12, T=150)
    lp, lens = synth.gen_batch(w, pad="zero")
    lens[:] = w.T
    cfg = cfg_of(w, max_seq_len=150)
    dev = torch.device("cuda")
    st = D.StreamState(cfg, w.B, w.V, device=dev)
    x = torch.from_numpy(lp).to(dev)
    for t0 in range(0, w.T, 70):  # chunks spanning several 64-frame tiles
        st.step_chunk(x[:, t0:t0 + 70])
    tok, ln, sc = st.read(out_len=w.T)
    torch.cuda.synchronize()
    assert st.status() == 0
    assert D.read_counters(st.buf)["fused"] >= 1
    off = _run(cfg, lp, lens, split=False)[0]
    assert np.array_equal(ln.cpu().numpy(), off[1])
    assert np.array_equal(tok.cpu().numpy(), off[0])
    assert np.array_equal(sc.cpu().numpy(), off[2])
