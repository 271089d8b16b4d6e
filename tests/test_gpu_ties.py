"""The CUDA path breaks ties by the rule, on the hand-derived decodes of
tests/tie_cases.py ("GPU CTC Prefix Beam Search Decoder", sections 3.3 and
3.4.4-3.4.6): expected N-best lists written out from the rule, not taken from
the oracle.  Offline through the warp kernel, the block kernel (paged storage) and the host-buffer call, and streamed one frame at a time."""
import numpy as np
import pytest
import torch

import tie_cases
from ctc_prefix_beam_gb300 import decoder as D

pytestmark = pytest.mark.gpu


def _offline(lp, beam, nbest, blank, **kw):
    cfg = D.Config(beam=beam, nbest=nbest, blank_id=blank, **kw)
    tok, ln, sc = D.decode_offline(cfg, torch.from_numpy(np.ascontiguousarray(lp)).cuda())
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), sc.cpu().numpy()


def _host(lp, beam, nbest, blank):
    cfg = D.Config(beam=beam, nbest=nbest, blank_id=blank)
    tok, ln, sc = D.decode_offline_host(cfg, torch.from_numpy(np.ascontiguousarray(lp)).pin_memory(), None,
                                        device="cuda:0")
    return tok.numpy(), ln.numpy(), sc.numpy()


def _streamed(lp, beam, nbest, blank):
    T = lp.shape[1]
    st = D.StreamState(D.Config(beam=beam, nbest=nbest, blank_id=blank, max_seq_len=T), 1, lp.shape[2],
                       device="cuda:0")
    x = torch.from_numpy(np.ascontiguousarray(lp)).cuda()
    for t in range(T):
        st.step(x[:, t])
    tok, ln, sc = (v.cpu().numpy() for v in st.read(out_len=T))
    assert st.status() == 0
    return tok, ln, sc


@pytest.mark.parametrize("path", ["warp", "block", "host", "stream"])
def test_gpu_breaks_ties_by_the_rule(path):
    if path == "warp":
        fn = _offline
    elif path == "block":
        # paged token storage always runs the block kernel, at the cases' own beams
        fn = lambda lp, beam, nbest, blank: _offline(lp, beam, nbest, blank, paged=True, page_size=4)
    elif path == "host":
        fn = _host
    else:
        fn = _streamed
    res = tie_cases.check(fn)
    assert all(res.values()), [k for k, v in res.items() if not v]
