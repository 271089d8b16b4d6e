"""The library from several host threads and on several devices of one process.

A kernel's dynamic shared-memory limit is an attribute per device, which the
launchers raise once per device under a lock.  These tests make the first
launch of each step kernel happen from several host threads at once (in a fresh
process, so no launch came earlier), and decode on every visible device of one
process; each result must match the oracle."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_first_launches_from_several_host_threads():
    p = subprocess.run([sys.executable, os.path.join(HERE, "threads_child.py")], capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = dict(l.split(" ", 1) for l in p.stdout.strip().splitlines())
    assert lines and all(v == "ok" for v in lines.values()), lines


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two visible GPUs")
def test_decode_on_every_device_of_one_process():
    w = synth.workload("bpe", B=4, T=80)
    lp_np, lens_np = synth.gen_batch(w)
    for beam, paged in ((10, False), (24, True)):
        cfg = D.Config(beam=beam, nbest=4, paged=paged, page_size=8)
        ot, ol, os_ = O.decode(lp_np, lens_np, beam=beam, nbest=4)
        for d in range(torch.cuda.device_count()):
            dev = torch.device(f"cuda:{d}")
            tok, ln, sc = D.decode_offline(cfg, torch.from_numpy(lp_np).to(dev), torch.from_numpy(lens_np).to(dev))
            torch.cuda.synchronize(dev)
            assert np.array_equal(ln.cpu().numpy(), ol) and np.array_equal(tok.cpu().numpy(), ot), d
            assert np.abs(sc.cpu().numpy() - os_).max() <= 1e-4, d
