"""Child process of tests/test_gpu_threads.py: first launches of every step
kernel from two host threads at once, in a process that has launched nothing
yet.  Prints one line per thread: its name and "ok" or the failure."""
import os
import sys
import threading

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle as O  # noqa: E402
from ctc_prefix_beam_gb300 import decoder as D  # noqa: E402
from ctc_prefix_beam_gb300 import synth  # noqa: E402


def main():
    dev = torch.device("cuda:0")
    torch.cuda.init()
    w = synth.workload("bpe", B=6, T=120)
    lp_np, lens_np = synth.gen_batch(w)
    jobs = {  # name: (config, expected)
        "warp-a": D.Config(beam=10, nbest=10),
        "warp-b": D.Config(beam=10, nbest=10),
        "block": D.Config(beam=24, nbest=4),
        "paged": D.Config(beam=20, nbest=4, paged=True, page_size=8),
    }
    want = {k: O.decode(lp_np, lens_np, beam=c.beam, nbest=c.nbest) for k, c in jobs.items()}
    lp = torch.from_numpy(lp_np).to(dev)
    lens = torch.from_numpy(lens_np).to(dev)
    out, start = {}, threading.Barrier(len(jobs))

    def run(name):
        try:
            s = torch.cuda.Stream(dev)
            with torch.cuda.stream(s):
                start.wait()
                for _ in range(3):
                    tok, ln, sc = D.decode_offline(jobs[name], lp, lens)
                s.synchronize()
            ot, ol, os_ = want[name]
            ok = (np.array_equal(ln.cpu().numpy(), ol) and np.array_equal(tok.cpu().numpy(), ot) and
                  np.abs(sc.cpu().numpy() - os_).max() <= 1e-4)
            out[name] = "ok" if ok else "differs from the oracle"
        except Exception as e:  # reported to the parent
            out[name] = f"{type(e).__name__}: {e}"

    th = [threading.Thread(target=run, args=(k,)) for k in jobs]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for k in jobs:
        print(k, out.get(k, "did not finish"))


if __name__ == "__main__":
    main()
