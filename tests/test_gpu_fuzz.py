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
