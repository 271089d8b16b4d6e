"""Seeded synthetic CTC log-probability generators.

This module only draws inputs: it holds none of the decoder's arithmetic and is
the one piece of code that both the CUDA path's tests/benchmark and the CPU
oracle consume.  Every tensor is produced as

    float64 logits  ->  float64 log-softmax over V  ->  cast to float32

from a NumPy PCG64 stream.  Each row (utterance) or each 16-frame block of a
stream has its own child seed (``numpy.random.SeedSequence.spawn``), so any
single row can be regenerated on its own and is bit-identical to the same row
of the full batch.

The five workloads follow the decoder's statement of the problem ("GPU CTC
Prefix Beam Search Decoder", sections 3 and 14) and the benchmark workloads
named for it:

    tiny       B=1,   T=50,   V=32,   logits N(0, 2^2), +4 on blank, seed 0
    bpe        B=32,  T=500,  V=5000, N(0,1); per frame w.p. 0.7 blank +8 else one
               uniform non-blank label +8; lengths uniform in [250, 500]
    stream     128 streams x 1600 frames, V=5000, generated as ``bpe``; stream i
               starts at global frame o_i ~ U{0..159}; 16-frame chunks
    char       B=16,  T=1000, V=29, N(0, 1.5^2), +3 on blank, +2 on a label held
               for geometric run lengths (mean 3 frames)
    skip       B=256, T=2000, V=1024, N(0,1); per frame w.p. 0.8 blank +12 else
               one uniform non-blank label +6

Distribution parameters written as N(mu, s) are read as (mean, standard deviation).
"""
from __future__ import annotations

import dataclasses
import hashlib
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "log_softmax64", "gen_row", "gen_batch",
    "gen_lengths", "stream_offsets", "gen_stream_block", "stream_tick",
    "checksum", "workload",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    V: int
    beam: int
    nbest: int
    blank_id: int = 0
    max_seq_len: int = 0          # 0 = decoder default (offline: T)
    blank_threshold: float = 1.0  # >= 1 keeps every frame
    paged: int = 0
    page_size: int = 16
    seed: int = 0
    streaming: bool = False
    chunk: int = 16


WORKLOADS = {
    "tiny": Workload("tiny", B=1, T=50, V=32, beam=4, nbest=4),
    "bpe": Workload("bpe", B=32, T=500, V=5000, beam=10, nbest=10),
    "stream": Workload("stream", B=128, T=1600, V=5000, beam=10, nbest=10,
                       max_seq_len=4096, streaming=True, chunk=16),
    "char": Workload("char", B=16, T=1000, V=29, beam=128, nbest=128,
                     max_seq_len=400, paged=1, page_size=16),
    "skip": Workload("skip", B=256, T=2000, V=1024, beam=16, nbest=16,
                     blank_threshold=0.999),
}


def workload(name: str, **over) -> Workload:
    return dataclasses.replace(WORKLOADS[name], **over)


def log_softmax64(x: np.ndarray) -> np.ndarray:
    """float64 log-softmax over the last axis (input preparation only)."""
    m = x.max(axis=-1, keepdims=True)
    z = x - m
    return z - np.log(np.exp(z).sum(axis=-1, keepdims=True))


def _child(seed: int, *path: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed)] + [int(p) for p in path])
    return np.random.Generator(np.random.PCG64(ss))


_KIND = {"tiny": 1, "bpe": 2, "stream": 3, "char": 4, "skip": 5}


def _logits(kind: str, rng: np.random.Generator, T: int, V: int, blank: int,
            state: Optional[dict] = None) -> np.ndarray:
    if kind == "tiny":
        x = rng.normal(0.0, 2.0, size=(T, V))
        x[:, blank] += 4.0
        return x
    if kind in ("bpe", "stream"):
        x = rng.normal(0.0, 1.0, size=(T, V))
        is_blank = rng.random(T) < 0.7
        lab = rng.integers(1, V, size=T)  # 1..V-1, blank_id 0
        idx = np.where(is_blank, blank, lab)
        x[np.arange(T), idx] += 8.0
        return x
    if kind == "char":
        x = rng.normal(0.0, 1.5, size=(T, V))
        x[:, blank] += 3.0
        t = 0
        # a run of one label for a geometric number of frames, mean 3
        while t < T:
            run = int(rng.geometric(1.0 / 3.0))
            lab = int(rng.integers(1, V))
            x[t:t + run, lab] += 2.0
            t += run
        return x
    if kind == "skip":
        x = rng.normal(0.0, 1.0, size=(T, V))
        is_blank = rng.random(T) < 0.8
        lab = rng.integers(1, V, size=T)
        rows = np.arange(T)
        x[rows[is_blank], blank] += 12.0
        x[rows[~is_blank], lab[~is_blank]] += 6.0
        return x
    raise ValueError(kind)


def gen_row(w: Workload, b: int, T: Optional[int] = None) -> np.ndarray:
    """Row ``b`` of workload ``w`` as float32 [T, V] log-probabilities."""
    T = w.T if T is None else T
    rng = _child(w.seed, _KIND[w.name], b)
    x = _logits(w.name, rng, T, w.V, w.blank_id)
    return log_softmax64(x).astype(np.float32)


def gen_lengths(w: Workload) -> np.ndarray:
    """Per-row valid lengths (int32).  ``bpe`` draws U{250..500}; others use T."""
    if w.name == "bpe":
        rng = _child(w.seed, _KIND[w.name], 1 << 20)
        lo, hi = 250 * w.T // 500, w.T
        return rng.integers(lo, hi + 1, size=w.B).astype(np.int32)
    return np.full(w.B, w.T, dtype=np.int32)


def gen_batch(w: Workload, pad: str = "nan", threads: int = 8,
              rows: Optional[range] = None) -> tuple[np.ndarray, np.ndarray]:
    """Full [B, T, V] float32 batch and its lengths.

    Frames at t >= len_b are padding: ``pad='nan'`` fills them with NaN (so any
    read of padding is visible in the output), ``pad='zero'`` with 0.0.
    """
    lens = gen_lengths(w)
    rows = range(w.B) if rows is None else rows
    out = np.empty((len(rows), w.T, w.V), dtype=np.float32)

    def one(i_b):
        i, b = i_b
        out[i] = gen_row(w, b)
        if lens[b] < w.T:
            out[i, lens[b]:, :] = np.nan if pad == "nan" else 0.0

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(one, enumerate(rows)))
    return out, np.ascontiguousarray(lens[np.asarray(list(rows), dtype=np.int64)])


# ---------------------------------------------------------------- streaming

def stream_offsets(w: Workload) -> np.ndarray:
    """Start frame of each stream on the global tick clock, U{0..159}."""
    rng = _child(w.seed, _KIND[w.name], 1 << 21)
    return rng.integers(0, 160, size=w.B).astype(np.int64)


def gen_stream_block(w: Workload, i: int, blk: int) -> np.ndarray:
    """Local frames [16*blk, 16*blk+16) of stream ``i`` as float32 [16, V]."""
    rng = _child(w.seed, _KIND[w.name], i, blk)
    x = _logits("stream", rng, 16, w.V, w.blank_id)
    return log_softmax64(x).astype(np.float32)


def gen_stream(w: Workload, i: int) -> np.ndarray:
    """All ``w.T`` local frames of stream ``i`` (for the offline comparison)."""
    nb = (w.T + 15) // 16
    return np.concatenate([gen_stream_block(w, i, k) for k in range(nb)])[: w.T]


def stream_tick(w: Workload, k: int, offsets: np.ndarray, cache: dict,
                threads: int = 8) -> tuple[np.ndarray, np.ndarray]:
    """Chunk for global tick ``k`` (global frames [16k, 16k+16)).

    Returns ``(chunk [B, 16, V] float32, n_frames [B] int32)``: stream i's frames
    that fall in the window are packed at rows 0..n-1; the rest is NaN.
    ``cache`` keeps generated 16-frame blocks between ticks.
    """
    C = w.chunk
    chunk = np.full((w.B, C, w.V), np.nan, dtype=np.float32)
    nfr = np.zeros(w.B, dtype=np.int32)
    lo_g, hi_g = C * k, C * k + C

    def one(i):
        a = max(lo_g, int(offsets[i]))
        e = min(hi_g, int(offsets[i]) + w.T)
        if e <= a:
            return
        la, le = a - int(offsets[i]), e - int(offsets[i])  # local frame range
        pos = 0
        f = la
        while f < le:
            blk = f // 16
            key = (i, blk)
            if key not in cache:
                cache[key] = gen_stream_block(w, i, blk)
            take = min(le, 16 * blk + 16) - f
            chunk[i, pos:pos + take] = cache[key][f - 16 * blk: f - 16 * blk + take]
            pos += take
            f += take
        nfr[i] = pos
        # blocks entirely before this tick's window are no longer needed
        for blk in range(max(0, la // 16 - 2), la // 16):
            cache.pop((i, blk), None)

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(one, range(w.B)))
    return chunk, nfr


def n_ticks(w: Workload, offsets: np.ndarray) -> int:
    return int((int(offsets.max()) + w.T + w.chunk - 1) // w.chunk)


def checksum(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()[:16]
