"""CPU oracle for batched CTC prefix beam search -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It wraps ``ctcpb_oracle.cpp`` (plain C++17,
float32 in the operation order of "GPU CTC Prefix Beam Search Decoder",
section 3) through ctypes and shares no code with the CUDA decoder.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against brute-force enumeration of CTC alignments in float64, closed forms,
invariants and independent library routines (see each test's docstring).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ctcpb_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libctcpb_oracle.so")
_lock = threading.Lock()
_lib = None

NEG = float(np.finfo(np.float32).min)  # -FLT_MAX


def build_cmd() -> list[str]:
    return ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-pthread", "-o", _LIB, _SRC]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (plain gcc, a few seconds)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.run(build_cmd(), check=True)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
            i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
            L.ctcpb_oracle_F.restype, L.ctcpb_oracle_F.argtypes = ctypes.c_float, [ctypes.c_float]
            L.ctcpb_oracle_F_coefficients.restype = None
            L.ctcpb_oracle_F_coefficients.argtypes = [f32p]
            for n in ("lse", "add"):
                fn = getattr(L, f"ctcpb_oracle_{n}")
                fn.restype, fn.argtypes = ctypes.c_float, [ctypes.c_float, ctypes.c_float]
            L.ctcpb_oracle_log_threshold.restype = ctypes.c_float
            L.ctcpb_oracle_log_threshold.argtypes = [ctypes.c_float]
            L.ctcpb_oracle_map.restype = None
            L.ctcpb_oracle_map.argtypes = [ctypes.c_int, f32p, f32p, f32p, ctypes.c_int64]
            L.ctcpb_oracle_select_frames.restype = ctypes.c_int
            L.ctcpb_oracle_select_frames.argtypes = [
                f32p, ctypes.c_int64, ctypes.c_int64, i32p, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_float, i32p, i32p]
            L.ctcpb_oracle_frame_lists.restype = ctypes.c_int
            L.ctcpb_oracle_frame_lists.argtypes = [
                f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                i32p, f32p, i32p, f32p, f32p, i32p]
            L.ctcpb_oracle_decode.restype = ctypes.c_int
            L.ctcpb_oracle_decode.argtypes = [
                f32p, ctypes.c_int64, ctypes.c_int64, i32p, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_float, ctypes.c_int, i32p, i32p, f32p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_void_p]
            _lib = L
    return _lib


def _f32(x):
    return np.array(x, dtype=np.float32, order="C", copy=True)


def F(d):
    """log(1 + e^-d) for d >= 0 (piecewise Taylor polynomial), elementwise."""
    a = _f32(d)
    out = np.empty_like(a)
    lib().ctcpb_oracle_map(0, a.ravel(), a.ravel(), out.ravel(), a.size)
    return out


def F_coefficients() -> np.ndarray:
    """F's coefficient table: [96 segments, 6] float32, c[k][n] ~ F^(n)(k/4 + 1/8) / n!."""
    out = np.empty((96, 6), np.float32)
    lib().ctcpb_oracle_F_coefficients(out.ravel())
    return out


def lse(a, b):
    """Section 3 logsumexp in float32, elementwise."""
    a, b = np.broadcast_arrays(_f32(a), _f32(b))
    a, b = _f32(a), _f32(b)
    out = np.empty_like(a)
    lib().ctcpb_oracle_map(2, a.ravel(), b.ravel(), out.ravel(), a.size)
    return out


def add(a, b):
    """max(a + b, -FLT_MAX) in float32, elementwise."""
    a, b = np.broadcast_arrays(_f32(a), _f32(b))
    a, b = _f32(a), _f32(b)
    out = np.empty_like(a)
    lib().ctcpb_oracle_map(3, a.ravel(), b.ravel(), out.ravel(), a.size)
    return out


def log_threshold(thr: float) -> float:
    return float(lib().ctcpb_oracle_log_threshold(thr))


def select_frames(lp: np.ndarray, lens: np.ndarray, blank: int, thr: float):
    """Section 3.5 frame selection: (sel [B, T] int32 padded -1, nsel [B])."""
    lp = _f32(lp)
    B, T, V = lp.shape
    sel = np.empty((B, T), np.int32)
    nsel = np.empty(B, np.int32)
    lib().ctcpb_oracle_select_frames(lp.ravel(), T * V, V, np.ascontiguousarray(lens, np.int32),
                                     B, T, blank, thr, sel.ravel(), nsel)
    return sel, nsel


def frame_lists(rows: np.ndarray, blank: int, C: int):
    """Ranked non-blank labels per frame row ([R, V] float32).

    Returns dict(ids [R, C], lps [R, C], cnt [R], lpb [R], front_lp [R], front_id [R]).
    """
    rows = _f32(rows)
    R, V = rows.shape
    ids = np.empty((R, C), np.int32)
    lps = np.empty((R, C), np.float32)
    cnt = np.empty(R, np.int32)
    lpb = np.empty(R, np.float32)
    flp = np.empty(R, np.float32)
    fid = np.empty(R, np.int32)
    lib().ctcpb_oracle_frame_lists(rows.ravel(), V, R, V, blank, C, ids.ravel(), lps.ravel(),
                                   cnt, lpb, flp, fid)
    return dict(ids=ids, lps=lps, cnt=cnt, lpb=lpb, front_lp=flp, front_id=fid)


def decode(lp: np.ndarray, lens=None, *, beam: int, nbest: int | None = None, blank: int = 0,
           cap: int | None = None, thr: float = 1.0, threads: int = 0, out_len: int | None = None,
           mask: np.ndarray | None = None, space: int = -1, boost=None):
    """Offline CTC prefix beam search of a [B, T, V] float32 batch.

    ``cap`` is max_seq_len (default T), ``thr`` the blank-skip threshold
    (>= 1 keeps all frames), ``mask`` an optional [B, T] speech mask (frames
    marked 0 are skipped too), ``space`` the word-boundary label (-1: none),
    ``boost`` the label bonuses: a [B, V] array (0: not boosted) or one
    {label: bonus} dict per row.  Returns (tokens [B, nbest, out_len] int32
    padded with -1, lengths [B, nbest] int32, scores [B, nbest] float32).
    """
    lp = _f32(lp)
    B, T, V = lp.shape
    nbest = beam if nbest is None else nbest
    cap = max(T, 1) if cap is None else cap
    out_len = min(cap, T) if out_len is None else out_len
    lens = np.full(B, T, np.int32) if lens is None else np.ascontiguousarray(lens, np.int32)
    tok = np.empty((B, nbest, out_len), np.int32)
    ln = np.empty((B, nbest), np.int32)
    sc = np.empty((B, nbest), np.float32)
    mk = None
    if mask is not None:
        mk = np.ascontiguousarray(mask, np.uint8)
        if mk.shape != (B, T):
            raise ValueError("mask must be [B, T]")
    bon = None
    if boost is not None:
        if isinstance(boost, np.ndarray):
            bon = np.ascontiguousarray(boost, np.float32)
        else:
            bon = np.zeros((B, V), np.float32)
            for b, row in enumerate(boost):
                for c, v in (row or {}).items():
                    bon[b, int(c)] = np.float32(v)
        if bon.shape != (B, V):
            raise ValueError("boost must be [B, V]")
    rc = lib().ctcpb_oracle_decode(lp.ravel(), T * V, V, lens, B, T, V, beam, nbest, blank, cap,
                                   float(thr), threads, tok.ravel(), ln.ravel(), sc.ravel(),
                                   out_len, None if mk is None else mk.ctypes.data, int(space),
                                   None if bon is None else bon.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle decode rejected its arguments (rc={rc})")
    return tok, ln, sc
