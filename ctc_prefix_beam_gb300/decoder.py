"""Thin Python binding of the C-ABI decoder library (include/ctcpb.h).

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current CUDA stream.  The
library is loaded on first use; if it has not been built, calls raise
``RuntimeError`` -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

OK, EINVAL, ENULL, EALIGN, ESIZE, ECUDA = 0, -1, -2, -3, -4, -5
DEV_HEADER, DEV_PAGES, DEV_TIMEOUT, DEV_OVERFLOW, DEV_BOOST = 0x1, 0x2, 0x4, 0x8, 0x10
NEG = -3.4028234663852886e38


class CtcpbError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class _Cfg(ctypes.Structure):
    _fields_ = [("beam", ctypes.c_int32), ("nbest", ctypes.c_int32), ("blank_id", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("blank_threshold", ctypes.c_float),
                ("paged", ctypes.c_int32), ("page_size", ctypes.c_int32), ("list_len", ctypes.c_int32),
                ("word_boundary", ctypes.c_int32), ("space_id", ctypes.c_int32), ("max_boost", ctypes.c_int32)]


class _Boost(ctypes.Structure):
    _fields_ = [("row_ptr", ctypes.c_void_p), ("tokens", ctypes.c_void_p), ("bonus", ctypes.c_void_p)]


@dataclasses.dataclass
class Config:
    """Mirror of ``ctcpb_config`` (section 11 of the decoder's description)."""
    beam: int = 10
    nbest: Optional[int] = None
    blank_id: int = 0
    max_seq_len: int = 0
    blank_threshold: float = 1.0
    paged: bool = False
    page_size: int = 16
    list_len: int = 0
    space_id: int = -1  # word-boundary label (sections 3.4.1/3.4.2), -1: none
    max_boost: int = 0  # boosted labels per row (0: no label boosting)

    def c(self) -> _Cfg:
        return _Cfg(self.beam, self.beam if self.nbest is None else self.nbest, self.blank_id,
                    self.max_seq_len, self.blank_threshold, int(bool(self.paged)), self.page_size,
                    self.list_len, 1 if self.space_id >= 0 else 0, max(self.space_id, 0), self.max_boost)


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load the decoder library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(f"decoder library not built: {path} is missing "
                                   "(run `python -m ctc_prefix_beam_gb300.build`)")
            L = ctypes.CDLL(path)
            P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            cfgp = ctypes.POINTER(_Cfg)
            sig = {
                "ctcpb_status_string": (ctypes.c_char_p, [I]),
                "ctcpb_list_len": (I, [cfgp, I]),
                "ctcpb_workspace_size": (I, [cfgp, I, I, I, ctypes.POINTER(SZ)]),
                "ctcpb_decode_offline": (I, [cfgp, P, I64, I64, P, I, I, I, P, SZ, P, P, P, I, P]),
                "ctcpb_decode_offline_staged": (I, [cfgp, P, I64, I64, P, I, I, I, P, SZ, P, P, P, I,
                                                    ctypes.c_uint32, P]),
                "ctcpb_decode_offline_boosted": (I, [cfgp, ctypes.POINTER(_Boost), P, I64, I64, P, I, I, I, P, SZ,
                                                     P, P, P, I, P]),
                "ctcpb_stream_set_boost": (I, [cfgp, P, SZ, I, I, ctypes.POINTER(_Boost), P]),
                "ctcpb_host_workspace_size": (I, [cfgp, I, I, I, I, ctypes.POINTER(SZ)]),
                "ctcpb_decode_offline_host": (I, [cfgp, P, I64, I64, P, I, I, I, P, SZ, P, P, P, I, P]),
                "ctcpb_decode_offline_host_boosted": (I, [cfgp, ctypes.POINTER(_Boost), P, I64, I64, P, I, I, I, P,
                                                          SZ, P, P, P, I, P]),
                "ctcpb_state_size": (I, [cfgp, I, I, ctypes.POINTER(SZ)]),
                "ctcpb_stream_init": (I, [cfgp, P, SZ, I, I, P]),
                "ctcpb_stream_step_chunk": (I, [cfgp, P, SZ, I, I, P, I64, I64, P, I, P]),
                "ctcpb_stream_step_chunk_masked": (I, [cfgp, P, SZ, I, I, P, I64, I64, P, P, I64, I, P]),
                "ctcpb_stream_step": (I, [cfgp, P, SZ, I, I, P, I64, P, P]),
                "ctcpb_selftest_waits": (I, [P, I, ctypes.c_longlong, P, P]),
                "ctcpb_read_state": (I, [cfgp, P, SZ, I, I, P, P, P, I, P]),
                "ctcpb_read_status": (I, [P, ctypes.POINTER(ctypes.c_uint32)]),
                "ctcpb_read_counters": (I, [P, ctypes.POINTER(ctypes.c_uint32)]),
                "ctcpb_select_frames": (I, [cfgp, P, I64, I64, P, I, I, I, P, P, P]),
                "ctcpb_topk_prepass": (I, [cfgp, P, I64, I, I, P, P, P, P, P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = res, args
            _lib = L
    return _lib


def status_string(code: int) -> str:
    try:
        return lib().ctcpb_status_string(code).decode()
    except RuntimeError:
        return "library not loaded"


def _check(rc: int, what: str):
    if rc != OK:
        raise CtcpbError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _row_strides(x: torch.Tensor):
    """(batch, time) element strides of a [B, T, V] tensor as the library takes
    them.  A dimension of extent 1 is never stepped over, and torch and NumPy
    leave its stride arbitrary (often 0: an expanded or inserted axis), so it
    is given a valid one instead."""
    B, T, V = x.shape[0], x.shape[1], x.shape[2]
    st = x.stride(1) if T > 1 else V
    sb = x.stride(0) if B > 1 else st * max(T, 1)
    return sb, st


def _f32_3d(lp: torch.Tensor) -> torch.Tensor:
    if lp.dtype != torch.float32 or lp.dim() != 3 or not lp.is_cuda:
        raise ValueError("log_prob must be a CUDA float32 tensor [B, T, V]")
    if lp.stride(2) != 1:
        lp = lp.contiguous()
    return lp


def _cuda_device(device) -> torch.device:
    """``device`` as an indexed CUDA device (``"cuda"`` is the current one)."""
    d = torch.device(device)
    if d.type != "cuda":
        raise ValueError(f"{device} is not a CUDA device")
    return d if d.index is not None else torch.device("cuda", torch.cuda.current_device())


def _call(dev: torch.device, fn, *args):
    """Call a library entry point with ``dev`` current: the library launches on
    the current CUDA device."""
    with torch.cuda.device(dev):
        return fn(*args)


def _check_buf(buf: torch.Tensor, need: int, device: torch.device, what: str) -> int:
    """A caller's workspace or state: contiguous, on ``device``, at least
    ``need`` bytes.  Returns its size in bytes."""
    if not isinstance(buf, torch.Tensor) or buf.device != device or not buf.is_contiguous():
        raise ValueError(f"{what} must be a contiguous tensor on {device}")
    nbytes = buf.numel() * buf.element_size()
    if nbytes < need:
        raise ValueError(f"{what} holds {nbytes} bytes, {need} are needed")
    return nbytes


def _check_outputs(outputs, B: int, nbest: int, out_len: int, device: torch.device):
    """Caller-supplied (tokens, lengths, scores): the library writes exactly
    B*nbest*out_len, B*nbest and B*nbest elements through plain pointers."""
    tok, ln, sc = outputs
    for t, dt, n, name in ((tok, torch.int32, B * nbest * out_len, "tokens"), (ln, torch.int32, B * nbest, "lengths"),
                           (sc, torch.float32, B * nbest, "scores")):
        if not isinstance(t, torch.Tensor) or t.dtype != dt or t.device != device or not t.is_contiguous() \
                or t.numel() != n:
            raise ValueError(f"output {name} must be a contiguous {dt} tensor of {n} elements on {device}")
    return tok, ln, sc


def _alloc(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def list_len(cfg: Config, V: int) -> int:
    rc = lib().ctcpb_list_len(ctypes.byref(cfg.c()), V)
    if rc < 0:
        raise CtcpbError(rc, "list_len")
    return rc


def workspace_size(cfg: Config, B: int, T: int, V: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().ctcpb_workspace_size(ctypes.byref(cfg.c()), B, T, V, ctypes.byref(n)), "workspace_size")
    return n.value


def state_size(cfg: Config, B: int, V: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().ctcpb_state_size(ctypes.byref(cfg.c()), B, V, ctypes.byref(n)), "state_size")
    return n.value


def _outputs(B, nbest, out_len, device):
    return (torch.empty((B, nbest, out_len), dtype=torch.int32, device=device),
            torch.empty((B, nbest), dtype=torch.int32, device=device),
            torch.empty((B, nbest), dtype=torch.float32, device=device))


STAGE_INIT, STAGE_SELECT, STAGE_RANK, STAGE_STEPS, STAGE_OUTPUT, STAGE_ALL = 0x1, 0x2, 0x4, 0x8, 0x10, 0x1f


def boost_tables(boost, B: int, device):
    """Label boosts in the compressed-row form of ``ctcpb_boost``: from one
    {label: bonus} dict (or None) per row, or from (row_ptr, tokens, bonus)
    tensors, which are moved to ``device``."""
    if isinstance(boost, (tuple, list)) and len(boost) == 3 and all(isinstance(x, torch.Tensor) for x in boost):
        rp, tk, bn = boost
    else:
        rows = list(boost)
        if len(rows) != B:
            raise ValueError("boost needs one entry per row")
        rp, tk, bn = [0], [], []
        for row in rows:
            for c, v in (row or {}).items():
                tk.append(int(c))
                bn.append(float(v))
            rp.append(len(tk))
        rp, tk, bn = torch.tensor(rp, dtype=torch.int32), torch.tensor(tk, dtype=torch.int32), \
            torch.tensor(bn, dtype=torch.float32)
    rp = rp.to(device=device, dtype=torch.int32).contiguous()
    tk = tk.to(device=device, dtype=torch.int32).contiguous()
    bn = bn.to(device=device, dtype=torch.float32).contiguous()
    if rp.numel() != B + 1:
        raise ValueError("row_ptr must hold B + 1 offsets")
    if tk.numel() == 0:  # the arrays must be non-null even when no row boosts a label
        tk = torch.zeros(1, dtype=torch.int32, device=device)
        bn = torch.zeros(1, dtype=torch.float32, device=device)
    return rp, tk, bn


def _boost_arg(tables):
    rp, tk, bn = tables
    return _Boost(rp.data_ptr(), tk.data_ptr(), bn.data_ptr())


def decode_offline(cfg: Config, log_prob: torch.Tensor, seq_lengths: Optional[torch.Tensor] = None, *,
                   workspace: Optional[torch.Tensor] = None, out_len: Optional[int] = None, outputs=None,
                   stages: int = STAGE_ALL, boost=None):
    """Offline decode of a CUDA float32 [B, T, V] batch.

    Returns (tokens [B, nbest, out_len] int32 padded -1, lengths [B, nbest]
    int32, scores [B, nbest] float32), all on the device.  ``out_len``
    defaults to min(max_seq_len, T) (T when the cap is unset).  ``boost``:
    the rows' label boosts (``boost_tables``; needs ``cfg.max_boost``).
    """
    lp = _f32_3d(log_prob)
    dev = lp.device
    B, T, V = lp.shape
    c = cfg.c()
    nbest = c.nbest
    if out_len is None:
        out_len = min(cfg.max_seq_len, T) if cfg.max_seq_len > 0 else T
    if seq_lengths is not None:
        if seq_lengths.dtype != torch.int32 or seq_lengths.device != dev or seq_lengths.numel() != B:
            raise ValueError(f"seq_lengths must be an int32 tensor [B] on {dev}")
        seq_lengths = seq_lengths.contiguous()
    need = workspace_size(cfg, B, T, V)
    if workspace is None:
        workspace = _alloc(need, dev)
    ws_bytes = _check_buf(workspace, need, dev, "workspace")
    tok, ln, sc = _outputs(B, nbest, out_len, dev) if outputs is None else _check_outputs(outputs, B, nbest, out_len,
                                                                                          dev)
    if boost is not None:
        if stages != STAGE_ALL:
            raise ValueError("a boosted decode runs every stage")
        tables = boost_tables(boost, B, dev)
        rc = _call(dev, lib().ctcpb_decode_offline_boosted, ctypes.byref(c), ctypes.byref(_boost_arg(tables)),
                   _ptr(lp), *_row_strides(lp), _ptr(seq_lengths), B, T, V, _ptr(workspace), ws_bytes,
                   _ptr(tok), _ptr(ln), _ptr(sc), out_len, _stream(dev))
    elif stages == STAGE_ALL:
        rc = _call(dev, lib().ctcpb_decode_offline, ctypes.byref(c), _ptr(lp), *_row_strides(lp),
                   _ptr(seq_lengths), B, T, V, _ptr(workspace), ws_bytes, _ptr(tok), _ptr(ln), _ptr(sc), out_len,
                   _stream(dev))
    else:
        rc = _call(dev, lib().ctcpb_decode_offline_staged, ctypes.byref(c), _ptr(lp), *_row_strides(lp),
                   _ptr(seq_lengths), B, T, V, _ptr(workspace), ws_bytes, _ptr(tok), _ptr(ln), _ptr(sc), out_len,
                   stages, _stream(dev))
    _check(rc, "decode_offline")
    return tok, ln, sc


def host_workspace_size(cfg: Config, B: int, T: int, V: int, out_len: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().ctcpb_host_workspace_size(ctypes.byref(cfg.c()), B, T, V, out_len, ctypes.byref(n)),
           "host_workspace_size")
    return n.value


def decode_offline_host(cfg: Config, log_prob: torch.Tensor, seq_lengths: Optional[torch.Tensor] = None, *,
                        workspace: Optional[torch.Tensor] = None, out_len: Optional[int] = None, outputs=None,
                        device="cuda", synchronize: bool = True, boost=None):
    """Offline decode of a HOST float32 [B, T, V] batch into host outputs
    (``ctcpb_decode_offline_host``): the frames are copied in chunks while the
    decode runs.  Page-locked tensors (``pin_memory()``) keep the call
    asynchronous; the outputs are valid once the device's current stream is
    synchronised, which this function does unless ``synchronize`` is False.
    ``boost``: the rows' label boosts (``boost_tables``; needs ``cfg.max_boost``)."""
    if log_prob.dtype != torch.float32 or log_prob.dim() != 3 or log_prob.is_cuda:
        raise ValueError("log_prob must be a host float32 tensor [B, T, V]")
    if log_prob.stride(2) != 1:
        log_prob = log_prob.contiguous()
    B, T, V = log_prob.shape
    c = cfg.c()
    if out_len is None:
        out_len = min(cfg.max_seq_len, T) if cfg.max_seq_len > 0 else T
    if seq_lengths is not None:
        if seq_lengths.dtype != torch.int32 or seq_lengths.is_cuda or seq_lengths.numel() != B:
            raise ValueError("seq_lengths must be a host int32 tensor [B]")
        seq_lengths = seq_lengths.contiguous()
    dev = _cuda_device(device)
    need = host_workspace_size(cfg, B, T, V, out_len)
    if workspace is None:
        workspace = _alloc(need, dev)
    ws_bytes = _check_buf(workspace, need, dev, "workspace")
    if outputs is None:
        pin = log_prob.is_pinned()
        outputs = (torch.empty((B, c.nbest, out_len), dtype=torch.int32, pin_memory=pin),
                   torch.empty((B, c.nbest), dtype=torch.int32, pin_memory=pin),
                   torch.empty((B, c.nbest), dtype=torch.float32, pin_memory=pin))
    tok, ln, sc = _check_outputs(outputs, B, c.nbest, out_len, torch.device("cpu"))
    if boost is not None:
        tables = boost_tables(boost, B, dev)
        rc = _call(dev, lib().ctcpb_decode_offline_host_boosted, ctypes.byref(c), ctypes.byref(_boost_arg(tables)),
                   _ptr(log_prob), *_row_strides(log_prob), _ptr(seq_lengths), B, T, V,
                   _ptr(workspace), ws_bytes, _ptr(tok), _ptr(ln), _ptr(sc), out_len, _stream(dev))
    else:
        rc = _call(dev, lib().ctcpb_decode_offline_host, ctypes.byref(c), _ptr(log_prob),
                   *_row_strides(log_prob), _ptr(seq_lengths), B, T, V, _ptr(workspace), ws_bytes, _ptr(tok), _ptr(ln),
                   _ptr(sc), out_len, _stream(dev))
    _check(rc, "decode_offline_host")
    if synchronize:
        torch.cuda.current_stream(dev).synchronize()
    return tok, ln, sc


class StreamState:
    """A device buffer holding B streams' beam state (caller-owned memory)."""

    def __init__(self, cfg: Config, B: int, V: int, device="cuda"):
        self.cfg, self.B, self.V = cfg, B, V
        self.nbytes = state_size(cfg, B, V)
        self.buf = _alloc(self.nbytes, _cuda_device(device))
        self.init()

    def _state(self):
        """(device, state bytes) of the buffer, checked before every call."""
        dev = self.buf.device
        return dev, _check_buf(self.buf, self.nbytes, dev, "state")

    def _on(self, t: Optional[torch.Tensor], dev: torch.device, what: str):
        if t is not None and t.device != dev:
            raise ValueError(f"{what} must be on the state's device {dev}")

    def init(self):
        dev, nb = self._state()
        _check(_call(dev, lib().ctcpb_stream_init, ctypes.byref(self.cfg.c()), _ptr(self.buf), nb, self.B, self.V,
                     _stream(dev)), "stream_init")

    def set_boost(self, boost):
        """Replace every stream's label boosts (``boost_tables``) from the next frame on."""
        dev, nb = self._state()
        tables = boost_tables(boost, self.B, dev)
        _check(_call(dev, lib().ctcpb_stream_set_boost, ctypes.byref(self.cfg.c()), _ptr(self.buf), nb, self.B,
                     self.V, ctypes.byref(_boost_arg(tables)), _stream(dev)), "stream_set_boost")

    def step_chunk(self, lp_chunk: torch.Tensor, n_frames: Optional[torch.Tensor] = None,
                   is_speech: Optional[torch.Tensor] = None):
        """Decode one chunk [B, chunk_T, V] for every stream.  ``n_frames``
        (CUDA int32 [B]) limits stream b to its first n_frames[b] rows;
        ``is_speech`` (CUDA uint8 [B, chunk_T]) skips the frames it marks 0."""
        dev, nb = self._state()
        lp = _f32_3d(lp_chunk)
        self._on(lp, dev, "the chunk")
        if lp.shape[0] != self.B or lp.shape[2] != self.V:
            raise ValueError("chunk must be [B, chunk_T, V] for this state")
        if n_frames is not None:
            if n_frames.dtype != torch.int32 or n_frames.numel() != self.B:
                raise ValueError("n_frames must be an int32 tensor [B]")
            self._on(n_frames, dev, "n_frames")
            n_frames = n_frames.contiguous()
        if is_speech is not None:
            if is_speech.dtype != torch.uint8 or is_speech.dim() != 2 or is_speech.shape[0] != self.B \
                    or is_speech.shape[1] < lp.shape[1] or is_speech.stride(1) != 1:
                raise ValueError("is_speech must be a uint8 tensor [B, >= chunk_T] with unit column stride")
            self._on(is_speech, dev, "is_speech")
            _check(_call(dev, lib().ctcpb_stream_step_chunk_masked, ctypes.byref(self.cfg.c()), _ptr(self.buf), nb,
                         self.B, self.V, _ptr(lp), *_row_strides(lp), _ptr(n_frames), _ptr(is_speech),
                         is_speech.stride(0), lp.shape[1], _stream(dev)), "stream_step_chunk_masked")
            return
        _check(_call(dev, lib().ctcpb_stream_step_chunk, ctypes.byref(self.cfg.c()), _ptr(self.buf), nb, self.B,
                     self.V, _ptr(lp), *_row_strides(lp), _ptr(n_frames), lp.shape[1], _stream(dev)),
               "stream_step_chunk")

    def step(self, lp_frame: torch.Tensor, is_speech: Optional[torch.Tensor] = None):
        """Decode one frame [B, V] for every stream.  ``is_speech`` (CUDA uint8
        [B]) skips the streams it marks 0; their frame counters still advance."""
        dev, nb = self._state()
        if lp_frame.dtype != torch.float32 or not lp_frame.is_cuda or lp_frame.dim() != 2:
            raise ValueError("frame must be a CUDA float32 tensor [B, V]")
        lp = lp_frame if lp_frame.stride(1) == 1 else lp_frame.contiguous()
        self._on(lp, dev, "the frame")
        if lp.shape[0] != self.B or lp.shape[1] != self.V:
            raise ValueError("frame must be [B, V] for this state")
        if is_speech is not None:
            if is_speech.dtype != torch.uint8 or is_speech.shape != (self.B,):
                raise ValueError("is_speech must be a uint8 tensor [B]")
            self._on(is_speech, dev, "is_speech")
            is_speech = is_speech.contiguous()
        _check(_call(dev, lib().ctcpb_stream_step, ctypes.byref(self.cfg.c()), _ptr(self.buf), nb, self.B, self.V,
                     _ptr(lp), lp.stride(0) if self.B > 1 else self.V, _ptr(is_speech), _stream(dev)),
               "stream_step")

    def read(self, out_len: Optional[int] = None, outputs=None):
        """The current N best of every stream; the state is not modified."""
        dev, nb = self._state()
        c = self.cfg.c()
        if out_len is None:
            out_len = self.cfg.max_seq_len if self.cfg.max_seq_len > 0 else 4096
        tok, ln, sc = _outputs(self.B, c.nbest, out_len, dev) if outputs is None else \
            _check_outputs(outputs, self.B, c.nbest, out_len, dev)
        _check(_call(dev, lib().ctcpb_read_state, ctypes.byref(c), _ptr(self.buf), nb, self.B, self.V, _ptr(tok),
                     _ptr(ln), _ptr(sc), out_len, _stream(dev)), "read_state")
        return tok, ln, sc

    def status(self) -> int:
        return read_status(self.buf)


def read_status(buf: torch.Tensor) -> int:
    v = ctypes.c_uint32()
    _check(_call(buf.device, lib().ctcpb_read_status, _ptr(buf), ctypes.byref(v)), "read_status")
    return v.value


def selftest_waits(flags: torch.Tensor, max_spins: int = 1000) -> tuple:
    """Run the bounded-wait self-test (``ctcpb_selftest_waits``) on a CUDA
    uint32 flag array; returns (flags found set in order, flag-wait status,
    barrier-wait status), the statuses CTCPB_DEV_TIMEOUT when a wait gave up."""
    if flags.dtype != torch.int32 or not flags.is_cuda or flags.dim() != 1:
        raise ValueError("flags must be a 1-D CUDA int32 tensor (read as uint32)")
    flags = flags.contiguous()
    out = torch.zeros(3, dtype=torch.int32, device=flags.device)
    _check(_call(flags.device, lib().ctcpb_selftest_waits, _ptr(flags), flags.numel(), max_spins, _ptr(out),
                 _stream(flags.device)), "selftest_waits")
    return tuple(int(v) for v in out.cpu())


def read_counters(buf: torch.Tensor) -> dict:
    v = (ctypes.c_uint32 * 6)()
    _check(_call(buf.device, lib().ctcpb_read_counters, _ptr(buf), v), "read_counters")
    return dict(steps=v[0], unproven=v[1], exhaustive=v[2], frame_scans=v[3], hash_merges=v[4], fused=v[5])


def select_frames(cfg: Config, log_prob: torch.Tensor, seq_lengths: Optional[torch.Tensor] = None):
    lp = _f32_3d(log_prob)
    dev = lp.device
    B, T, V = lp.shape
    if seq_lengths is not None:
        if seq_lengths.dtype != torch.int32 or seq_lengths.device != dev or seq_lengths.numel() != B:
            raise ValueError(f"seq_lengths must be an int32 tensor [B] on {dev}")
        seq_lengths = seq_lengths.contiguous()
    sel = torch.empty((B, T), dtype=torch.int32, device=dev)
    nsel = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(_call(dev, lib().ctcpb_select_frames, ctypes.byref(cfg.c()), _ptr(lp), *_row_strides(lp),
                 _ptr(seq_lengths), B, T, V, _ptr(sel), _ptr(nsel), _stream(dev)), "select_frames")
    return sel, nsel


def topk_prepass(cfg: Config, rows: torch.Tensor):
    """Ranked labels of each row of a CUDA float32 [R, V] tensor (section 3.4.7)."""
    if rows.dtype != torch.float32 or rows.dim() != 2 or not rows.is_cuda or rows.stride(1) != 1:
        raise ValueError("rows must be a CUDA float32 [R, V] tensor with V contiguous")
    R, V = rows.shape
    L = list_len(cfg, V)
    dev = rows.device
    ids = torch.empty((R, L), dtype=torch.int32, device=dev)
    lps = torch.empty((R, L), dtype=torch.float32, device=dev)
    cnt = torch.empty((R,), dtype=torch.int32, device=dev)
    lpb = torch.empty((R,), dtype=torch.float32, device=dev)
    flp = torch.empty((R,), dtype=torch.float32, device=dev)
    fid = torch.empty((R,), dtype=torch.int32, device=dev)
    _check(_call(dev, lib().ctcpb_topk_prepass, ctypes.byref(cfg.c()), _ptr(rows), rows.stride(0), R, V, _ptr(ids),
                 _ptr(lps), _ptr(cnt), _ptr(lpb), _ptr(flp), _ptr(fid), _stream(dev)), "topk_prepass")
    return dict(ids=ids, lps=lps, cnt=cnt, lpb=lpb, front_lp=flp, front_id=fid)
