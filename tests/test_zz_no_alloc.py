"""The no-allocation offline decode (for callers that may not call cudaMalloc).

Some callers cannot allocate device memory -- engine plugins whose host owns
the device heap and forbids allocations from outside it, real-time paths that
must not block in the allocator -- so ctcpb_decode_offline_noalloc keeps its
workspace in a fixed device array inside the library.  This test calls it
through the C ABI twice in a row, on two different batches, and checks each
result against ctcpb_decode_offline with a caller-owned workspace (tokens and
lengths exact, scores within the 1e-4 tolerance of the parity tests) and the
array's device status word (ctcpb_noalloc_read_status) against zero.  It sits
in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

from ctc_prefix_beam_gb300 import build
from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-4


def noalloc_fn():
    build.build()
    L = D.lib()
    fn = L.ctcpb_decode_offline_noalloc
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.restype = I
    fn.argtypes = [ctypes.POINTER(D._Cfg), P, I64, I64, P, I, I, I, P, P, P, I, P]
    return fn


def noalloc_status():
    fn = D.lib().ctcpb_noalloc_read_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    st = ctypes.c_uint32(0xFFFFFFFF)
    rc = fn(ctypes.byref(st))
    assert rc == D.OK, D.status_string(rc)
    return st.value


def call_noalloc(fn, cfg, lp, lens, out_len):
    B, T, V = lp.shape
    c = cfg.c()
    tok = torch.empty((B, c.nbest, out_len), dtype=torch.int32, device=lp.device)
    ln = torch.empty((B, c.nbest), dtype=torch.int32, device=lp.device)
    sc = torch.empty((B, c.nbest), dtype=torch.float32, device=lp.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream(lp.device).cuda_stream)
    rc = fn(ctypes.byref(c), ctypes.c_void_p(lp.data_ptr()), lp.stride(0), lp.stride(1),
            ctypes.c_void_p(lens.data_ptr()), B, T, V, ctypes.c_void_p(tok.data_ptr()),
            ctypes.c_void_p(ln.data_ptr()), ctypes.c_void_p(sc.data_ptr()), out_len, stream)
    return rc, (tok, ln, sc)


def test_noalloc_matches_workspace_decode_twice():
    fn = noalloc_fn()
    dev = torch.device("cuda")
    cfg = D.Config(beam=10, nbest=10)
    for seed in (0, 1):  # two calls in a row, different inputs
        w = synth.workload("bpe", B=8, T=200, seed=seed)
        lp_np, lens_np = synth.gen_batch(w)
        lp = torch.from_numpy(lp_np).to(dev)
        lens = torch.from_numpy(lens_np).to(dev)
        assert D.workspace_size(cfg, 8, 200, 5000) <= (32 << 20)
        rc, (tok, ln, sc) = call_noalloc(fn, cfg, lp, lens, 200)
        assert rc == D.OK, D.status_string(rc)
        rt, rl, rs = D.decode_offline(cfg, lp, lens, out_len=200)
        torch.cuda.synchronize()
        assert torch.equal(ln, rl)
        assert torch.equal(tok, rt)
        assert (sc - rs).abs().max().item() <= SCORE_TOL
        assert noalloc_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = noalloc_fn()
    dev = torch.device("cuda")
    cfg = D.Config(beam=10, nbest=10)
    B, T, V = 256, 2000, 1024
    assert D.workspace_size(cfg, B, T, V) > (32 << 20)
    lp = torch.zeros((1, 1, V), device=dev).expand(B, T, V)  # never read: the call is refused first
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    c = cfg.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    out = torch.empty((1,), dtype=torch.int32, device=dev)
    rc = fn(ctypes.byref(c), ctypes.c_void_p(lp.data_ptr()), T * V, V, ctypes.c_void_p(lens.data_ptr()), B, T, V,
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()), 1,
            stream)
    assert rc == D.ESIZE
