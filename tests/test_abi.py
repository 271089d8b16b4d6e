"""The C-ABI library builds, loads, exports every symbol include/ctcpb.h declares,
and rejects bad arguments on the host (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

from ctc_prefix_beam_gb300 import build as B
from ctc_prefix_beam_gb300 import decoder as D

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return D.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ctcpb.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ctcpb_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert D.status_string(code) not in ("", "unknown status")
    assert D.status_string(-99) == "unknown status"


def cfg(**kw):
    base = dict(beam=10, nbest=10, blank_id=0, max_seq_len=0, blank_threshold=1.0, paged=False,
                page_size=16, list_len=0)
    base.update(kw)
    return D.Config(**base)


@pytest.mark.parametrize("bad", [dict(beam=0), dict(beam=129), dict(nbest=11), dict(nbest=0),
                                 dict(blank_id=-1), dict(blank_id=5000), dict(paged=True, page_size=0),
                                 dict(list_len=-1), dict(blank_threshold=float("nan")),
                                 dict(space_id=5000)])
def test_size_query_rejects_bad_config(lib, bad):
    with pytest.raises(D.CtcpbError) as e:
        D.workspace_size(cfg(**bad), 4, 10, 5000)
    assert e.value.code == D.EINVAL


def test_word_boundary_fields(lib):
    # a zero-initialised config has no word-boundary label; word_boundary must be 0 or 1
    c = cfg().c()
    c.word_boundary, c.space_id = 0, 9999  # ignored while word_boundary is 0
    n = ctypes.c_size_t()
    assert lib.ctcpb_workspace_size(ctypes.byref(c), 2, 10, 50, ctypes.byref(n)) == D.OK
    c.word_boundary = 2
    assert lib.ctcpb_workspace_size(ctypes.byref(c), 2, 10, 50, ctypes.byref(n)) == D.EINVAL
    c.word_boundary, c.space_id = 1, -1
    assert lib.ctcpb_workspace_size(ctypes.byref(c), 2, 10, 50, ctypes.byref(n)) == D.EINVAL
    c.space_id = 7
    assert lib.ctcpb_workspace_size(ctypes.byref(c), 2, 10, 50, ctypes.byref(n)) == D.OK


def test_size_queries(lib):
    c = cfg()
    a = D.workspace_size(c, 32, 500, 5000)
    b = D.workspace_size(c, 64, 500, 5000)
    assert 0 < a < b and a % 256 == 0
    s1 = D.state_size(c, 128, 5000)
    s2 = D.state_size(cfg(max_seq_len=400), 128, 5000)
    assert s2 < s1
    p = D.state_size(cfg(beam=128, nbest=128, paged=True, max_seq_len=400), 16, 29)
    assert p > 0
    with pytest.raises(D.CtcpbError):
        D.workspace_size(c, -1, 10, 5000)
    assert D.list_len(c, 5000) == 22
    assert D.list_len(cfg(beam=128, nbest=128), 29) == 28
    assert D.list_len(cfg(list_len=3), 5000) == 10
    assert D.list_len(cfg(beam=2, nbest=2, list_len=3), 5000) == 3


def test_host_validation_before_any_launch(lib):
    c = cfg().c()
    NULL = None
    # B = 0 is a no-op
    assert lib.ctcpb_decode_offline(ctypes.byref(c), NULL, 5000, 5000, NULL, 0, 10, 5000, NULL, 0, NULL, NULL,
                                    NULL, 0, NULL) == D.OK
    # missing outputs
    assert lib.ctcpb_decode_offline(ctypes.byref(c), ctypes.c_void_p(256), 5000, 5000, NULL, 2, 10, 5000,
                                    ctypes.c_void_p(256), 1 << 30, NULL, NULL, NULL, 10, NULL) == D.ENULL
    # bad stride
    assert lib.ctcpb_decode_offline(ctypes.byref(c), ctypes.c_void_p(256), 5000, 10, NULL, 2, 10, 5000,
                                    ctypes.c_void_p(256), 1 << 30, ctypes.c_void_p(256), ctypes.c_void_p(256),
                                    ctypes.c_void_p(256), 10, NULL) == D.EINVAL
    # misaligned / too small workspace
    args = (ctypes.byref(c), ctypes.c_void_p(256), 50000, 5000, NULL, 2, 10, 5000)
    outs = (ctypes.c_void_p(512), ctypes.c_void_p(512), ctypes.c_void_p(512), 10, NULL)
    assert lib.ctcpb_decode_offline(*args, ctypes.c_void_p(260), 1 << 30, *outs) == D.EALIGN
    assert lib.ctcpb_decode_offline(*args, ctypes.c_void_p(512), 1024, *outs) == D.ESIZE
    assert lib.ctcpb_decode_offline(*args, NULL, 1 << 30, *outs) == D.ENULL
    # streaming: bad state sizes
    assert lib.ctcpb_stream_init(ctypes.byref(c), ctypes.c_void_p(512), 16, 4, 5000, NULL) == D.ESIZE
    assert lib.ctcpb_stream_step_chunk(ctypes.byref(c), ctypes.c_void_p(512), 16, 4, 5000, NULL, 5000, 5000,
                                       NULL, 16, NULL) == D.ENULL
    # speech-masked streaming: a null mask, a mask row shorter than the chunk
    big = ctypes.c_void_p(1 << 20)
    assert lib.ctcpb_stream_step_chunk_masked(ctypes.byref(c), big, 1 << 40, 4, 5000, big, 5000, 5000, NULL, NULL,
                                              16, 16, NULL) == D.ENULL
    assert lib.ctcpb_stream_step_chunk_masked(ctypes.byref(c), big, 1 << 40, 4, 5000, big, 5000, 5000, NULL, big,
                                              8, 16, NULL) == D.EINVAL
    # single-frame step: a null frame, a row stride below V, a state too small, B = 0
    assert lib.ctcpb_stream_step(ctypes.byref(c), big, 1 << 40, 4, 5000, NULL, 5000, NULL, NULL) == D.ENULL
    assert lib.ctcpb_stream_step(ctypes.byref(c), big, 1 << 40, 4, 5000, big, 4999, big, NULL) == D.EINVAL
    assert lib.ctcpb_stream_step(ctypes.byref(c), big, 16, 4, 5000, big, 5000, NULL, NULL) == D.ESIZE
    assert lib.ctcpb_stream_step(ctypes.byref(c), NULL, 0, 0, 5000, NULL, 5000, NULL, NULL) == D.OK
    # wait self-test: counts, spin bounds and pointers are checked before the launch
    assert lib.ctcpb_selftest_waits(big, -1, 10, big, NULL) == D.EINVAL
    assert lib.ctcpb_selftest_waits(big, 4, 0, big, NULL) == D.EINVAL
    assert lib.ctcpb_selftest_waits(big, 4, (1 << 20) + 1, big, NULL) == D.EINVAL
    assert lib.ctcpb_selftest_waits(NULL, 4, 10, big, NULL) == D.ENULL
    assert lib.ctcpb_selftest_waits(big, 4, 10, NULL, NULL) == D.ENULL
    assert lib.ctcpb_read_status(NULL, NULL) == D.ENULL
    assert lib.ctcpb_topk_prepass(ctypes.byref(c), NULL, 10, 5, 5000, NULL, NULL, NULL, NULL, NULL, NULL,
                                  NULL) == D.EINVAL


def test_label_boost_config_and_host_validation(lib):
    n0, n1 = ctypes.c_size_t(), ctypes.c_size_t()
    c = cfg().c()
    assert lib.ctcpb_workspace_size(ctypes.byref(c), 4, 50, 5000, ctypes.byref(n0)) == D.OK
    c.max_boost = 100  # a label-boost table of 256 slots per row
    assert lib.ctcpb_workspace_size(ctypes.byref(c), 4, 50, 5000, ctypes.byref(n1)) == D.OK
    assert n1.value >= n0.value + 4 * 256 * 8
    for bad in (-1, 4097):
        c.max_boost = bad
        assert lib.ctcpb_workspace_size(ctypes.byref(c), 4, 50, 5000, ctypes.byref(n1)) == D.EINVAL
    NULL = None
    big = ctypes.c_void_p(1 << 20)
    tables = D._Boost(1 << 20, 1 << 20, 1 << 20)
    no_tokens = D._Boost(1 << 20, None, 1 << 20)
    args = (big, 50000, 5000, NULL, 2, 10, 5000, big, 1 << 40, big, big, big, 10, NULL)
    c.max_boost = 0  # boosting not configured
    assert lib.ctcpb_decode_offline_boosted(ctypes.byref(c), ctypes.byref(tables), *args) == D.EINVAL
    assert lib.ctcpb_stream_set_boost(ctypes.byref(c), big, 1 << 40, 2, 5000, ctypes.byref(tables), NULL) == D.EINVAL
    c.max_boost = 8
    assert lib.ctcpb_decode_offline_boosted(ctypes.byref(c), ctypes.byref(no_tokens), *args) == D.ENULL
    assert lib.ctcpb_stream_set_boost(ctypes.byref(c), big, 1 << 40, 2, 5000, NULL, NULL) == D.ENULL
    assert lib.ctcpb_stream_set_boost(ctypes.byref(c), ctypes.c_void_p(512), 16, 2, 5000, ctypes.byref(tables),
                                      NULL) == D.ESIZE


def test_boost_tables_compressed_rows():
    rp, tk, bn = D.boost_tables([{3: 1.5, 7: -2.0}, None, {1: 0.25}], 3, "cpu")
    assert rp.tolist() == [0, 2, 2, 3]
    assert tk.tolist() == [3, 7, 1]
    assert bn.tolist() == [1.5, -2.0, 0.25]
    rp, tk, bn = D.boost_tables([None, None], 2, "cpu")
    assert rp.tolist() == [0, 0, 0] and tk.numel() == 1  # non-null arrays even when empty
    with pytest.raises(ValueError):
        D.boost_tables([{1: 1.0}], 2, "cpu")


def test_host_decode_sizes_and_validation(lib):
    c = cfg()
    a = D.host_workspace_size(c, 4, 200, 5000, 10)
    b = D.host_workspace_size(c, 4, 200, 5000, 200)
    assert 0 < a < b and a % 256 == 0
    NULL = None
    cc = c.c()
    big = ctypes.c_void_p(1 << 20)
    outs = (big, big, big, 10, NULL)
    # B = 0 is a no-op; a null input, a bad stride, a small workspace
    assert lib.ctcpb_decode_offline_host(ctypes.byref(cc), NULL, 5000, 5000, NULL, 0, 10, 5000, NULL, 0,
                                         *outs) == D.OK
    assert lib.ctcpb_decode_offline_host(ctypes.byref(cc), NULL, 50000, 5000, NULL, 2, 10, 5000, big, 1 << 40,
                                         *outs) == D.ENULL
    assert lib.ctcpb_decode_offline_host(ctypes.byref(cc), big, 50000, 10, NULL, 2, 10, 5000, big, 1 << 40,
                                         *outs) == D.EINVAL
    assert lib.ctcpb_decode_offline_host(ctypes.byref(cc), big, 50000, 5000, NULL, 2, 10, 5000,
                                         ctypes.c_void_p(512), 1024, *outs) == D.ESIZE
    assert lib.ctcpb_decode_offline_host(ctypes.byref(cc), big, 50000, 5000, NULL, 2, 10, 5000,
                                         ctypes.c_void_p(260), 1 << 40, *outs) == D.EALIGN


def test_lse_table_equals_the_oracle_and_mpmath(lib):
    """The library's logsumexp coefficients (computed at compile time by its
    own series) equal the oracle's (computed by its own code from libm) and the
    Taylor coefficients mpmath computes to 40 digits, bit for bit."""
    import numpy as np
    import oracle as O
    out = np.empty(576, np.float32)
    fn = lib.ctcpb_lse_table
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int]
    assert fn(out.ctypes.data, 576) == 576
    assert fn(None, 0) == 576 and fn(None, -1) < 0
    ours = out.reshape(96, 6)
    assert np.array_equal(ours.view(np.int32), O.F_coefficients().view(np.int32))
    from test_oracle_math import exact_coefficients
    assert np.array_equal(ours.view(np.int32), exact_coefficients().view(np.int32))
