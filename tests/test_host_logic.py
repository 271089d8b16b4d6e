"""Host-side logic that needs no GPU: the seeded input generators, the
streaming tick schedule, the benchmark's traffic-record lookup, and the
binding's argument checks (raised before any device call)."""
import json

import numpy as np
import pytest
import torch

import bench
from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth


@pytest.mark.parametrize("name", ["bpe", "char", "skip", "tiny"])
def test_rows_regenerate_alone(name):
    """Every row comes from its own child seed: generating a subset of rows
    gives the same bytes as those rows of the whole batch."""
    w = synth.workload(name, B=5, T=40)
    full, lens = synth.gen_batch(w, threads=2)
    part, plens = synth.gen_batch(w, threads=1, rows=range(2, 4))
    assert np.array_equal(part, full[2:4], equal_nan=True)
    assert np.array_equal(plens, lens[2:4])
    for b in range(w.B):
        np.testing.assert_array_equal(synth.gen_row(w, b)[:lens[b]], full[b, :lens[b]])


def test_rows_are_log_probabilities_with_nan_padding():
    w = synth.workload("bpe", B=4, T=60)
    lp, lens = synth.gen_batch(w)
    for b in range(w.B):
        valid = lp[b, :lens[b]].astype(np.float64)
        np.testing.assert_allclose(np.exp(valid).sum(-1), 1.0, rtol=1e-5)
        assert np.isnan(lp[b, lens[b]:]).all()
    zero, _ = synth.gen_batch(w, pad="zero")
    assert not np.isnan(zero).any()
    assert synth.checksum(lp[:, :int(lens.min())]) == synth.checksum(zero[:, :int(lens.min())])


def test_stream_ticks_cover_every_frame_once_in_order():
    """The tick schedule packs each stream's frames, in order, from its start
    offset on: concatenated over the ticks they are the stream's frames."""
    w = synth.workload("stream", B=6, T=70)
    offs = synth.stream_offsets(synth.WORKLOADS["stream"])[:w.B]
    cache = {}
    got = [[] for _ in range(w.B)]
    for k in range(synth.n_ticks(w, offs)):
        chunk, nf = synth.stream_tick(w, k, offs, cache, threads=2)
        for i in range(w.B):
            assert np.isnan(chunk[i, nf[i]:]).all()
            got[i].append(chunk[i, :nf[i]])
            lo = max(0, int(offs[i]) - 16 * k)  # the stream starts within or before this window
            assert nf[i] <= 16 - min(lo, 16)
    for i in range(w.B):
        np.testing.assert_array_equal(np.concatenate(got[i]), synth.gen_stream(w, i))


def test_traffic_record_requires_the_current_sources(tmp_path, monkeypatch):
    rec = {"k/w": {"bytes_per_launch": 123, "sources_sha": "abc"}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "sources_sha", lambda: "abc")
    assert bench.traffic_record("k", "w") == 123
    assert bench.traffic_record("k", "other") is None
    monkeypatch.setattr(bench, "sources_sha", lambda: "changed")
    assert bench.traffic_record("k", "w") is None


def test_committed_traffic_records_match_the_kernel_sources():
    recs = json.load(open(f"{bench.ROOT}/profiles/traffic.json"))
    assert {"k_fused/bpe", "k_rank_tma/bpe", "k_step_warp/bpe", "k_step/char"} <= set(recs)
    for key, r in recs.items():
        assert r["bytes_per_launch"] > 0 and r["command"].startswith("ncu "), key


def test_binding_rejects_bad_tensors_before_any_device_call():
    cfg = D.Config(beam=4, nbest=2)
    with pytest.raises(ValueError):
        D.decode_offline(cfg, torch.zeros((2, 5, 10)))  # host tensor
    with pytest.raises(ValueError):
        D.decode_offline(cfg, torch.zeros((2, 5, 10), dtype=torch.float64))
    with pytest.raises(ValueError):
        D.decode_offline(cfg, torch.zeros((5, 10)))
    with pytest.raises(ValueError):
        D.selftest_waits(torch.zeros(4, dtype=torch.int32))  # host tensor


def test_config_maps_the_word_boundary_label():
    c = D.Config(beam=8, nbest=3).c()
    assert (c.beam, c.nbest, c.word_boundary) == (8, 3, 0)
    c = D.Config(beam=8, space_id=5).c()
    assert (c.word_boundary, c.space_id, c.nbest) == (1, 5, 8)


def test_caller_buffers_are_validated():
    """The library writes through plain pointers, so the binding checks every
    caller-supplied buffer: outputs of exactly the written sizes and types,
    workspaces of enough bytes, all on the call's device."""
    cpu = torch.device("cpu")
    good = (torch.empty((2, 3, 5), dtype=torch.int32), torch.empty((2, 3), dtype=torch.int32),
            torch.empty((2, 3), dtype=torch.float32))
    assert all(a is b for a, b in zip(D._check_outputs(good, 2, 3, 5, cpu), good))
    bad = [(torch.empty((2, 3, 4), dtype=torch.int32),) + good[1:],              # too short
           (good[0], torch.empty((2, 3), dtype=torch.int64), good[2]),            # wrong type
           (good[0], good[1], torch.empty((3, 2), dtype=torch.float32).t()),      # not contiguous
           good[:2] + (torch.empty((2, 4), dtype=torch.float32),)]                 # too long
    for outs in bad:
        with pytest.raises(ValueError):
            D._check_outputs(outs, 2, 3, 5, cpu)
    ws = torch.empty(1024, dtype=torch.uint8)
    assert D._check_buf(ws, 1000, cpu, "workspace") == 1024
    assert D._check_buf(torch.empty(256, dtype=torch.float32), 1000, cpu, "workspace") == 1024
    with pytest.raises(ValueError):
        D._check_buf(ws, 2048, cpu, "workspace")
    with pytest.raises(ValueError):
        D._check_buf(ws[::2], 100, cpu, "workspace")
    with pytest.raises(ValueError):
        D._cuda_device("cpu")


def test_algorithmic_bytes_follow_the_measurement_rule():
    """Kept rows read once (4V), one 32-byte sector per skipped valid frame,
    beam x 20 bytes of state per decoded frame and row, 4 bytes per output label;
    the ranked lists of the pre-pass are not counted."""
    import bench
    w = synth.workload("skip", B=3, T=10, V=8, beam=2, nbest=2)
    lens = np.array([10, 4, 0], np.int32)
    kept = np.array([7, 4, 0])
    by = bench.algorithmic_bytes(w, lens, kept, np.array([[3, 2], [1, 0], [0, 0]]))
    assert by["rank"] == 11 * 4 * 8
    assert by["select"] == 3 * 32
    assert by["state"] == 11 * 2 * 20 + 6 * 4
    assert by["decode"] == by["rank"] + by["select"] + by["state"]


def test_row_strides_of_extent_one_dimensions():
    """An inserted batch axis has stride 0 (NumPy's x[None]); the library is
    given a valid stride for it instead, and real strides pass unchanged."""
    x = torch.from_numpy(np.zeros((3, 8), np.float32)[None])
    assert x.stride(0) == 0
    assert D._row_strides(x) == (24, 8)
    y = torch.zeros((2, 1, 8))[:, :, :]
    assert D._row_strides(y) == (8, 8)
    z = torch.zeros((4, 6, 8))
    assert D._row_strides(z) == (48, 8)
