"""CUDA decoder vs the CPU oracle, element by element, through the C ABI.

Bars: token sequences and lengths bit-exact; scores within 1e-4 absolute (the
decoder's contract) and, by construction, bit-identical (both sides evaluate
the same float32 operations in the same order).
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle as O
from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import NEG, assert_same, cfg_of, gpu_offline, oracle_offline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    O.lib()
    assert torch.cuda.is_available()


def log_softmax(x):
    x = np.asarray(x, np.float64)
    m = x.max(-1, keepdims=True)
    return (x - m - np.log(np.exp(x - m).sum(-1, keepdims=True))).astype(np.float32)


# ------------------------------------------------------------ pre-pass (a2)

def adversarial_rows(rng, R, V):
    rows = rng.normal(-8.0, 2.0, size=(R, V)).astype(np.float32)
    rows[0, :] = -3.0                              # one value everywhere (overflow fallback)
    rows[1, V // 3:] = -np.inf                     # dead tail
    rows[2, ::7] = np.nan                          # NaN labels are dead
    rows[3, 0::2] = -0.0                           # -0 and +0 tie
    rows[3, 1::2] = 0.0
    rows[4, 1:] = NEG                              # no live non-blank label
    rows[5, :] = np.round(rows[5, :])              # many ties
    rows[6, V - 1] = 5.0                           # peak at the last label
    rows[7, :] = np.float32(-1e-30)                # tiny equal values
    return rows


@pytest.mark.parametrize("V,beam,list_len", [(5000, 10, 0), (1024, 16, 0), (29, 128, 0), (32, 4, 0),
                                              (5000, 32, 0), (5000, 64, 0), (1024, 100, 0),
                                             (7, 4, 0), (5000, 2, 3), (5000, 1, 1), (300, 31, 0),
                                             (5000, 40, 0), (2, 1, 0), (3000, 128, 0)])
def test_prepass_lists_match_oracle(V, beam, list_len):
    rng = np.random.default_rng(V + beam)
    R = 200
    rows = np.concatenate([adversarial_rows(rng, 8, V), rng.normal(-8.0, 2.0, size=(R - 8, V))]).astype(np.float32)
    rows[10:60, rng.integers(0, V, 50)] += 9.0
    cfg = D.Config(beam=beam, list_len=list_len)
    L = D.list_len(cfg, V)
    g = D.topk_prepass(cfg, torch.from_numpy(rows).cuda())
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = O.frame_lists(rows, 0, L)
    for k in ("cnt", "ids", "front_id"):
        assert np.array_equal(g[k], o[k]), k
    for k in ("lps", "lpb", "front_lp"):
        assert np.array_equal(g[k].view(np.int32), o[k].view(np.int32)), k


# ------------------------------------------------------------ frame selection (a1)

@pytest.mark.parametrize("thr", [0.999, 0.98, 0.5, 1.0, 0.0])
def test_select_frames_match_oracle(thr):
    w = synth.workload("skip", B=8, T=700)
    lp, lens = synth.gen_batch(w)
    lens = np.array([700, 0, 1, 350, 699, 200, 700, 5], np.int32)
    cfg = cfg_of(w, blank_threshold=thr)
    sel, nsel = D.select_frames(cfg, torch.from_numpy(lp).cuda(), torch.from_numpy(lens).cuda())
    osel, onsel = O.select_frames(lp, lens, 0, thr)
    assert np.array_equal(nsel.cpu().numpy(), onsel)
    assert np.array_equal(sel.cpu().numpy(), osel)


# ------------------------------------------------------------ full decodes, small

SMALL = [
    ("tiny", {}, {}),
    ("bpe", dict(B=6, T=160), {}),
    ("bpe", dict(B=4, T=90), dict(paged=True)),
    ("char", dict(B=3, T=120), {}),
    ("char", dict(B=3, T=120), dict(paged=False)),
    ("skip", dict(B=6, T=300), {}),
    ("skip", dict(B=4, T=200), dict(blank_threshold=0.9)),
]


@pytest.mark.parametrize("name,shape,over", SMALL)
def test_decode_small_matches_oracle(name, shape, over):
    w = synth.workload(name, **shape)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w, **over)
    assert_same(gpu_offline(cfg, lp, lens), oracle_offline(cfg, lp, lens), f"{name}{shape}{over}")


EDGE = [
    dict(beam=1, nbest=1),
    dict(beam=2, nbest=1),
    dict(beam=8, nbest=8, V=3),            # vocabulary narrower than the beam
    dict(beam=32, nbest=5),
    dict(beam=33, nbest=33),               # first beam on the 128-thread path
    dict(beam=10, blank_id=4),
    dict(beam=10, max_seq_len=3),          # the cap binds
    dict(beam=10, max_seq_len=1),
    dict(beam=10, list_len=1),             # list of `beam` labels: frequent full-row re-ranks
    dict(beam=3, list_len=3, V=40),        # short list on a wider vocabulary
    dict(beam=4, list_len=66, V=100),      # longest list the warp-per-row kernel takes
    dict(beam=10, list_len=80, V=200),     # a longer list goes to the block kernel
    dict(beam=10, list_len=2, paged=True, page_size=3),
    dict(beam=6, paged=True, page_size=1),
    dict(beam=6, blank_threshold=0.0),     # no frame decoded
    dict(beam=6, blank_threshold=0.7),
    dict(beam=16, nbest=4, out_len=5),     # truncated output, lengths stay full
]


@pytest.mark.parametrize("case", EDGE, ids=[str(c) for c in EDGE])
def test_edge_cases_match_oracle(case):
    case = dict(case)
    V = case.pop("V", 12)
    out_len = case.pop("out_len", None)
    rng = np.random.default_rng(len(str(case)))
    B, T = 5, 60
    x = rng.normal(0.0, 2.0, size=(B, T, V))
    x[:, :, case.get("blank_id", 0)] += 2.0
    lp = log_softmax(x)
    lens = np.array([60, 0, 1, 37, 59], np.int32)
    cfg = D.Config(**case)
    assert_same(gpu_offline(cfg, lp, lens, out_len), oracle_offline(cfg, lp, lens, out_len), str(case))


@pytest.mark.parametrize("beam,V,paged,cap", [(32, 3000, False, 0), (64, 2000, False, 0), (40, 700, True, 0),
                                               (128, 1500, False, 0), (48, 1000, True, 5)])
def test_block_kernel_frame_scans_match_oracle(beam, V, paged, cap):
    """Every other frame gives all non-blank labels one log-prob, so the
    first unlisted label ties with the listed ones and with the beam-th
    candidate: the list cannot bound the unlisted labels and the step scans
    the frame, where every unlisted label passes the filter (the kept-label
    list flushes several times a frame)."""
    rng = np.random.default_rng(beam * V)
    B, T = 3, 30
    x = rng.normal(0.0, 1.0, size=(B, T, V))
    x[:, :, 0] += 1.0
    lp = log_softmax(x)
    lp[:, 1::2, 1:] = lp[:, 1::2, 1:].mean(-1, keepdims=True)
    lens = np.array([30, 17, 1], np.int32)
    cfg = D.Config(beam=beam, nbest=beam, max_seq_len=cap, paged=paged, page_size=4)
    dev = torch.device("cuda")
    ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device=dev)
    tok, ln, sc = D.decode_offline(cfg, torch.from_numpy(lp).to(dev), torch.from_numpy(lens).to(dev), workspace=ws)
    torch.cuda.synchronize()
    g = (tok.cpu().numpy(), ln.cpu().numpy(), sc.cpu().numpy())
    assert_same(g, oracle_offline(cfg, lp, lens), f"beam {beam} V {V} paged {paged} cap {cap}")
    cnt = D.read_counters(ws)
    assert cnt["steps"] == int(lens.sum())
    assert cnt["frame_scans"] > 0, cnt


@pytest.mark.parametrize("beam,V,list_len,flat", [(16, 3000, 0, "tie"), (8, 1024, 0, "tie"),
                                                   (16, 400, 66, "near"), (12, 200, 40, "near")])
def test_warp_kernel_exhaustive_paths_match_oracle(beam, V, list_len, flat):
    """The warp-per-row kernel's slow selections.  "tie": every other frame
    gives all non-blank labels one log-prob, so the first unlisted label ties
    with the listed ones and the exhaustive selection must scan the frame.
    "near": frames close to uniform with a long list, so that more candidates
    reach the beam-th kept score than the compacting selection takes and the
    general one runs."""
    rng = np.random.default_rng(beam * V + list_len)
    B, T = 4, 40
    x = rng.normal(0.0, 1.0 if flat == "tie" else 0.05, size=(B, T, V))
    x[:, :, 0] += 1.0 if flat == "tie" else 0.5
    lp = log_softmax(x)
    if flat == "tie":
        lp[:, 1::2, 1:] = lp[:, 1::2, 1:].mean(-1, keepdims=True)
    lens = np.array([40, 23, 1, 39], np.int32)
    cfg = D.Config(beam=beam, nbest=beam, list_len=list_len)
    dev = torch.device("cuda")
    ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device=dev)
    tok, ln, sc = D.decode_offline(cfg, torch.from_numpy(lp).to(dev), torch.from_numpy(lens).to(dev), workspace=ws)
    torch.cuda.synchronize()
    g = (tok.cpu().numpy(), ln.cpu().numpy(), sc.cpu().numpy())
    assert_same(g, oracle_offline(cfg, lp, lens), f"beam {beam} V {V} L {list_len} {flat}")
    cnt = D.read_counters(ws)
    assert cnt["steps"] == int(lens.sum())
    assert cnt["exhaustive"] > 0, cnt
    if flat == "tie":
        assert cnt["frame_scans"] > 0, cnt


def test_ties_and_dead_labels_match_oracle():
    rng = np.random.default_rng(77)
    B, T, V = 4, 40, 9
    lp = np.round(log_softmax(rng.normal(0, 1.0, size=(B, T, V))), 1).astype(np.float32)
    lp[1, :, 3] = -np.inf
    lp[2, 5:9, :] = NEG
    lp[2, 5:9, 0] = 0.0
    lp[3, :, :] = np.float32(-2.0)
    for paged in (False, True):
        cfg = D.Config(beam=6, paged=paged, page_size=4)
        assert_same(gpu_offline(cfg, lp, None), oracle_offline(cfg, lp, None), f"ties paged={paged}")


def test_paged_equals_flat():
    w = synth.workload("char", B=4, T=300)
    lp, lens = synth.gen_batch(w)
    a = gpu_offline(cfg_of(w, paged=False), lp, lens)
    b = gpu_offline(cfg_of(w, paged=True), lp, lens)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


# ------------------------------------------------------------ full-size workloads, every row

@pytest.mark.parametrize("name", ["tiny", "bpe", "char", "skip"])
def test_full_size_every_row(name):
    """Each offline workload at its full size, in the launch configuration the
    benchmark times, compared with the oracle on every row."""
    w = synth.WORKLOADS[name]
    lp, lens = synth.gen_batch(w, pad="nan")
    cfg = cfg_of(w)
    g = gpu_offline(cfg, lp, lens)
    o = oracle_offline(cfg, lp, lens)
    assert_same(g, o, f"{name}: all {w.B} rows")


# ------------------------------------------------------------ streaming

def stream_decode(cfg, frames, chunks, nframes_list=None):
    B, T, V = frames.shape
    st = D.StreamState(cfg, B, V)
    t0 = 0
    for i, c in enumerate(chunks):
        x = torch.from_numpy(np.ascontiguousarray(frames[:, t0:t0 + c])).cuda()
        st.step_chunk(x)
        t0 += c
    out = st.read(out_len=T)
    torch.cuda.synchronize()
    return tuple(v.cpu().numpy() for v in out), st


@pytest.mark.parametrize("paged", [False, True])
def test_streaming_chunk_invariance_and_offline_equality(paged):
    w = synth.workload("bpe", B=3, T=150)
    lp, _ = synth.gen_batch(w)
    cfg = cfg_of(w, paged=paged, max_seq_len=150)
    ref = oracle_offline(cfg, lp, None, out_len=150)
    for chunks in ([150], [16] * 9 + [6], [1] * 20 + [130], [64, 64, 22], [7, 70, 73]):
        got, st = stream_decode(cfg, lp, chunks)
        assert_same(got, ref, f"chunks {chunks[:4]}")
        assert st.status() == 0


def test_streaming_partial_chunks_and_resume():
    w = synth.workload("bpe", B=4, T=100)
    lp, _ = synth.gen_batch(w)
    cfg = cfg_of(w, max_seq_len=100)
    V = w.V
    st = D.StreamState(cfg, 4, V)
    # stream b receives its frames in chunks of 16 rows with n_frames[b] valid
    offs = [0, 5, 16, 31]
    total = [100, 95, 84, 69]
    ticks = (max(o + t for o, t in zip(offs, total)) + 15) // 16
    consumed = [0] * 4
    snap = None
    for k in range(ticks):
        chunk = np.full((4, 16, V), np.nan, np.float32)
        nf = np.zeros(4, np.int32)
        for b in range(4):
            a, e = max(16 * k, offs[b]), min(16 * k + 16, offs[b] + total[b])
            if e > a:
                chunk[b, :e - a] = lp[b, consumed[b]:consumed[b] + e - a]
                consumed[b] += e - a
                nf[b] = e - a
        st.step_chunk(torch.from_numpy(chunk).cuda(), torch.from_numpy(nf).cuda())
        if k == ticks // 2:
            snap = st.buf.clone()
    got = tuple(v.cpu().numpy() for v in st.read(out_len=100))
    trimmed = lp.copy()
    for b in range(4):
        trimmed[b, total[b]:] = np.nan
    ref = oracle_offline(cfg, trimmed, np.array(total, np.int32), out_len=100)
    assert_same(got, ref, "partial chunks")
    # read_state does not mutate the state
    again = tuple(v.cpu().numpy() for v in st.read(out_len=100))
    assert all(np.array_equal(x, y) for x, y in zip(got, again))
    # a snapshot taken mid-stream resumes to the same result
    st2 = D.StreamState(cfg, 4, V)
    st2.buf.copy_(snap)
    consumed = [0] * 4
    for k in range(ticks):
        chunk = np.full((4, 16, V), np.nan, np.float32)
        nf = np.zeros(4, np.int32)
        for b in range(4):
            a, e = max(16 * k, offs[b]), min(16 * k + 16, offs[b] + total[b])
            if e > a:
                chunk[b, :e - a] = lp[b, consumed[b]:consumed[b] + e - a]
                consumed[b] += e - a
                nf[b] = e - a
        if k > ticks // 2:
            st2.step_chunk(torch.from_numpy(chunk).cuda(), torch.from_numpy(nf).cuda())
    got2 = tuple(v.cpu().numpy() for v in st2.read(out_len=100))
    assert all(np.array_equal(x, y) for x, y in zip(got, got2))


def test_stream_workload_full():
    """The streaming workload exactly as the benchmark runs it: 128 streams x
    1,600 frames, staggered offsets, one stream_step_chunk call per 16-frame
    global tick with per-stream n_frames; every stream against the oracle's
    offline decode of its frames ("GPU CTC Prefix Beam Search Decoder",
    sections 3.4.9 and 8)."""
    w = synth.WORKLOADS["stream"]
    offs = synth.stream_offsets(w)
    full = np.empty((w.B, w.T, w.V), np.float32)
    with ThreadPoolExecutor(8) as ex:
        for i, x in enumerate(ex.map(lambda i: synth.gen_stream(w, i), range(w.B))):
            full[i] = x
    cfg = cfg_of(w)
    st = D.StreamState(cfg, w.B, w.V)
    ticks = synth.n_ticks(w, offs)
    for k in range(ticks):
        chunk, nf = tick_from_streams(full, offs, k, w.chunk)
        if k in (0, ticks // 2):  # the same bytes as the generator's own tick
            ref_chunk, ref_nf = synth.stream_tick(w, k, offs, {})
            assert np.array_equal(nf, ref_nf) and np.array_equal(chunk, ref_chunk, equal_nan=True)
        st.step_chunk(torch.from_numpy(chunk).cuda(), torch.from_numpy(nf).cuda())
    got = tuple(v.cpu().numpy() for v in st.read(out_len=w.T))
    assert st.status() == 0
    ref = oracle_offline(cfg, full, None, out_len=w.T)
    assert_same(got, ref, "stream workload, all 128 streams")


def tick_from_streams(full, offs, k, C):
    """Tick k's chunk: stream i's local frames that fall in global frames
    [C k, C k + C), packed at the chunk's first rows, NaN after them."""
    B, T, V = full.shape
    chunk = np.full((B, C, V), np.nan, np.float32)
    nf = np.zeros(B, np.int32)
    for i in range(B):
        a, e = max(C * k, int(offs[i])), min(C * k + C, int(offs[i]) + T)
        if e > a:
            chunk[i, :e - a] = full[i, a - int(offs[i]):e - int(offs[i])]
            nf[i] = e - a
    return chunk, nf


def test_state_header_mismatch_sets_status():
    cfg = D.Config(beam=4)
    st = D.StreamState(cfg, 2, 50)
    # reinterpret the same buffer as a state for V = 60: the header disagrees
    bad = D.StreamState.__new__(D.StreamState)
    bad.cfg, bad.B, bad.V, bad.buf, bad.nbytes = cfg, 2, 60, st.buf, st.nbytes
    if D.state_size(cfg, 2, 60) > st.buf.numel():
        pytest.skip("state for V=60 does not fit")
    bad.step_chunk(torch.zeros((2, 3, 60), device="cuda"))
    assert st.status() & D.DEV_HEADER


@pytest.mark.parametrize("beam,paged", [(128, False), (64, False), (128, True)])
def test_long_rows_with_mid_window_token_writes(beam, paged):
    """Long utterances on the 128-thread block kernel with label boosts, whose
    merges are proposed by prefix hashes: the token store is written in the
    middle of a ring window (before each check) as well as every 64 steps, by
    several warps at once; tokens and scores must match the oracle."""
    # the draws of the randomised sweep's case that found a race in the flat
    # token-store write: the shape and options first, then boosts and frames
    rng = np.random.default_rng(777_001)
    V = int(rng.choice([29, 100, 1024, 5000]))
    assert int(rng.choice([8, 10, 16, 20, 32, 64, 128])) == 128
    T = int(rng.integers(100, 700))
    B = int(rng.integers(1, 5))
    rng.integers(1, 16)
    rng.random(4)  # (storage, cap, threshold and word-boundary draws: none applied)
    assert (V, T, B) == (100, 507, 2) and rng.random() < 0.3
    nb = min(int(rng.integers(1, 40)), V - 1)
    boost = [{int(c): float(np.float32(rng.uniform(-3, 5))) for c in rng.choice(np.arange(1, V), nb, replace=False)}
             for _ in range(B)]
    x = rng.normal(0, float(rng.choice([1.0, 2.0])), size=(B, T, V))
    x[:, :, 0] += np.where(rng.random((B, T)) < 0.7, 6.0, 0.0)
    lp = x - x.max(-1, keepdims=True)
    lp = (lp - np.log(np.exp(lp).sum(-1, keepdims=True))).astype(np.float32)
    lens = rng.integers(T // 2, T + 1, size=B).astype(np.int32)
    cfg = D.Config(beam=beam, nbest=3, max_boost=nb, paged=paged)
    dev = torch.device("cuda")
    ws = torch.empty(D.workspace_size(cfg, B, T, V), dtype=torch.uint8, device=dev)
    tok, ln, sc = D.decode_offline(cfg, torch.from_numpy(lp).to(dev), torch.from_numpy(lens).to(dev),
                                   workspace=ws, boost=boost)
    torch.cuda.synchronize()
    assert D.read_counters(ws)["hash_merges"] > 0
    assert_same((tok.cpu().numpy(), ln.cpu().numpy(), sc.cpu().numpy()),
                oracle_offline(cfg, lp, lens, boost=boost), f"beam {beam} paged {paged}")
