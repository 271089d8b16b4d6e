"""Failure detection without a GPU fault: the decoder's bounded waits give up
and report CTCPB_DEV_TIMEOUT instead of hanging (ctcpb_selftest_waits runs
both forms of wait against conditions that never complete), and the context
stays usable: a decode right after matches the oracle."""
import time

import numpy as np
import pytest
import torch

from ctc_prefix_beam_gb300 import decoder as D
from ctc_prefix_beam_gb300 import synth
from gpu_util import assert_same, cfg_of, gpu_offline, oracle_offline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from ctc_prefix_beam_gb300 import build
    build.build()
    D.lib()
    assert torch.cuda.is_available()


def test_waits_on_flags_nothing_sets_give_up():
    flags = torch.zeros(64, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    published, flag_status, bar_status = D.selftest_waits(flags, max_spins=2000)
    assert time.perf_counter() - t0 < 5.0
    assert published == 0
    assert flag_status == D.DEV_TIMEOUT
    assert bar_status == D.DEV_TIMEOUT  # the barrier phase lacks an arrival


@pytest.mark.parametrize("nset", [1, 10, 31, 32, 33, 63])
def test_flag_wait_reports_how_far_it_got(nset):
    flags = torch.zeros(64, dtype=torch.int32, device="cuda")
    flags[:nset] = 1
    flags[nset + 1:] = 1  # set flags after the first unset one are not reached in order
    published, flag_status, _ = D.selftest_waits(flags, max_spins=500)
    assert published == nset
    assert flag_status == D.DEV_TIMEOUT


def test_flags_all_set_complete_without_timeout():
    """Each try acquires up to 32 flags: 100 set flags take exactly 4 tries."""
    flags = torch.ones(100, dtype=torch.int32, device="cuda")
    assert D.selftest_waits(flags, max_spins=3)[:2] == (96, D.DEV_TIMEOUT)
    published, flag_status, bar_status = D.selftest_waits(flags, max_spins=4)
    assert published == 100
    assert flag_status == 0
    assert bar_status == D.DEV_TIMEOUT


def test_context_usable_after_waits_gave_up():
    D.selftest_waits(torch.zeros(8, dtype=torch.int32, device="cuda"), max_spins=100)
    w = synth.workload("bpe", B=4, T=60)
    lp, lens = synth.gen_batch(w)
    cfg = cfg_of(w)
    assert_same(gpu_offline(cfg, lp, lens), oracle_offline(cfg, lp, lens), "after the self-test")
