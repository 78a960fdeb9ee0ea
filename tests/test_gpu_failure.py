"""Failure detection on the GPU without a fault.  Every wait inside the
attention kernels is bounded: the merger's poll of its partials' flags and the
mbarrier waits of the TMA rings.  Here each wait is made to run out on a flag
or barrier that nothing sets, with a short poll limit; the kernel must return,
PKV_DEVERR_TIMEOUT must be read back, and the context must stay usable (a
decode right after matches the oracle)."""
import pytest
import torch

import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl
from harness import assert_bf16_close, make_decode_case, oracle_out, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_errors():
    pkv.read_device_errors(clear=True)
    yield
    pkv.read_device_errors(clear=True)


def test_flag_wait_runs_out_on_flags_nothing_sets():
    flags = torch.zeros(5, dtype=torch.int64, device="cuda")
    pkv.bounded_wait_check(flags, tag=7, arrive=True, polls=2000)
    assert pkv.read_device_errors() == pkv.DEVERR_TIMEOUT


def test_flag_wait_runs_out_when_one_flag_is_missing():
    flags = torch.full((40,), 7, dtype=torch.int64, device="cuda")
    flags[33] = 6  # one piece (beyond the first 32 lanes) never announced
    pkv.bounded_wait_check(flags, tag=7, arrive=True, polls=2000)
    assert pkv.read_device_errors() == pkv.DEVERR_TIMEOUT


def test_flag_wait_passes_when_every_flag_is_set():
    flags = torch.full((40,), 7, dtype=torch.int64, device="cuda")
    pkv.bounded_wait_check(flags, tag=7, arrive=True, polls=2000)
    assert pkv.read_device_errors() == 0


def test_mbarrier_wait_runs_out_without_an_arrival():
    pkv.bounded_wait_check(None, tag=0, arrive=False, polls=2000)
    assert pkv.read_device_errors() == pkv.DEVERR_TIMEOUT


def test_mbarrier_wait_passes_with_the_arrival():
    pkv.bounded_wait_check(None, tag=0, arrive=True, polls=2000)
    assert pkv.read_device_errors() == 0


def test_bad_arguments_are_refused_on_the_host():
    with pytest.raises(pkv.PkvError):
        pkv.bounded_wait_check(None, tag=0, arrive=True, polls=0)


def test_context_usable_after_a_timeout():
    flags = torch.zeros(3, dtype=torch.int64, device="cuda")
    pkv.bounded_wait_check(flags, tag=1, arrive=False, polls=500)
    assert pkv.read_device_errors() == pkv.DEVERR_TIMEOUT
    shape = wl.DecodeShape("after_timeout", 0, 32, 8, 128, 16, torch.bfloat16)
    lens = [1, 17, 300, 1000]
    case = make_decode_case(shape, lens, seed=3)
    out = run_decode(case, shape)  # balanced kernel, cooperative launch
    assert_bf16_close(out, oracle_out(case, shape), "decode after a timeout")
    assert pkv.read_device_errors() == 0
