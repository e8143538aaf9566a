"""Failure detection on the GPU without a fault: a wait whose completion
never comes gives up after its limit, reports PKV_DEVERR_TIMEOUT through the
error word, and the context stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_18_gb300 as pkv
from paged_kv_cache_18_gb300 import binding
from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import DeviceBatch, assert_close, host_f64, oracle_after_append

pytestmark = pytest.mark.gpu
PKV_DEVERR_TIMEOUT = 4


@pytest.mark.parametrize("limit_us", [1000, 50000])
def test_a_wait_nothing_completes_gives_up_and_reports(limit_us):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    binding.check_bounded_wait(err, limit_us, waited)
    code = binding.read_error_word(err)
    elapsed = time.perf_counter() - t0
    assert code == PKV_DEVERR_TIMEOUT
    w = int(waited.item())
    assert limit_us * 1000 <= w < limit_us * 1000 + 50_000_000
    assert elapsed < 5.0


def test_the_first_error_is_kept():
    err = torch.full((1,), 2, dtype=torch.int32, device="cuda")   # an earlier bad block id
    binding.check_bounded_wait(err, 100)
    assert binding.read_error_word(err) == 2


def test_the_context_stays_usable_after_a_timeout():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.check_bounded_wait(err, 2000)
    assert binding.read_error_word(err) == PKV_DEVERR_TIMEOUT
    wl = W.Workload("after a timeout", 3, 8, 2, 128, "bf16", context_lens=[17, 100, 300],
                    seed=77)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    got = host_f64(d.attend(), "bf16")
    assert binding.read_error_word(d.err) == 0
    assert_close(got, oracle_after_append(b), "bf16", "decode after a timeout")
