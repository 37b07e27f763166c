"""The error path of the time-bounded waits, on the GPU and without a fault:
gqa_wait_timeout_selftest makes one warp wait, through the library's own
bounded waits, on a condition that nothing satisfies.  Each wait must give
up after about a second, leave GQA_DEVERR_TIMEOUT (and nothing else) in the
error word, and leave the context usable: a decode call right after it
matches the oracle with no flag."""
import time

import pytest
import torch

import grouped_query_decode_kv_b300 as gqa
import workloads

from test_gpu_parity import check_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    gqa.load_library()
    gqa.gqa_get_device_error()
    yield


@pytest.mark.parametrize("which", [0, 1, 2], ids=["mbarrier_wait", "warp_wait", "step_signal_wait"])
def test_a_wait_that_nothing_completes_times_out_and_the_context_stays_usable(which):
    assert gqa.gqa_get_device_error() == 0
    t0 = time.perf_counter()
    gqa.gqa_wait_timeout_selftest(which)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert gqa.gqa_get_device_error() == gqa.DEVERR_TIMEOUT
    assert gqa.gqa_get_device_error() == 0  # the read cleared it
    assert 0.9 <= elapsed < 20.0, elapsed
    # 16 query heads on 2 KV heads: the tcgen05 kernel, split over CTAs
    w = workloads.Workload(f"after_timeout_{which}", 2, 16, 2, 128, 300, "bf16", ("fixed", 300), 10400 + which)
    check_case(w)
