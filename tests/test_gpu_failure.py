"""The failure path of the bounded pipeline waits, on the GPU, without a fault.

moe_selftest_wait_timeout runs one CTA with the roles of a pipeline (a landed
bulk copy, tensor memory held, a wait on an mbarrier that nothing arrives at).
The wait must give up after the library's limit (about 2 s), report
MOE_STATUS_WAIT_TIMEOUT and its site in the status word, drain its copy and
free tensor memory; the context must stay usable for the next layer call.
"""

import time

import pytest
import torch

from tests.test_gpu_layer import check_layer

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_and_leaves_the_context_usable(moe):
    moe.moe_get_status()
    moe.moe_get_timeout_site()  # start from a clear status word
    src = torch.arange(1024, dtype=torch.int32, device="cuda").to(torch.uint8)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert moe.moe_selftest_wait_timeout(src) == moe.MOE_OK
    rc, st = moe.moe_get_status()
    elapsed = time.perf_counter() - t0
    assert rc == moe.MOE_OK
    assert st & moe.MOE_STATUS_WAIT_TIMEOUT
    assert not st & moe.MOE_STATUS_BAD_EXPERT_ID
    rc, site = moe.moe_get_timeout_site()
    assert rc == moe.MOE_OK and site == (15 << 24) | (2 << 20), hex(site)
    assert 1.5 <= elapsed <= 60.0, elapsed  # the 2 s limit, not an early exit
    assert moe.moe_get_status() == (moe.MOE_OK, 0)  # read and cleared

    # the context still runs a layer correctly (routing bit-exact where clear, 1e-4 of float64)
    check_layer(moe, 0, 3, moe.MOE_RAIL_GEMV, seed=7)
    assert moe.moe_get_status() == (moe.MOE_OK, 0)


def test_selftest_rejects_a_bad_source(moe):
    assert moe.moe_selftest_wait_timeout(None) == moe.MOE_EINVAL
    src = torch.zeros(2048, dtype=torch.uint8, device="cuda")
    assert moe.moe_selftest_wait_timeout(src[1:]) == moe.MOE_EINVAL  # not 16-byte aligned
