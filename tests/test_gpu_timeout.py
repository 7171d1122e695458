"""The timeout path on the GPU, without faulting or hanging it: a test-only kernel waits, through
the pipelines' own bounded mbarrier wait, on a barrier that nothing arrives on, with a 1 ms
limit.  The wait runs out and records a timeout in the device status word, which the host
reads back (and which reading clears); no copy or tensor-core work is in flight, so the
device stays usable, and a GEMV launched right after it is correct."""
import numpy as np
import pytest

import oracle
import q8_block_quantized_act_gb300 as q8
from gpu_util import assert_within_tolerance, ensure_built, host, cuda, problem

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_device_stays_usable():
    ensure_built()
    assert q8.q8act_device_status() == q8.Q8ACT_OK          # nothing pending from earlier tests
    q8.check(q8.q8act_debug_wait_timeout(1_000_000))         # a 1 ms limit
    assert q8.q8act_device_status() == q8.Q8ACT_ERR_TIMEOUT
    assert q8.q8act_device_status() == q8.Q8ACT_OK          # reading the word cleared it
    # the device and the library still work
    m, n, k = 3, 700, 2048
    _, _, wb, xq, xd = problem(m, n, k, "outliers")
    y = host(q8.gemv_q8_0(cuda(wb), cuda(xq), cuda(xd), n))
    assert q8.q8act_device_status() == q8.Q8ACT_OK
    _, y64, S = oracle.matmul(wb, xq, xd, k)
    assert_within_tolerance(y, y64, S)


def test_wait_timeout_limit_range():
    ensure_built()
    assert q8.q8act_debug_wait_timeout(999) == q8.Q8ACT_ERR_DIMS
    assert q8.q8act_debug_wait_timeout(2_000_000_000) == q8.Q8ACT_ERR_DIMS
    assert q8.q8act_device_status() == q8.Q8ACT_OK
