"""The bounded device waits give up and report instead of hanging: a wait on a
barrier that nothing completes returns after its limit, the next device-error
check reports a timeout (once), and the context stays usable for FFN calls."""
import time

import pytest

import oracle
import workloads
from tests.gpu_util import TIGHT_L2, TIGHT_MAX, check_close, lib, to_dev, torch

pytestmark = pytest.mark.gpu

Q4K_OK, Q4K_ERR_SHAPE, Q4K_ERR_TIMEOUT = 0, 2, 7


def test_wait_that_nothing_completes_reports_timeout():
    q = lib()
    assert q.q4k_check_device_error() == Q4K_OK  # nothing pending from earlier tests
    t0 = time.monotonic()
    q.q4k_test_bounded_wait(50_000_000)  # 50 ms
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert 0.04 < waited < 1.5, waited
    assert q.q4k_check_device_error() == Q4K_ERR_TIMEOUT
    assert q.q4k_check_device_error() == Q4K_OK  # the word was cleared


def test_limit_out_of_range_is_rejected_without_launch():
    q = lib()
    for bad in (0, 999, 3_000_000_000):
        with pytest.raises(q.Q4KError) as e:
            q.q4k_test_bounded_wait(bad)
        assert e.value.status == Q4K_ERR_SHAPE
    assert q.q4k_check_device_error() == Q4K_OK


def test_context_usable_after_a_timeout():
    q = lib()
    q.q4k_test_bounded_wait(1_000_000)  # 1 ms
    assert q.q4k_check_device_error() == Q4K_ERR_TIMEOUT
    cfg = workloads.CONFIGS[0]
    wg, wu, wd = workloads.weights(cfg)
    x, _ = workloads.activations(cfg)
    y = q.ffn_q4k_swiglu(to_dev(x), to_dev(wg), to_dev(wu), to_dev(wd))
    torch.cuda.synchronize()
    ref, _ = oracle.ffn_decode(x, wg, wu, wd)
    check_close(y.cpu().numpy(), ref, TIGHT_L2, TIGHT_MAX)
    assert q.q4k_check_device_error() == Q4K_OK

