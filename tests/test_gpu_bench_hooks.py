"""The benchmark hooks bench.py reports from: the int8 mma.sync rate kernel and the tcgen05
issue-rate kernel run, stay within their bounded waits, and return figures the hardware can
deliver."""
import pytest

from tests.gpu_util import lib, torch

pytestmark = pytest.mark.gpu


def test_int8_rate_hook():
    q = lib()
    ops = q.q4k_bench_int8_mma(16)
    torch.cuda.synchronize()
    assert ops > 0
    assert q.q4k_check_device_error() == 0


def test_tcgen05_issue_hook():
    """Cycles per MMA of one issuing thread: at least what the tensor pipe needs for the
    issuers' MMAs together (128 x n x 16 multiply-adds each at 4096 per cycle: n / 2 cycles
    per MMA and issuer), and far below a stalled pipe."""
    q = lib()
    for n, k in ((128, 1), (256, 1), (128, 2), (64, 4)):
        c = q.q4k_bench_tcgen05_issue(n, k, 64)
        assert 0.9 * k * n / 2 <= c < 5000, (n, k, c)
    assert q.q4k_check_device_error() == 0
    with pytest.raises(q.Q4KError):
        q.q4k_bench_tcgen05_issue(256, 2, 64)  # 512 accumulator columns: refused
