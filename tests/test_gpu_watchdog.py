"""Bounded waits: a wait that nothing completes runs out, the kernel reports
JETFP8_ERR_TIMEOUT through the device error word and exits, and the context
stays usable.  No fault, trap or hang is involved."""
import pytest
import torch

import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import jetfp8 as J
from e4m3_group_quantise_gb300 import synthetic as syn
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_selftest_times_out_and_recovers():
    assert jf.jetfp8_poll_device_error() == J.OK
    assert jf.jetfp8_watchdog_selftest(2000) == J.OK           # ~2 ms bounded wait
    assert jf.jetfp8_poll_device_error() == J.ERR_TIMEOUT
    assert jf.jetfp8_poll_device_error() == J.OK               # the word was cleared
    # the context still works: a real call succeeds afterwards
    x = syn.activation(128, 256, seed=0, device="cuda")
    q, s = jf.quantize_act(x)
    torch.cuda.synchronize()
    assert jf.jetfp8_poll_device_error() == J.OK
    assert q.shape == (128, 256)


def test_selftest_rejects_bad_timeout():
    assert jf.jetfp8_watchdog_selftest(0) == J.ERR_SHAPE
    assert jf.jetfp8_watchdog_selftest(10**7) == J.ERR_SHAPE
