"""Failure detection without a GPU fault: a bounded on-chip wait that runs out
is reported through the device status word, and the context stays usable."""

import pytest

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    fa = cuda_lib
    assert fa.fa_last_device_status() == fa.FA_OK
    fa.fa_selftest_wait_timeout(50)
    assert fa.fa_last_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_last_device_status() == fa.FA_OK  # reading clears the record
    # the context still runs real work correctly
    dev, _ = gu.device_inputs(77, 1, 2, 256, 64, ("q", "k", "v"))
    o, lse = gu.run_fwd(fa, dev, True, 0.125)
    assert bool(o.isfinite().all()) and bool(lse.isfinite().all())


def test_selftest_rejects_bad_limits(cuda_lib):
    with pytest.raises(cuda_lib.FaError):
        cuda_lib.fa_selftest_wait_timeout(0)
    with pytest.raises(cuda_lib.FaError):
        cuda_lib.fa_selftest_wait_timeout(5000)
