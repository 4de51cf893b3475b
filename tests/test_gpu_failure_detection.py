"""Failure detection without a GPU fault: a device wait that nothing completes gives up after its
limit, the kernel records OSF_ERR_TIMEOUT in the status word and exits, and the context keeps
working (the next library call is correct)."""
import time

import numpy as np
import pytest

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_expired_wait_is_reported_and_the_context_survives(osf):
    assert osf.osf_device_status() == osf.OSF_OK        # clean start (reads and clears)
    t0 = time.perf_counter()
    assert osf.osf_selftest_bounded_wait(2_000_000) == osf.OSF_OK   # 2 ms limit
    assert osf.osf_device_status() == osf.OSF_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 1.0                # gave up on its own, no hang
    assert osf.osf_device_status() == osf.OSF_OK         # the word was cleared by the read
    # the context still runs the hot path correctly
    x = si.softmax_rows_input(8, 1000, seed=1)
    z = osf.osf_softmax_rows(torch.from_numpy(x).cuda())
    assert np.abs(z.cpu().numpy() - oracle.softmax(x)).max() <= 1e-4
    assert osf.osf_device_status() == osf.OSF_OK


def test_selftest_rejects_out_of_range_limits(osf):
    assert osf.osf_selftest_bounded_wait(0) == osf.OSF_ERR_INVALID
    assert osf.osf_selftest_bounded_wait(3_000_000_000) == osf.OSF_ERR_INVALID
