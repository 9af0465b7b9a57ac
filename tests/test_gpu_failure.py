"""Failure detection without a GPU fault.

Every wait in the staging pipelines is bounded; when a bound runs out the
kernel records ADALN_DEV_TIMEOUT in the device status word and returns.  Here
a wait is made to run out on purpose (an mbarrier that nothing completes, a
2 ms bound), and the status is read back on the host; the device must stay
usable afterwards.  Data errors are injected from the host as bad segment ids
(tests/test_gpu_parity.py).
"""
import pytest

import gpu_helpers as H
from adaln_video_dit_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(adaln):
    rc, bits = adaln.adaln_get_status()
    assert rc == adaln.ADALN_OK, (rc, bits)
    adaln.adaln_selftest_wait_timeout(2000)
    rc, bits = adaln.adaln_get_status()
    assert rc == adaln.ADALN_ERR_TIMEOUT and bits & adaln.ADALN_DEV_TIMEOUT, (rc, bits)
    # read-and-clear: the word is clean again
    rc, bits = adaln.adaln_get_status()
    assert rc == adaln.ADALN_OK and bits == 0
    # the context is still usable: a normal call passes parity
    c = I.random_case(11, 600, 1024, 3, dtype="bf16")
    d = H.device_inputs(c)
    out = H.run_gpu(d, c["eps"])
    H.check_against_oracle(c, d, out)
    H.status_ok()
