"""The kernels' bounded waits: a wait that nothing completes gives up after its limit,
records GVA_DEV_TIMEOUT in the device status word and lets its kernel return, so the
context stays usable (a decode right after it still matches the oracle).  The failure is
made by a barrier nobody arrives on: no fault, trap or endless loop."""
import time

import pytest

from gva_inputs import make_case, workload
from helpers import Dev, assert_close, gva, oracle_decode

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    g = gva()
    assert g.gva_get_device_status() == 0
    t0 = time.time()
    g.gva_selftest_bounded_wait(2000)              # 2 ms limit
    assert g.gva_get_device_status() == g.GVA_DEV_TIMEOUT
    assert time.time() - t0 < 5.0
    assert g.gva_get_device_status() == 0          # reading cleared it
    c = make_case(workload("350m", T=300, B=2))
    out, lse = Dev(c).decode()
    ref, ref_lse = oracle_decode(c)
    assert g.gva_get_device_status() == 0
    assert_close(out, ref, "bf16", "decode after an expired wait, out")
    assert_close(lse, ref_lse, "bf16", "decode after an expired wait, lse")
