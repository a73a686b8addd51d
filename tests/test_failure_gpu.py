"""Failure detection without a GPU fault: a kernel whose bounded mbarrier wait
is never satisfied gives up after its budget, records a timeout in the
device error word and returns; the context stays usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    assert va.varlen_attn_get_device_status() == 0
    t0 = time.time()
    assert va.varlen_attn_selftest_wait_timeout(50_000_000) == 0  # 50 ms budget
    st = va.varlen_attn_get_device_status()
    assert st == va.VARLEN_ERR_TIMEOUT
    assert time.time() - t0 < 10
    # the error word is cleared by the read, and the context still works
    assert va.varlen_attn_get_device_status() == 0
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0
