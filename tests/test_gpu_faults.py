"""Failure detection without a GPU fault.

Every device wait in the library is bounded; when one runs out, the kernel
records a timeout in the device status word and unwinds (waits, bounded, for
its own copies and frees what it holds) instead of trapping. Here a test-only
flag (rf_debug_inject_fault site 1) makes the row-softmax kernel's first CTA
arm a barrier for a copy it never issues, so its waits run out: the call
must report RF_ERR_TIMEOUT through rf_device_status, and the context must stay
usable -- the next call on it computes the right answer.
"""

import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_F32, assert_close, f64

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives(cuda_device):
    x = inputs.make_rows(2, 1000, 31).cuda()
    api.inject_fault(1)
    try:
        api.softmax_rows(x)
        with pytest.raises(api.RFError) as err:
            api.device_status()
        assert err.value.status == api.RF_ERR_TIMEOUT
    finally:
        api.inject_fault(0)
    # the status word was cleared by the read; the context still works
    assert api.device_status() == 0
    y = api.softmax_rows(x)
    assert api.device_status() == 0
    assert_close(y, oracle.softmax_rows(f64(x.cpu())), TOL_F32, "y after the fault")
