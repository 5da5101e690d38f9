"""Failure detection on the GPU without a fault: a bounded wait that runs
out is reported through the device error word, and the context stays
usable afterwards."""
import pytest

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import check_close, f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda):
    assert bi.bi_check_device_errors() == bi.OK
    assert bi.bi_selftest_wait_timeout(0) == bi.ERR_INVALID_ARG
    assert bi.bi_selftest_wait_timeout(20000) == bi.OK       # launch
    assert bi.bi_check_device_errors() == bi.ERR_TIMEOUT     # recorded by the kernel
    assert bi.bi_check_device_errors() == bi.OK              # cleared by the read
    # the context is intact: a kernel runs and is right afterwards
    x = synth.normal_bf16((4, 4096), 7700)
    w = synth.normal_bf16((4096,), 7701, std=0.1, mean=1.0)
    y = bi.rmsnorm(x.to(cuda), w.to(cuda), 1e-6)
    r = oracle.rmsnorm(x, w, 1e-6)
    check_close(f64(y), r, 1e-2 * abs(r) + 1e-30, "rmsnorm after a timeout")
    assert bi.bi_check_device_errors() == bi.OK
