"""Failure detection on the GPU without a fault: a bounded in-kernel wait on
an mbarrier that nothing arrives at gives up after the wait limit, reports
IMP_DEV_TIMEOUT through the device status word, and the context stays
usable (a GEMM afterwards still matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle
from _gpu import check_within_tolerance, dev_bf16, dev_nvfp4

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    st = pkg.imp_selftest_bounded_wait(status.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == pkg.IMP_OK
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert int(status.item()) == pkg.IMP_DEV_TIMEOUT
    assert 0.5 < waited < 30.0  # the 1 s limit, not a hang

    # the context still works: a small decode GEMM against the oracle
    rng = np.random.default_rng(7)
    w = rng.standard_normal((256, 1024)).astype(np.float32) * 0.02
    x = rng.standard_normal((1, 1024)).astype(np.float32)
    w_bits = (w.view(np.uint32) >> 16).astype(np.uint16)
    x_bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    c, s, ts, _ = oracle.quantize(w_bits)
    wq = dev_nvfp4(c, s, ts)
    y = torch.empty((1, 256), dtype=torch.bfloat16, device="cuda")
    status.zero_()
    pkg.gemm(dev_bf16(x_bits), wq, y=y, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, bound = oracle.reference_gemm(x_bits, 1, c, s, ts)
    check_within_tolerance(y.float().cpu().numpy(), y_ref, bound, "after timeout")


def test_selftest_rejects_bad_status_pointer():
    assert pkg.imp_selftest_bounded_wait(None, None) == pkg.IMP_ERR_INVALID_ARG
