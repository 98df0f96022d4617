"""The allocation-free quantizer entry point, through the C ABI.

Some callers cannot allocate device memory when they quantize (an engine that
forbids allocation after start-up, code inside a stream capture, a process
living in one fixed memory pool).  imp_nvfp4_quantize_noalloc serves them
with its scratch in a fixed array inside the library.  Its results must equal
imp_nvfp4_quantize's byte for byte -- the quantizer is bit-exact -- on two
calls in a row with different inputs, so nothing left in the shared array by
one call leaks into the next.

This file sorts last so that a run stopping at its first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import synth

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _quantize_both(bits):
    x = _bf16(bits)
    rows, K = bits.shape
    ref = pkg.quantize(x)  # existing entry point, caller workspace
    out = pkg.NVFP4Tensor.empty(rows, K)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = pkg.imp_nvfp4_quantize_noalloc(x.data_ptr(), rows, K, x.stride(0), out.c_struct(),
                                        status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == pkg.IMP_OK, pkg.imp_status_string(st)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ref, out


def test_noalloc_quantizer_matches_workspace_quantizer_on_two_calls():
    # first call: a large tensor (many partial maxima, global amax in a late row)
    a = synth.workload("decode_27b")[0].weight_bf16(0, 8192)
    # second call: a small tensor with a much smaller amax than the first
    b = synth.workload("single_1k")[0].weight_bf16(0, 96)
    for bits in (a, b):
        ref, out = _quantize_both(bits)
        assert torch.equal(ref.codes, out.codes)
        assert torch.equal(ref.scales, out.scales)
        assert torch.equal(ref.tensor_scale, out.tensor_scale)
