"""The C ABI without a GPU: the library loads, exports every function that
include/imp_nvfp4.h declares, and rejects bad arguments before touching the
device."""
import ctypes

import pytest

import nvfp4_weight_quantized_02_gb300 as pkg
from nvfp4_weight_quantized_02_gb300 import ImpNvfp4Tensor


@pytest.fixture(scope="module")
def lib():
    return pkg.load()


def test_exports_every_declared_function(lib):
    names = pkg.header_functions()
    assert {"imp_nvfp4_quantize", "imp_nvfp4_gemm", "imp_nvfp4_quantize_workspace_size",
            "imp_nvfp4_gemm_workspace_size", "imp_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert hasattr(pkg, n), n  # the binding uses the same names


def test_status_strings():
    assert pkg.imp_status_string(0) == "IMP_OK"
    assert pkg.imp_status_string(pkg.IMP_ERR_MISALIGNED) == "IMP_ERR_MISALIGNED"
    assert pkg.imp_status_string(99) == "IMP_ERR_UNKNOWN"


def test_workspace_sizes():
    assert pkg.imp_nvfp4_quantize_workspace_size(0, 64) == 0
    assert 0 < pkg.imp_nvfp4_quantize_workspace_size(151936, 5120) <= 4096
    # decode shapes on the FP4 tensor-core path need room for X's components
    ws1 = pkg.imp_nvfp4_gemm_workspace_size(1, 17408, 5120)
    assert 16 * 2560 + 80 * 512 <= ws1 <= 16 * 2560 + 80 * 512 + (2 << 20)
    # one pass over W for every M: X's components (8 operand rows per row of
    # X, rounded up to 16/32/64/128) and the partial sums grow with M
    ws = [pkg.imp_nvfp4_gemm_workspace_size(m, 17408, 5120) for m in (1, 2, 3, 4, 5, 8, 9, 16)]
    assert ws[0] == ws[1] == ws1 < ws[2] == ws[3] < ws[4] == ws[5] < ws[6] == ws[7]
    assert ws[7] >= 128 * 2560 + 80 * 512
    # shapes that path does not take need none
    assert pkg.imp_nvfp4_gemm_workspace_size(1, 100, 5120) == 0
    assert pkg.imp_nvfp4_gemm_workspace_size(1, 17408, 320) == 0
    assert pkg.imp_nvfp4_gemm_workspace_size(1, 17408, 768) == 0


def test_gemm_plan():
    # decode, one or two rows of X on an FP4-eligible shape (K % 256 == 0,
    # K >= 1024, N >= 128) -> FP4 tensor cores: a split kernel writing X's
    # components once, then the GEMV holding its chunks of them -- or, with
    # at most six K chunks per CTA, the GEMV alone, splitting them itself;
    # more rows -> the FP4 path with X's components streamed with W
    assert pkg.imp_nvfp4_gemm_plan(1, 151936, 5120) == (2, "gemv_f4r_kernel")
    assert pkg.imp_nvfp4_gemm_plan(1, 17408, 5120) == (2, "gemv_f4r_kernel")
    assert pkg.imp_nvfp4_gemm_plan(1, 5120, 17408) == (2, "gemv_f4r_kernel")
    assert pkg.imp_nvfp4_gemm_plan(2, 5120, 17408) == (2, "gemv_f4r_kernel")
    assert pkg.imp_nvfp4_gemm_plan(4, 17408, 5120) == (2, "gemv_f4_kernel")
    assert pkg.imp_nvfp4_gemm_plan(1, 1024, 1024) == (1, "gemv_f4r_kernel")
    assert pkg.imp_nvfp4_gemm_plan(2, 3072, 1024) == (1, "gemv_f4r_kernel")
    # several rows of X: FP4, split kernel + GEMV
    assert pkg.imp_nvfp4_gemm_plan(16, 17408, 5120) == (2, "gemv_f4_kernel")
    assert pkg.imp_nvfp4_gemm_plan(3, 5120, 17408) == (2, "gemv_f4_kernel")
    # FP4 shape rules not met (K % 256): f16 passes
    assert pkg.imp_nvfp4_gemm_plan(16, 5120, 17344) == (8, "gemv_tc_kernel")
    assert pkg.imp_nvfp4_gemm_plan(2048, 17408, 5120) == (4, "gemm_mxf4_kernel")
    for bad in [(0, 128, 1024), (1, 0, 1024), (1, 128, 100), (1, 128, 0)]:
        assert pkg.imp_nvfp4_gemm_plan(*bad) == (0, None)


def test_grouped_plan():
    # one weight stream for all groups at M <= 2 (plus the split kernel when
    # a CTA holds more than six K chunks) (a 0.6B-class
    # layer's q/k/v and gate/up, a 27B-class layer's gate/up)
    gp = pkg.imp_nvfp4_gemm_grouped_plan
    assert gp(1, 1024, [2048, 1024, 1024]) == (1, "gemv_f4r_kernel")
    assert gp(1, 1024, [3072, 3072]) == (1, "gemv_f4r_kernel")
    assert gp(2, 5120, [17408, 17408]) == (2, "gemv_f4r_kernel")
    assert gp(1, 1024, [100, 28, 1]) == (1, "gemv_f4r_kernel")  # ragged groups
    # otherwise one imp_nvfp4_gemm_mma call per group
    assert gp(4, 5120, [17408, 17408]) == (4, "gemv_f4_kernel")
    assert gp(2048, 5120, [17408, 17408]) == (6, "gemm_mxf4_kernel")
    for bad in [(1, 1024, []), (1, 1024, [128] * 5), (1, 1000, [128]), (1, 1024, [0])]:
        assert gp(*bad) == (0, None)
    assert pkg.imp_nvfp4_gemm_grouped_workspace_size(1, 1024, [2048, 1024, 1024]) >= \
        pkg.imp_nvfp4_gemm_workspace_size(1, 2048, 1024)


A16 = 0x7F0000000000  # fake, 16-byte aligned "device" addresses: never dereferenced


def _chain(spec):
    """ChainLinks from [(K, [N...], chained?)] with fake aligned addresses
    (outputs 16 MB apart, explicit X beyond them)."""
    links, k = [], 0
    for c, (K, Ns, chained) in enumerate(spec):
        gs = []
        for N in Ns:
            gs.append(pkg.ImpNvfp4Group(_t(N, K), A16 + (1 + k) * (1 << 24), (N + 7) // 8 * 8))
            k += 1
        links.append((gs, None if chained else A16 + (100 + c) * (1 << 24), K))
    return pkg.ChainLinks(links)


def test_chain_plan():
    # the 27B-class decode step as one persistent launch: up, gate (x), down
    # (gate's output), LM head (down's output); a 0.6B-class layer
    step = [(5120, [17408], False), (5120, [17408], False), (17408, [5120], True),
            (5120, [151936], True)]
    assert pkg.imp_nvfp4_gemm_chain_plan(1, _chain(step)) == 1
    assert pkg.imp_nvfp4_gemm_chain_plan(2, _chain(step)) == 1
    small = [(1024, [2048, 1024, 1024], False), (2048, [1024], True), (1024, [3072, 3072], False),
             (3072, [1024], False)]
    assert pkg.imp_nvfp4_gemm_chain_plan(1, _chain(small)) == 1
    # grouped calls one after another: more rows of X, a K below 1024, a
    # CTA needing more than 24 K chunks (17408 x 17408: ~60 per CTA)
    assert pkg.imp_nvfp4_gemm_chain_plan(4, _chain(step)) == 0
    assert pkg.imp_nvfp4_gemm_chain_plan(1, _chain([(512, [1024], False)])) == 0
    assert pkg.imp_nvfp4_gemm_chain_plan(1, _chain([(17408, [17408], False)])) == 0
    ws = pkg.imp_nvfp4_gemm_chain_workspace_size(1, _chain(step))
    assert ws >= pkg.imp_nvfp4_gemm_workspace_size(1, 151936, 5120)
    # invalid: chained link 0, chained K != the previous output's length, 5 links
    assert pkg.imp_nvfp4_gemm_chain_plan(1, _chain([(1024, [128], True)])) == 0
    assert pkg.imp_nvfp4_gemm_chain_workspace_size(1, _chain([(1024, [512], False),
                                                              (1024, [128], True)])) == 0
    assert pkg.imp_nvfp4_gemm_chain_workspace_size(1, _chain([(1024, [1024], False)] * 5)) == 0


def test_chain_rejects_overlaps():
    g = pkg.imp_nvfp4_gemm_chain
    ok = _chain([(1024, [1024], False), (1024, [512], True)])
    assert g(1, ok, None, None, 0, None) == pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    # two links writing the same output
    y = A16 + (1 << 30)
    dup = pkg.ChainLinks([([pkg.ImpNvfp4Group(_t(1024, 1024), y, 1024)], A16, 1024),
                          ([pkg.ImpNvfp4Group(_t(512, 1024), y + 512, 512)], None, 0)])
    assert g(1, dup, None, A16, 1 << 30, None) == pkg.IMP_ERR_INVALID_ARG
    # an output over an explicit X
    over = pkg.ChainLinks([([pkg.ImpNvfp4Group(_t(1024, 1024), y, 1024)], y + 1024, 1024)])
    assert g(1, over, None, A16, 1 << 30, None) == pkg.IMP_ERR_INVALID_ARG
    # M = 0: nothing to do
    assert g(0, ok, None, None, 0, None) == pkg.IMP_OK


def _t(rows, K, codes=A16, scales=A16 + 0x100000, ts=A16 + 0x200000):
    return ImpNvfp4Tensor(codes, scales, ts, rows, K)


def test_gemm_rejects_bad_arguments():
    g = pkg.imp_nvfp4_gemm
    assert g(A16, -1, 64, 64, _t(8, 64), A16, 8, None, None, 0, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 96, 96, _t(8, 96), A16, 8, None, None, 0, None) == pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert g(A16, 1, 0, 64, _t(8, 0), A16, 8, None, None, 0, None) == pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert g(A16, 1, 64, 64, _t(8, 128), A16, 8, None, None, 0, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 64, 64, _t(8, 64, codes=0), A16, 8, None, None, 0, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 64, 64, _t(8, 64, codes=A16 + 8), A16, 8, None, None, 0, None) == pkg.IMP_ERR_MISALIGNED
    assert g(A16, 1, 64, 64, _t(8, 64, ts=A16 + 2), A16, 8, None, None, 0, None) == pkg.IMP_ERR_MISALIGNED
    assert g(None, 1, 64, 64, _t(8, 64), A16, 8, None, None, 0, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 64, 64, _t(8, 64), None, 8, None, None, 0, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 64, 32, _t(8, 64), A16, 8, None, None, 0, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 64, 64, _t(8, 64), A16, 4, None, None, 0, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16 + 2, 1, 64, 64, _t(8, 64), A16, 8, None, None, 0, None) == pkg.IMP_ERR_MISALIGNED
    assert g(A16, 2, 64, 68, _t(8, 64), A16, 8, None, None, 0, None) == pkg.IMP_ERR_MISALIGNED
    assert g(A16, 2, 64, 64, _t(8, 64), A16, 12, None, None, 0, None) == pkg.IMP_ERR_MISALIGNED
    # the decode path's workspace: missing, short or misaligned
    need = pkg.imp_nvfp4_gemm_workspace_size(1, 256, 1024)
    assert g(A16, 1, 1024, 1024, _t(256, 1024), A16, 256, None, None, 0, None) == \
        pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    assert g(A16, 1, 1024, 1024, _t(256, 1024), A16, 256, None, A16, need - 1, None) == \
        pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    assert g(A16, 1, 1024, 1024, _t(256, 1024), A16, 256, None, A16 + 8, need, None) == \
        pkg.IMP_ERR_MISALIGNED
    # a long K that no decode kernel takes (X beyond the register-resident
    # plans, K % 256 != 0 or N < 128 for the FP4 path): rejected, nothing enqueued
    assert pkg.imp_nvfp4_gemm_plan(2, 100, 65472) == (0, None)
    assert g(A16, 2, 65472, 65472, _t(100, 65472), A16, 104, None, None, 0, None) == \
        pkg.IMP_ERR_UNSUPPORTED_SHAPE
    # empty problems are valid and enqueue nothing
    assert g(A16, 0, 64, 64, _t(8, 64), A16, 8, None, None, 0, None) == pkg.IMP_OK
    assert g(A16, 4, 64, 64, _t(0, 64), A16, 8, None, None, 0, None) == pkg.IMP_OK


def test_quantize_rejects_bad_arguments():
    q = pkg.imp_nvfp4_quantize
    assert q(A16, -1, 64, 64, _t(-1, 64), None, A16, 4096, None) == pkg.IMP_ERR_INVALID_ARG
    assert q(A16, 4, 40, 40, _t(4, 40), None, A16, 4096, None) == pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert q(A16, 4, 64, 32, _t(4, 64), None, A16, 4096, None) == pkg.IMP_ERR_INVALID_ARG
    assert q(A16, 4, 64, 64, _t(5, 64), None, A16, 4096, None) == pkg.IMP_ERR_INVALID_ARG
    assert q(A16 + 4, 4, 64, 64, _t(4, 64), None, A16, 4096, None) == pkg.IMP_ERR_MISALIGNED
    assert q(A16, 4, 64, 68, _t(4, 64), None, A16, 4096, None) == pkg.IMP_ERR_MISALIGNED
    assert q(A16, 4, 64, 64, _t(4, 64), None, None, 0, None) == pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    assert q(A16, 4, 64, 64, _t(4, 64), None, A16, 2, None) == pkg.IMP_ERR_WORKSPACE_TOO_SMALL


def test_grouped_rejects_bad_arguments():
    g = pkg.imp_nvfp4_gemm_grouped
    G = pkg.ImpNvfp4Group
    ok = [G(_t(2048, 1024), A16, 2048), G(_t(1024, 1024), A16, 1024)]
    ws = pkg.imp_nvfp4_gemm_grouped_workspace_size(1, 1024, [2048, 1024])
    assert g(A16, 1, 1024, 1024, [], None, A16, ws, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 1024, 1024, ok * 3, None, A16, ws, None) == pkg.IMP_ERR_INVALID_ARG
    assert g(A16, 1, 1000, 1000, ok, None, A16, ws, None) == pkg.IMP_ERR_UNSUPPORTED_SHAPE
    bad_k = [G(_t(2048, 1024), A16, 2048), G(_t(1024, 2048), A16, 1024)]
    assert g(A16, 1, 1024, 1024, bad_k, None, A16, ws, None) == pkg.IMP_ERR_INVALID_ARG
    short_ldy = [G(_t(2048, 1024), A16, 1024)]
    assert g(A16, 1, 1024, 1024, short_ldy, None, A16, ws, None) == pkg.IMP_ERR_INVALID_ARG
    odd_y = [G(_t(2048, 1024), A16 + 8, 2048)]
    assert g(A16, 1, 1024, 1024, odd_y, None, A16, ws, None) == pkg.IMP_ERR_MISALIGNED
    assert g(A16, 1, 1024, 1024, ok, None, A16, ws - 16, None) == pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    assert g(A16, 1, 1024, 1024, ok, None, None, 0, None) == pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    assert g(A16 + 8, 1, 1024, 1024, ok, None, A16, ws, None) == pkg.IMP_ERR_MISALIGNED
    # M = 0: nothing to do
    assert g(A16, 0, 1024, 1024, ok, None, None, 0, None) == pkg.IMP_OK


def test_formats_reject_bad_arguments():
    MX, F8 = pkg.ImpMxfp4Tensor, pkg.ImpFp8Tensor
    q = pkg.imp_mxfp4_quantize
    assert q(A16, 4, 48, 48, MX(A16, A16, 4, 48), None, None) == pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert q(A16, 4, 64, 64, MX(A16, A16, 5, 64), None, None) == pkg.IMP_ERR_INVALID_ARG
    assert q(A16 + 8, 4, 64, 64, MX(A16, A16, 4, 64), None, None) == pkg.IMP_ERR_MISALIGNED
    c = pkg.imp_mxfp4_to_nvfp4
    ws = pkg.imp_mxfp4_to_nvfp4_workspace_size()
    assert c(MX(A16, A16, 4, 32), _t(4, 32), None, A16, ws, None) == pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert c(MX(A16, A16, 4, 64), _t(5, 64), None, A16, ws, None) == pkg.IMP_ERR_INVALID_ARG
    assert c(MX(A16, A16, 4, 64), _t(4, 64), None, None, 0, None) == pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    f = pkg.imp_fp8_quantize
    fws = pkg.imp_fp8_quantize_workspace_size(4, 64)
    assert f(A16, 4, 40, 40, F8(A16, A16, 4, 40), None, A16, fws, None) == pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert f(A16, 4, 64, 64, F8(A16, A16, 4, 64), None, None, 0, None) == pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    g = pkg.imp_fp8_gemm
    gws = pkg.imp_fp8_gemm_workspace_size(1, 1024, 1024)
    assert gws > 0
    assert g(A16, 1, 1000, 1000, F8(A16, A16, 1024, 1000), A16, 1024, None, A16, gws, None) == \
        pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert g(A16, 17, 1024, 1024, F8(A16, A16, 1024, 1024), A16, 1024, None, A16, gws, None) == \
        pkg.IMP_ERR_UNSUPPORTED_SHAPE
    assert g(A16, 1, 1024, 1024, F8(A16, A16, 1024, 1024), A16, 1024, None, A16, gws - 16, None) == \
        pkg.IMP_ERR_WORKSPACE_TOO_SMALL
    assert g(A16, 1, 1024, 1024, F8(A16, A16, 1024, 1024), A16 + 8, 1024, None, A16, gws, None) == \
        pkg.IMP_ERR_MISALIGNED
    assert g(A16, 0, 1024, 1024, F8(A16, A16, 1024, 1024), A16, 1024, None, None, 0, None) == pkg.IMP_OK
    assert pkg.imp_fp8_gemm_plan(1, 17408, 5120) == (2, "gemv_f4r_kernel")
    assert pkg.imp_fp8_gemm_plan(1, 5120, 17408) == (2, "gemv_f4r_kernel")
