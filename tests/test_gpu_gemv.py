"""Decode path (M <= 16) vs the oracle: every element of Y within
|y - y_ref| <= 2e-3 * sum|x w| + 1e-5, on the workload shapes (full size;
the largest checked on sampled output columns) and edge shapes; results
bitwise repeatable."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import check_within_tolerance, dev_bf16, dev_nvfp4, sample_rows

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def run_gemm(x_bits, w_dev, ldx=None, ldy=None, via="gemm"):
    x = dev_bf16(x_bits, ldx)
    M, N = x_bits.shape[0], w_dev.rows
    ldy = ldy or N
    ybig = torch.full((M, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = ybig[:, :N]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if via == "gemm":
        pkg.gemm(x, w_dev, y=y, dev_status=status)
    else:  # the weight in MMA layout (decode kernels read 16 KB tiles)
        pkg.gemm_mma(x, pkg.prepare_mma(w_dev), y=y, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y.float().cpu().numpy()


def mma_ok(M, K, N):
    """Shapes the decode path of gemm_mma takes."""
    return K % 256 == 0 and K >= 1024 and N >= 128


def oracle_w(lin):
    bits = lin.weight_bf16()
    c, s, ts, _ = oracle.quantize(bits)
    return c, s, ts


SMALL = synth.workload("single_1k") + synth.workload("decode_0p6b")


@pytest.mark.parametrize("via", ["gemm", "gemm_mma"])
@pytest.mark.parametrize("lin", SMALL, ids=lambda l: f"{l.name}_{l.K}x{l.N}")
def test_small_workloads_every_element(lin, via):
    c, s, ts = oracle_w(lin)
    x = lin.act_bf16()
    y = run_gemm(x, dev_nvfp4(c, s, ts), via=via)
    y_ref, bound = oracle.reference_gemm(x, lin.M, c, s, ts)
    check_within_tolerance(y, y_ref, bound, lin.name)


FULL = synth.workload("decode_27b") + synth.workload("skinny_27b")


@pytest.mark.parametrize("via", ["gemm", "gemm_mma"])
@pytest.mark.parametrize("lin", FULL, ids=lambda l: f"{l.name}_M{l.M}_{l.K}x{l.N}")
def test_full_size_sampled(lin, via):
    w_bits = lin.weight_bf16()
    w = pkg.quantize(dev_bf16(w_bits))
    x = lin.act_bf16()
    y = run_gemm(x, w, via=via)
    _, ts, _ = oracle.tensor_scale(w_bits)
    rows = sample_rows(lin.N, seed=lin.N + lin.M)
    c, s = oracle.quantize_rows(w_bits[rows], ts)
    # the device weight equals the oracle's on the sampled rows
    assert np.array_equal(w.codes.cpu().numpy()[rows], c)
    assert np.array_equal(w.scales.cpu().numpy()[rows], s)
    y_ref, bound = oracle.reference_gemm(x, lin.M, c, s, ts)
    check_within_tolerance(y[:, rows], y_ref, bound, lin.name)
    assert np.isfinite(y).all()


@pytest.mark.parametrize("M,K,N,ldx,ldy", [
    (1, 64, 1, 64, 8), (1, 64, 7, 72, 16), (1, 320, 333, 320, 336), (2, 192, 50, 200, 56),
    (3, 1024, 1000, 1024, 1000), (5, 2048, 77, 2056, 80), (7, 448, 9, 448, 16),
    (16, 64, 300, 64, 304), (9, 5120, 129, 5120, 136), (1, 17408, 5, 17408, 8),
    (16, 1024, 2, 1024, 8), (1, 4096, 152, 4096, 152), (1, 4096, 153, 4096, 160),
    # tensor-core tiles of 2, 4 and 8 rows of X: several units per warp,
    # partial last units (K % (128 * 8 / MT) != 0), scales read from global
    # memory (K % 256 != 0), several passes with inactive rows
    (8, 5120, 333, 5120, 336), (6, 3072, 200, 3080, 200), (8, 192, 70, 192, 72),
    (4, 17408, 100, 17408, 104), (11, 2304, 97, 2304, 104), (13, 1088, 40, 1088, 40),
    (2, 320, 19, 320, 24), (4, 576, 1500, 576, 1504),
    # the tensor-memory path (M <= 2, K % 256 == 0): one pair per row, a
    # half-filled last pair, a last stage with fewer pairs, ragged row
    # blocks, fewer row blocks than SMs, padded X rows
    (1, 512, 32, 512, 32), (1, 768, 1000, 768, 1000), (1, 1280, 4097, 1288, 4104),
    (2, 1280, 333, 1280, 336), (2, 768, 64, 776, 64), (1, 2560, 9733, 2560, 9736),
    (2, 17408, 200, 17408, 200),
    # the FP4 path's schedules for one or two rows of X: whole tiles (at
    # least 3/4 as many tiles as SMs, a ragged last tile), K split over
    # clusters of 3 and 8 CTAs (ragged last tile, uneven chunk parts),
    # stream-K (tiles between half and 3/4 of the SMs)
    (1, 1024, 15355, 1024, 15360), (2, 1024, 14600, 1032, 14600),
    (1, 3072, 6000, 3072, 6000), (2, 5120, 2431, 5120, 2432), (1, 2304, 300, 2304, 304),
    (1, 2048, 12000, 2048, 12000), (2, 6144, 1111, 6144, 1112)])
def test_edge_shapes(M, K, N, ldx, ldy):
    lin = synth.Linear("edge", M, K, N, 123, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.02, x_outlier_frac=0.02)
    c, s, ts = oracle_w(lin)
    x = lin.act_bf16()
    y_ref, bound = oracle.reference_gemm(x, M, c, s, ts)
    vias = ["gemm", "gemm_mma"] if mma_ok(M, K, N) else ["gemm"]
    for via in vias:
        y = run_gemm(x, dev_nvfp4(c, s, ts), ldx, ldy, via=via)
        check_within_tolerance(y, y_ref, bound, f"M{M} K{K} N{N} {via}")


@pytest.mark.parametrize("M,K,N", [(1, 41536, 100), (3, 41536, 40)])
def test_cuda_core_kernel_shapes(M, K, N):
    # K too long for the f16 path's register-resident X and K % 256 != 0
    # (no FP4 path): the CUDA-core kernel takes these
    assert pkg.imp_nvfp4_gemm_plan(M, N, K)[1] == "gemv_kernel"
    lin = synth.Linear("cc", M, K, N, 77, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.02, x_outlier_frac=0.02)
    c, s, ts = oracle_w(lin)
    x = lin.act_bf16()
    y_ref, bound = oracle.reference_gemm(x, M, c, s, ts)
    y = run_gemm(x, dev_nvfp4(c, s, ts), ldy=(N + 7) // 8 * 8)
    check_within_tolerance(y, y_ref, bound, f"M{M} K{K} N{N} cuda cores")


def test_gemm_mma_rejects_shapes_outside_the_decode_path():
    lin = synth.Linear("rej", 1, 320, 200, 3)
    c, s, ts = oracle_w(lin)
    with pytest.raises(pkg.ImpError, match="UNSUPPORTED_SHAPE"):
        run_gemm(lin.act_bf16(), dev_nvfp4(c, s, ts), via="gemm_mma")


def test_extreme_activation_magnitudes():
    # X spanning bf16's range (huge, tiny, subnormal): the f16 staging of X
    # must not overflow or flush.
    lin = synth.Linear("mag", 1, 1024, 64, 5)
    c, s, ts = oracle_w(lin)
    rng = np.random.default_rng(0)
    for exp in (-130, -60, -20, 0, 20, 60, 120):
        xf = (rng.standard_normal((1, 1024)) * 2.0 ** exp).astype(np.float32)
        xb = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        y = run_gemm(xb, dev_nvfp4(c, s, ts))
        y_ref, bound = oracle.reference_gemm(xb, 1, c, s, ts)
        if exp <= 120 - 10:
            check_within_tolerance(y, y_ref, bound, f"x ~ 2^{exp}")


@pytest.mark.parametrize("N", [96, 160])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 12])
def test_extreme_activation_magnitudes_per_row(M, N):
    # Rows of X of very different magnitude in one call: each row keeps its
    # own power-of-two staging factor (N = 160 takes the FP4 path, 96 not).
    lin = synth.Linear("mag", M, 2048, N, 6)
    c, s, ts = oracle_w(lin)
    rng = np.random.default_rng(M)
    exps = [(-130, -60, -20, 0, 20, 60, 100)[i % 7] for i in range(M)]
    xf = np.stack([rng.standard_normal(2048) * 2.0 ** e for e in exps]).astype(np.float32)
    xb = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = run_gemm(xb, dev_nvfp4(c, s, ts))
    y_ref, bound = oracle.reference_gemm(xb, M, c, s, ts)
    check_within_tolerance(y, y_ref, bound, f"M{M} rows ~ 2^{exps}")


@pytest.mark.parametrize("via", ["gemm", "gemm_mma"])
def test_bitwise_repeatable(via):
    lin = synth.workload("decode_27b")[2]
    w = pkg.quantize(dev_bf16(lin.weight_bf16()))
    x = lin.act_bf16()
    a = run_gemm(x, w, via=via)
    b = run_gemm(x, w, via=via)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_prepared_and_row_major_weights_give_identical_results():
    # same kernels and schedule, only the copies differ
    lin = synth.workload("decode_27b")[0]
    w = pkg.quantize(dev_bf16(lin.weight_bf16()))
    x = lin.act_bf16()
    a = run_gemm(x, w, via="gemm")
    b = run_gemm(x, w, via="gemm_mma")
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
