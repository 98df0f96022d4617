"""MXFP4 and FP8-E4M3 weights on the GPU vs the oracle: both quantizers
bit-exact; the MXFP4 -> NVFP4 conversion value-exact (and its range flag);
GEMV / GEMM on MXFP4 weights (through the NVFP4 kernels) and the FP8 GEMV
within the band on every checked element; repeatability."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _golden import format_cases
from _gpu import check_within_tolerance, dev_bf16, sample_rows

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def status0():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---- MXFP4 ------------------------------------------------------------------------

@pytest.mark.parametrize("case", format_cases("mxfp4"), ids=lambda c: c["name"])
def test_mx_quantize_golden(case):
    st = status0()
    t = pkg.mxfp4_quantize(dev_bf16(case["X"]), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(t.scales.cpu().numpy(), case["scales_arr"])
    np.testing.assert_array_equal(t.codes.cpu().numpy(), case["codes_arr"])


@pytest.mark.parametrize("rows,K,ld,seed", [(300, 1024, 1024, 0), (7, 96, 104, 1),
                                            (17408, 5120, 5120, 2)])
def test_mx_quantize_bit_exact(rows, K, ld, seed):
    lin = synth.Linear("mxq", 1, K, rows, seed, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.001)
    wb = lin.weight_bf16()
    t = pkg.mxfp4_quantize(dev_bf16(wb, ld))
    c, s, _ = oracle.mx_quantize(wb)
    np.testing.assert_array_equal(t.scales.cpu().numpy(), s)
    np.testing.assert_array_equal(t.codes.cpu().numpy(), c)


def test_mx_quantize_random_bit_patterns_and_nonfinite():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 16, size=(64, 256), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] &= 0xBFFF  # no NaN/Inf: clear an exponent bit
    t = pkg.mxfp4_quantize(dev_bf16(bits))
    c, s, bad = oracle.mx_quantize(bits)
    assert not bad
    np.testing.assert_array_equal(t.scales.cpu().numpy(), s)
    np.testing.assert_array_equal(t.codes.cpu().numpy(), c)
    bits[5, 17] = 0x7F80  # +Inf
    st = status0()
    pkg.mxfp4_quantize(dev_bf16(bits), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & pkg.IMP_DEV_NONFINITE_INPUT


def test_mx_to_nvfp4_value_exact():
    lin = synth.Linear("mxc", 1, 1024, 640, 4, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.01)
    wb = lin.weight_bf16()
    mx = pkg.mxfp4_quantize(dev_bf16(wb))
    st = status0()
    nv = pkg.mxfp4_to_nvfp4(mx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c, s, _ = oracle.mx_quantize(wb)
    ts = float(nv.tensor_scale.item())
    assert np.frexp(ts)[0] == 0.5  # a power of two
    np.testing.assert_array_equal(nv.codes.cpu().numpy(), c)
    np.testing.assert_array_equal(oracle.dequant(nv.codes.cpu().numpy(), nv.scales.cpu().numpy(), ts),
                                  oracle.mx_dequant(c, s))


def test_mx_to_nvfp4_range_flag():
    # two nonzero blocks 2^50 apart: the small one cannot be an E4M3 scale
    # under the large one's tensor scale
    codes = np.full((2, 32), 0x22, np.uint8)
    scales = np.array([[200, 200], [150, 150]], np.uint8)
    mx = pkg.MXFP4Tensor(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    st = status0()
    pkg.mxfp4_to_nvfp4(mx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & pkg.IMP_DEV_RANGE
    # 17 binades apart is still exact
    scales[1] = 200 - 17
    mx = pkg.MXFP4Tensor(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    st = status0()
    nv = pkg.mxfp4_to_nvfp4(mx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(
        oracle.dequant(nv.codes.cpu().numpy(), nv.scales.cpu().numpy(), float(nv.tensor_scale.item())),
        oracle.mx_dequant(codes, scales))


@pytest.mark.parametrize("M,K,N", [(1, 1024, 1024), (2, 5120, 640), (4, 2048, 312), (16, 1024, 256),
                                   (200, 1024, 512)])
@pytest.mark.parametrize("via", ["gemm", "gemm_mma"])
def test_mx_weights_gemm_every_element(M, K, N, via):
    lin = synth.Linear("mxg", M, K, N, 9, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.01, x_outlier_frac=0.01)
    wb, xb = lin.weight_bf16(), lin.act_bf16()
    nv = pkg.mxfp4_to_nvfp4(pkg.mxfp4_quantize(dev_bf16(wb)))
    st = status0()
    if via == "gemm":
        y = pkg.gemm(dev_bf16(xb), nv, dev_status=st)
    else:
        y = pkg.gemm_mma(dev_bf16(xb), pkg.prepare_mma(nv), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c, s, _ = oracle.mx_quantize(wb)
    y_ref, bound = oracle.mx_reference_gemm(xb, M, c, s)
    check_within_tolerance(y.float().cpu().numpy(), y_ref, bound, f"mxfp4 {via} M{M}")


def test_mx_weights_27b_lm_head_sampled():
    lin = [l for l in synth.workload("decode_27b") if l.name == "lm_head"][0]
    wb = lin.weight_bf16()
    nv = pkg.prepare_mma(pkg.mxfp4_to_nvfp4(pkg.mxfp4_quantize(dev_bf16(wb))))
    xb = lin.act_bf16()
    y = pkg.gemm_mma(dev_bf16(xb), nv).float().cpu().numpy()
    rows = sample_rows(lin.N, seed=11)
    c, s, _ = oracle.mx_quantize(wb[rows])
    y_ref, bound = oracle.mx_reference_gemm(xb, 1, c, s)
    check_within_tolerance(y[:, rows], y_ref, bound, "mxfp4 lm_head")


# ---- FP8 E4M3 weights --------------------------------------------------------------

@pytest.mark.parametrize("case", format_cases("fp8"), ids=lambda c: c["name"])
def test_fp8_quantize_golden(case):
    t = pkg.fp8_quantize(dev_bf16(case["X"]))
    assert np.float32(t.tensor_scale.item()) == np.float32(case["tensor_scale"])
    np.testing.assert_array_equal(t.codes.cpu().numpy(), case["codes_arr"])


@pytest.mark.parametrize("rows,K,ld,seed", [(300, 1024, 1024, 0), (9, 48, 56, 1),
                                            (5120, 17408, 17408, 2)])
def test_fp8_quantize_bit_exact(rows, K, ld, seed):
    lin = synth.Linear("f8q", 1, K, rows, seed, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.001)
    wb = lin.weight_bf16()
    t = pkg.fp8_quantize(dev_bf16(wb, ld))
    c, s8, _ = oracle.fp8_quantize(wb)
    assert np.float32(t.tensor_scale.item()) == np.float32(s8)
    np.testing.assert_array_equal(t.codes.cpu().numpy(), c)


def test_fp8_quantize_random_bit_patterns_and_zero():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=(32, 128), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] &= 0xBFFF
    t = pkg.fp8_quantize(dev_bf16(bits))
    c, s8, _ = oracle.fp8_quantize(bits)
    assert np.float32(t.tensor_scale.item()) == np.float32(s8)
    np.testing.assert_array_equal(t.codes.cpu().numpy(), c)
    z = pkg.fp8_quantize(dev_bf16(np.zeros((4, 64), np.uint16)))
    assert float(z.tensor_scale.item()) == 0.0 and not z.codes.cpu().numpy().any()


def run_fp8(lin, ldx=None, ldy=None, rows=None):
    wb, xb = lin.weight_bf16(), lin.act_bf16()
    w = pkg.fp8_quantize(dev_bf16(wb))
    st = status0()
    x = dev_bf16(xb, ldx)
    ybig = torch.full((lin.M, ldy or lin.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkg.gemm_fp8(x, w, y=ybig[:, :lin.N], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    y = ybig[:, :lin.N].float().cpu().numpy()
    s8, _ = oracle.fp8_tensor_scale(wb)
    rows = np.arange(lin.N) if rows is None else rows
    c = oracle.fp8_quantize_rows(wb[rows], s8)
    np.testing.assert_array_equal(w.codes.cpu().numpy()[rows], c)
    y_ref, bound = oracle.fp8_reference_gemm(xb, c, s8)
    check_within_tolerance(y[:, rows], y_ref, bound, f"fp8 {lin.name} M{lin.M}")
    return ybig


@pytest.mark.parametrize("M,K,N,ldx,ldy", [(1, 1024, 1024, None, None), (2, 1024, 3072, None, None),
                                           (1, 512, 128, None, None), (3, 640, 130, 648, 136),
                                           (5, 2048, 1000, None, 1000), (16, 1024, 256, None, None),
                                           (1, 3072, 1024, None, None), (2, 17408, 640, None, None)])
def test_fp8_gemv_every_element(M, K, N, ldx, ldy):
    lin = synth.Linear("f8g", M, K, N, 13, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.01, x_outlier_frac=0.01)
    run_fp8(lin, ldx, ldy)


@pytest.mark.parametrize("lin", synth.workload("decode_27b"), ids=lambda l: l.name)
def test_fp8_gemv_27b_sampled(lin):
    run_fp8(lin, rows=sample_rows(lin.N, seed=lin.N + 8))


def test_fp8_gemv_repeatable_and_plan():
    lin = synth.Linear("f8r", 1, 5120, 5120, 17, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02)
    w = pkg.fp8_quantize(dev_bf16(lin.weight_bf16()))
    x = dev_bf16(lin.act_bf16())
    outs = [pkg.gemm_fp8(x, w).clone() for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert pkg.imp_fp8_gemm_plan(1, 5120, 5120) == (2, "gemv_f4r_kernel")
    assert pkg.imp_fp8_gemm_plan(5, 5120, 5120) == (6, "gemv_f4r_kernel")
    assert pkg.imp_fp8_gemm_plan(17, 5120, 5120) == (0, None)


def test_fp8_quotients_next_to_rounding_boundaries():
    """Elements whose x / s8 lies within 2^-20 (relative) of the midpoint of
    two E4M3 values, where a quotient computed as x * (1/s8) could round
    differently from the division.  Each tensor's amax g (exact in bf16, not
    a multiple of 7) gives s8 = g / 448 a full 24-bit mantissa; the search
    runs over many g."""
    e4 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (e4[:-1] + e4[1:]) / 2
    mids = mids[mids > 2.0 ** -6]
    found = 0
    rng = np.random.default_rng(0)
    for gi in range(256, 448):
        g = np.float32(gi)
        if gi % 7 == 0:
            continue
        s8 = float(np.float32(g / np.float32(448.0)))
        cand = torch.tensor(mids * s8).bfloat16().float()
        near = []
        for c in (cand, torch.nextafter(cand, torch.zeros_like(cand)).bfloat16().float(),
                  torch.nextafter(cand, torch.full_like(cand, 1e30)).bfloat16().float()):
            v = c.double().numpy()
            ok = (v > 0) & (v < gi) & (np.abs(v / s8 - mids) / mids < 2.0 ** -20)
            near += v[ok].tolist()
        if not near:
            continue
        row = np.zeros(128, np.float32)
        row[0] = g
        row[1:1 + min(len(near), 127)] = near[:127]
        row *= np.where(rng.random(128) < 0.5, -1.0, 1.0).astype(np.float32)
        bits = torch.from_numpy(row.reshape(1, 128)).bfloat16().view(torch.int16).numpy().view(np.uint16)
        t = pkg.fp8_quantize(dev_bf16(bits))
        c, s, _ = oracle.fp8_quantize(bits)
        assert np.float32(t.tensor_scale.item()) == np.float32(s)
        np.testing.assert_array_equal(t.codes.cpu().numpy(), c)
        found += len(near)
    assert found >= 10
