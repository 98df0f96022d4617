"""Pins of the oracle's MXFP4 and FP8-E4M3 weight functions, against things
other than the oracle itself: hand-worked blocks (tests/golden/mxfp4,
tests/golden/fp8), torch's E8M0 and E4M3 casts, exact rational brute force,
and the definitions' invariants."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from _golden import bf16_bits, format_cases

E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---- MXFP4 --------------------------------------------------------------------

def test_e8m0_decode_all_bytes():
    # torch's float8_e8m0fnu (a library routine) and the power of two itself
    ref = torch.arange(255, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for b in range(255):
        v = oracle.e8m0_value(b)
        assert v == ref[b] == math.ldexp(1.0, b - 127), b
    assert math.isnan(oracle.e8m0_value(255))


@pytest.mark.parametrize("case", format_cases("mxfp4"), ids=lambda c: c["name"])
def test_mx_golden_blocks(case):
    codes, scales, bad = oracle.mx_quantize(case["X"])
    assert not bad
    np.testing.assert_array_equal(scales, case["scales_arr"])
    np.testing.assert_array_equal(codes, case["codes_arr"])


def _mx_blocks(seed):
    """Random bf16 rows of 32-element blocks: normal and heavy-tailed values
    over a wide exponent range, outliers, zeros, tiny and huge blocks."""
    rng = np.random.default_rng(seed)
    rows = []
    for kind in range(6):
        v = rng.standard_normal((16, 64)) * np.exp2(rng.integers(-30, 30, (16, 1)))
        if kind == 1:
            v *= rng.standard_t(4, (16, 64))
        if kind == 2:
            v[:, ::9] *= 20
        if kind == 3:
            v[rng.random((16, 64)) < 0.3] = 0
        if kind == 4:
            v = rng.standard_normal((16, 64)) * 2.0 ** -128  # subnormal bf16 range
        if kind == 5:
            v = rng.standard_normal((16, 64)) * 2.0 ** 120
        rows.append(v)
    x = np.concatenate(rows).astype(np.float32)
    x = np.clip(x, -3.3e38, 3.3e38)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_value(bits):
    return float(np.uint32(int(bits) << 16).view(np.float32))


@pytest.mark.parametrize("seed", [0, 1])
def test_mx_scale_and_codes_by_exact_bruteforce(seed):
    """Every block: the scale is 2^e with e the largest integer such that
    4 * 2^e <= amax (clamped to [-127, 127]); every code is the exact-rational
    nearest E2M1 magnitude of |x| / 2^e with ties to the even code, saturating,
    with x's sign."""
    x = _mx_blocks(seed)
    codes, scales, bad = oracle.mx_quantize(x)
    assert not bad
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            vals = [Fraction(_bf16_value(x[r, 32 * b + j])) for j in range(32)]
            amax = max(abs(v) for v in vals)
            e = -127
            if amax > 0:
                e = 127
                while e > -127 and Fraction(4) * Fraction(2) ** e > amax:
                    e -= 1
            assert scales[r, b] == e + 127, (r, b)
            X = Fraction(2) ** e
            for j in range(32):
                q = abs(vals[j]) / X
                d = [abs(q - Fraction(m)) for m in E2M1_MAG]
                best = min(d)
                cand = [i for i in range(8) if d[i] == best]
                want = cand[0] if len(cand) == 1 else [c for c in cand if c % 2 == 0][0]
                if q > 6:
                    want = 7
                bits = int(x[r, 32 * b + j])
                if bits & 0x8000:
                    want |= 8
                byte = int(codes[r, 16 * b + j // 2])
                got = byte & 15 if j % 2 == 0 else byte >> 4
                assert got == want, (r, b, j, float(q), got, want)


def test_mx_dequant_and_reference_gemm_exact():
    lin = synth.Linear("mx", 2, 64, 6, 3, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.05, x_outlier_frac=0.05)
    codes, scales, _ = oracle.mx_quantize(lin.weight_bf16())
    w = oracle.mx_dequant(codes, scales)
    for r in range(6):
        for k in range(64):
            byte = int(codes[r, k // 2])
            c = byte & 15 if k % 2 == 0 else byte >> 4
            mag = Fraction(E2M1_MAG[c & 7]) * Fraction(2) ** (int(scales[r, k // 32]) - 127)
            assert Fraction(w[r, k]) == (-mag if c & 8 else mag)
    x = lin.act_bf16()
    y, bound = oracle.mx_reference_gemm(x, 2, codes, scales)
    for m in range(2):
        for n in range(6):
            terms = [Fraction(_bf16_value(x[m, k])) * Fraction(w[n, k]) for k in range(64)]
            exact = sum(terms, Fraction(0))
            mag = sum((abs(t) for t in terms), Fraction(0))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(64, 2 ** 52) * mag + Fraction(1, 2 ** 1074)


def test_mx_roundtrip_bound_and_clipping():
    """Unclipped elements err by at most half an E2M1 step (times the scale);
    clipping happens only where |x| / 2^e > 6, and then the value is 6 * 2^e."""
    x = _mx_blocks(5)
    codes, scales, _ = oracle.mx_quantize(x)
    w = oracle.mx_dequant(codes, scales)
    xv = oracle.bf16_to_f64(x)
    X = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    q = np.abs(xv) / X
    step = np.where(q <= 2, 0.5, np.where(q <= 4, 1.0, 2.0))
    clip = q > 6
    err = np.abs(w - xv)
    assert np.all(err[~clip] <= 0.5 * step[~clip] * X[~clip])
    np.testing.assert_array_equal(np.abs(w[clip]), 6 * X[clip])
    assert clip.any()  # the workload does reach the clipping region


def test_mx_nonfinite_flag():
    x = bf16_bits([1.0] * 31 + [float("inf")]).reshape(1, 32)
    assert oracle.mx_quantize(x)[2]
    assert not oracle.mx_quantize(bf16_bits([1.0] * 32).reshape(1, 32))[2]


# ---- FP8 E4M3 weights -------------------------------------------------------------

@pytest.mark.parametrize("case", format_cases("fp8"), ids=lambda c: c["name"])
def test_fp8_golden(case):
    codes, s8, bad = oracle.fp8_quantize(case["X"])
    assert not bad
    assert np.float32(s8) == np.float32(case["tensor_scale"])
    np.testing.assert_array_equal(codes, case["codes_arr"])


@pytest.mark.parametrize("seed,dist", [(0, synth.DIST_NORMAL), (1, synth.DIST_STUDENT_T4)])
def test_fp8_vs_torch_cast(seed, dist):
    """codes == torch's E4M3 cast of fp32(x / s8) (torch rounds to nearest
    even; the oracle saturates, torch does not, so |x / s8| <= 448 here by
    construction of s8)."""
    lin = synth.Linear("f8", 1, 256, 48, seed, w_dist=dist, w_scale=0.02, zero_block_p=0.01)
    wb = lin.weight_bf16()
    codes, s8, _ = oracle.fp8_quantize(wb)
    xf = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    q = xf / torch.tensor(np.float32(s8))
    assert float(q.abs().max()) <= 448.0
    ref = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, ref)
    # s8 is the fp32 quotient of the global amax by 448 (torch division)
    amax = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).float().abs().max()
    assert np.float32(s8) == (amax / torch.tensor(448.0)).numpy()


def test_fp8_dequant_exact_and_zero_tensor():
    lin = synth.Linear("f8d", 1, 64, 4, 2, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02)
    codes, s8, _ = oracle.fp8_quantize(lin.weight_bf16())
    w = oracle.fp8_dequant(codes, s8)
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for idx in np.ndindex(codes.shape):
        assert Fraction(w[idx]) == Fraction(e4[codes[idx]]) * Fraction(np.float32(s8).item())
    z = np.zeros((2, 16), np.uint16)
    zc, zs, _ = oracle.fp8_quantize(z)
    assert zs == 0.0 and not zc.any()
    x = oracle.fp8_reference_gemm(lin.act_bf16(), codes, s8)[0]
    assert x.shape == (1, 4)


# ---- SwiGLU reference -------------------------------------------------------------

def test_silu_vs_scipy_expit():
    scipy_special = pytest.importorskip("scipy.special")
    v = np.concatenate([np.linspace(-30, 30, 2001), [-800.0, -1e-300, 0.0, 1e-300, 800.0]])
    ref = v * scipy_special.expit(v)
    got = oracle.silu(v)
    assert np.all(np.abs(got - ref) <= 4e-16 * np.abs(ref) + 1e-300)
    # the slope bound the band uses
    h = 1e-6
    slope = np.abs((oracle.silu(v + h) - oracle.silu(v - h)) / (2 * h))
    assert slope.max() <= oracle.SILU_SLOPE_MAX and slope.max() > 1.09


def test_swiglu_band_admits_worst_case_and_rejects_a_dropped_block():
    lin_g = synth.Linear("sg", 40, 256, 24, 1, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                         x_outlier_frac=0.01)
    lin_u = synth.Linear("su", 40, 256, 24, 2, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02)
    x = lin_g.act_bf16()
    gate = oracle.quantize(lin_g.weight_bf16())[:3]
    up = oracle.quantize(lin_u.weight_bf16())[:3]
    h, tol = oracle.reference_swiglu(x, 40, gate, up)
    g, bg = oracle.reference_gemm(x, 40, *gate)
    u, bu = oracle.reference_gemm(x, 40, *up)
    # worst-case g and u errors inside the GEMM band, then bf16 rounding
    tg = 2.0 ** -14 * bg + 2.0 ** -22 * np.abs(g)
    tu = 2.0 ** -14 * bu + 2.0 ** -22 * np.abs(u)
    for sg_, su_ in ((1, 1), (1, -1), (-1, 1), (-1, -1)):
        hp = oracle.silu(g + sg_ * tg) * (u + su_ * tu)
        hb = torch.from_numpy(hp.astype(np.float32)).bfloat16().double().numpy()
        assert np.all(np.abs(hb - h) <= tol)
    # a dropped 16-element block of the gate product leaves the band
    xh = oracle.activation_hat(x, 40)
    wg = oracle.dequant(gate[0], gate[1], gate[2])
    drop = (xh[:, 16:32] @ wg[:, 16:32].T)
    hd = oracle.silu(g - drop) * u
    assert np.mean(np.abs(hd - h) > tol) > 0.5
