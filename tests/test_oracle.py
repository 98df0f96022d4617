"""Pins for the oracle: checks against what the element-type definitions,
the NVFP4 recipe and plain mathematics fix, never against the oracle itself."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from _golden import all_cases, bf16_bits

# E2M1 magnitudes for codes 0..7, from the element definition
# (1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit, subnormal at e=0).
E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def torch_e4m3_values():
    """All 256 E4M3 bytes decoded by torch's float8_e4m3fn (a library routine)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e2m1_decode_table():
    for c in range(16):
        mag = E2M1_MAG[c & 7]
        v = oracle.e2m1_value(c)
        assert v == (-mag if c & 8 else mag)
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_e4m3_decode_all_bytes_vs_torch():
    ref = torch_e4m3_values()
    for b in range(256):
        v = oracle.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v), b
        else:
            assert v == ref[b], (b, v, ref[b])
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert math.isnan(oracle.e4m3_value(0x7F))


def _e4m3_probe_points():
    vals = torch_e4m3_values()[:127]
    mids = (vals[:-1] + vals[1:]) / 2
    pts = [vals, mids]
    f = mids.astype(np.float32)
    pts.append(np.nextafter(f, np.float32(np.inf)).astype(np.float64))
    pts.append(np.nextafter(f, np.float32(0)).astype(np.float64))
    rng = np.random.default_rng(1234)
    pts.append(rng.uniform(0, 448, 20000))
    pts.append(np.exp2(rng.uniform(-12, 8.8, 20000)))
    p = np.concatenate(pts).astype(np.float32)
    return p[(p >= 0) & (p <= 448)]


def test_e4m3_encode_vs_torch_cast():
    u = _e4m3_probe_points()
    ref = torch.from_numpy(u).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in u], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, list(zip(u[bad][:5], got[bad][:5], ref[bad][:5]))


def test_e4m3_encode_bruteforce_and_saturation():
    vals = torch_e4m3_values()[:127]
    u = _e4m3_probe_points()[::7]
    for x in u:
        d = np.abs(vals - float(x))
        cands = np.nonzero(d == d.min())[0]
        want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        assert oracle.e4m3_encode(float(x)) == want, x
    for big in [448.0, 448.00003, 460.0, 464.0, 500.0, 1e30, float("inf")]:
        assert oracle.e4m3_encode(big) == 0x7E


def test_e2m1_encode_bruteforce():
    mags = np.array(E2M1_MAG)
    mids = (mags[:-1] + mags[1:]) / 2
    f = np.concatenate([mags, mids]).astype(np.float32)
    pts = np.concatenate([f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(0)),
                          np.linspace(0, 8, 4001, dtype=np.float32), np.float32([6.4, 100, 1e30])])
    for q in pts:
        for sgn in (1.0, -1.0):
            x = np.float32(sgn * q)
            d = np.abs(mags - abs(float(x)))
            cands = np.nonzero(d == d.min())[0]
            want = int(cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0])
            if abs(float(x)) > 6.0:  # saturating encode
                want = 7
            if math.copysign(1.0, float(x)) < 0:
                want |= 8
            assert oracle.e2m1_encode(float(x)) == want, (x, want)
    assert oracle.e2m1_encode(float("inf")) == 7
    assert oracle.e2m1_encode(-0.0) == 8


@pytest.mark.parametrize("case", all_cases(), ids=lambda c: c["name"])
def test_golden_blocks(case):
    codes, scales, s, bad = oracle.quantize(case["X"])
    assert not bad
    assert np.float32(s) == np.float32(case["tensor_scale"])
    np.testing.assert_array_equal(scales, case["scales_arr"])
    np.testing.assert_array_equal(codes, case["codes_arr"])
    for xrow, yexp in case["y"]:
        xh = oracle.bf16_to_f64(bf16_bits(xrow)[None, :])
        y, _ = oracle.matmul_abt(xh, oracle.dequant(codes, scales, s))
        assert list(y[0]) == yexp


def test_golden_tensor_a_decodes_to_inputs():
    case = [c for c in all_cases() if c["name"] == "tensor_a_all_codes.txt"][0]
    codes, scales, s, _ = oracle.quantize(case["X"])
    w = oracle.dequant(codes, scales, s)
    np.testing.assert_array_equal(w, np.array([case["x"][0], case["x"][1]]))


def test_nonfinite_flag():
    x = bf16_bits([1.0] * 16)[None, :].copy()
    x[0, 3] = 0x7F80  # +inf
    assert oracle.quantize(x)[3]
    x[0, 3] = 0x7FC0  # nan
    assert oracle.quantize(x)[3]
    x[0, 3] = 0x3F80
    assert not oracle.quantize(x)[3]


def test_block_scale_saturates_when_u_rounds_above_448():
    # Search bf16 amax values for which fl(fl(g/6)/fl(g/2688)) > 448 and check
    # the scale saturates to 0x7E (never 0x7F, the NaN code).
    found = 0
    for bits in range(0x3F80, 0x4780):
        g = np.uint32(bits << 16).view(np.float32)
        s = np.float32(g) / np.float32(2688)
        u = (np.float32(g) / np.float32(6)) / s
        if u > 448:
            x = np.full((1, 16), bits, np.uint16)
            _, scales, _, _ = oracle.quantize(x)
            assert scales[0, 0] == 0x7E
            found += 1
    assert found > 0


def _dequant_independent(codes, scales, s):
    """Rows of W from codes/scales with the test's own tables (Fractions)."""
    e4 = torch_e4m3_values()
    rows, kh = codes.shape
    out = []
    for r in range(rows):
        row = []
        for k in range(kh * 2):
            byte = int(codes[r, k // 2])
            c = byte & 15 if k % 2 == 0 else byte >> 4
            mag = Fraction(E2M1_MAG[c & 7])
            row.append((-mag if c & 8 else mag) * Fraction(float(e4[scales[r, k // 16]])) * Fraction(float(s)))
        out.append(row)
    return out


@pytest.mark.parametrize("M,N,K,seed", [(1, 8, 64, 0), (3, 5, 128, 1), (2, 8, 128, 2)])
def test_matmul_exact_rational(M, N, K, seed):
    lin = synth.Linear("exact", M, K, N, seed, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.05, x_outlier_frac=0.05)
    w = lin.weight_bf16()
    x = lin.act_bf16()
    codes, scales, s, _ = oracle.quantize(w)
    y, bound = oracle.reference_gemm(x, M, codes, scales, s)
    wq = _dequant_independent(codes, scales, s)
    xf = x.astype(np.uint32) << 16
    xv = [[Fraction(float(np.uint32(b).view(np.float32))) for b in row] for row in xf]
    for m in range(M):
        for n in range(N):
            terms = [xv[m][k] * wq[n][k] for k in range(K)]
            exact = sum(terms, Fraction(0))
            mag = sum((abs(t) for t in terms), Fraction(0))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(K, 2 ** 52) * mag + Fraction(1, 2 ** 1074)
            assert abs(Fraction(bound[m, n]) - mag) <= Fraction(K, 2 ** 52) * mag


def test_quantize_rows_equals_whole_tensor():
    lin = synth.Linear("rows", 1, 256, 40, 7, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.02)
    w = lin.weight_bf16()
    codes, scales, s, _ = oracle.quantize(w)
    g, s2, _ = oracle.tensor_scale(w)
    assert s2 == s and g == np.abs((w.astype(np.uint32) << 16).view(np.float32)).max()
    sel = [0, 7, 39]
    c2, sc2 = oracle.quantize_rows(w[sel], s)
    np.testing.assert_array_equal(c2, codes[sel])
    np.testing.assert_array_equal(sc2, scales[sel])


def _e2m1_half_ulp(qabs):
    return np.where(qabs <= 2, 0.25, np.where(qabs <= 4, 0.5, 1.0))


@pytest.mark.parametrize("dist,scale", [(synth.DIST_STUDENT_T4, 0.02), (synth.DIST_NORMAL, 1.0),
                                        (synth.DIST_NORMAL, 1e-4)])
def test_roundtrip_error_bound(dist, scale):
    lin = synth.Linear("rt", 1, 1024, 64, 11, w_dist=dist, w_scale=scale, zero_block_p=0.01)
    w = lin.weight_bf16()
    codes, scales, s, _ = oracle.quantize(w)
    xq = oracle.dequant(codes, scales, s)
    xv = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    e4 = torch_e4m3_values()
    d = (e4[scales].astype(np.float32) * np.float32(s)).astype(np.float64)  # fp32 product, as defined
    d = np.repeat(d, 16, axis=1)
    err = np.abs(xq - xv)
    amax = np.repeat(np.abs(xv).reshape(64, -1, 16).max(axis=2), 16, axis=1)
    u = np.repeat(e4[scales], 16, axis=1)
    normal = u >= 2.0 ** -6
    with np.errstate(divide="ignore", invalid="ignore"):
        qabs = np.where(d > 0, np.abs(xv) / d, 0)
    # Normal block scales: at most half an E2M1 ulp (in units of d), clip
    # included, since E4M3 rounding keeps |q| <= 6.4.
    lim = _e2m1_half_ulp(np.minimum(qabs, 6.0)) * d * (1 + 1e-6)
    assert np.all(err[normal & (d > 0)] <= lim[normal & (d > 0)])
    assert np.all(qabs[normal] <= 6.4 + 1e-6)
    # Subnormal block scales may clip further: err <= max(half ulp * d, amax - 6 d).
    sub = ~normal & (d > 0)
    lim2 = np.maximum(lim, amax - 6 * d) * (1 + 1e-6)
    assert np.all(err[sub] <= lim2[sub])
    # Zero-scale blocks dequantize to zero.
    assert np.all(xq[d == 0] == 0)


def test_tolerance_admits_correctly_rounded_bf16_and_tight_band_catches_a_dropped_block():
    # One-signed short sums: |y| close to sum|x w|, where bf16 rounding alone
    # exceeds 2e-3 * sum|x w|; the acceptance band must still admit the
    # correctly rounded bf16 of the exact value.
    rng = np.random.default_rng(3)
    y = rng.uniform(0.5, 100.0, 10000) * rng.choice([-1, 1], 10000)
    yb = torch.from_numpy(y).to(torch.bfloat16).to(torch.float64).numpy()
    bound = np.abs(y)
    assert np.all(np.abs(yb - y) <= oracle.tolerance(bound, y))
    assert np.all(np.abs(yb - y) <= oracle.tight_tolerance(bound, y))
    # Plant a mistake in an oracle result (drop one 16-element block of a
    # K = 5120 row) and check the tight band rejects it.
    lin = synth.Linear("drop", 1, 5120, 64, 21, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02)
    codes, scales, s, _ = oracle.quantize(lin.weight_bf16())
    x = lin.act_bf16()
    y_ref, bound = oracle.reference_gemm(x, 1, codes, scales, s)
    scales2 = scales.copy()
    scales2[:, 100] = 0
    y_bad, _ = oracle.reference_gemm(x, 1, codes, scales2, s)
    err = np.abs(y_bad - y_ref)
    assert np.mean(err > oracle.tight_tolerance(bound, y_ref)) > 0.5
