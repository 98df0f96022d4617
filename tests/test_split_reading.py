"""The decode path's reading of a bf16 activation as eight NVFP4 components
(each component quantizes what the previous ones left: block amax / 6 ->
E4M3 scale in units of 2^(4 - 2c), value / scale -> E2M1 nearest, the
residual updated with the exact product), restated here with the oracle's
E4M3/E2M1 encoders.  As on the device, the power-of-two prescale comes from
the whole row's max|x| (it puts that max in [2^14, 2^15)), so a block far
below the row's largest value is split from small E4M3 scales.  After eight
components every residual is a tiny fraction of the row's largest value, and
its effect on a dot product is a negligible share of the GEMM's
2e-3 * sum|x w| band."""
import math

import numpy as np

import oracle


def _bf16(x):
    u = x.astype(np.float32).view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def prescale_exponent(row):
    """sh with max|row| * 2^sh in [2^14, 2^15) (0 for an all-zero row)."""
    mx = np.abs(row).max()
    if mx == 0:
        return 0
    _, e = math.frexp(mx)
    return 15 - e


def split_block(x, sh):
    """Residual of one 16-element block after the eight-component split, in
    true units (fp32 arithmetic as on the device)."""
    r = (x * 2.0 ** sh).astype(np.float32)
    for c in range(8):
        amax = np.float32(np.abs(r).max())
        u = np.float32(amax * np.float32(1.0 / 6.0) * np.float32(2.0 ** (2 * c - 4)))
        d = np.float32(oracle.e4m3_value(oracle.e4m3_encode(float(u))) * 2.0 ** (4 - 2 * c))
        if d == 0:
            continue
        inv = np.float32(1.0) / d
        for k in range(16):
            q = np.float32(r[k] * inv)
            v = oracle.e2m1_value(oracle.e2m1_encode(abs(float(q))))
            r[k] = np.float32(r[k] - np.float32(math.copysign(v, q) * d))
    return r.astype(np.float64) * 2.0 ** -sh


def split_row(row):
    sh = prescale_exponent(row)
    return np.concatenate([split_block(row[b:b + 16], sh) for b in range(0, len(row), 16)])


def test_residual_negligible_with_the_row_prescale():
    # rows of 16 blocks; an outlier channel in one block (x20 as in the decode
    # workloads, and far larger ratios), quiet blocks, zero blocks
    rng = np.random.default_rng(0)
    worst_rel, worst_band = 0.0, 0.0
    for trial in range(60):
        row = rng.standard_normal(256) * 2.0 ** int(rng.integers(-30, 30))
        k_out = int(rng.integers(256))
        row[k_out] *= [20.0, 1e3, 2.0 ** 20, 2.0 ** 40][trial % 4]
        if trial % 5 == 0:
            row[32:64] *= 2.0 ** -30  # blocks far below the row's max
        if trial % 7 == 0:
            row[96:112] = 0.0
        row = _bf16(row)
        r = split_row(row)
        worst_rel = max(worst_rel, float(np.abs(r).max() / np.abs(row).max()))
        # a dot product with a weight row: the split's error against the band
        w = rng.standard_normal(256) * 0.02
        band = 2e-3 * float(np.abs(row * w).sum())
        worst_band = max(worst_band, abs(float((r * w).sum())) / band)
    assert worst_rel < 4e-9, worst_rel
    assert worst_band < 1e-4, worst_band


def test_small_blocks_beside_an_outlier():
    # Blocks 2^10 .. 2^24 below the row's outlier.  The row prescale leaves
    # such a block's components with small (for the last ones subnormal) E4M3
    # scales, so its residual relative to its own largest value grows with
    # the distance (about 2e-7 at 2^10, 3e-3 at 2^24), while relative to the
    # row's largest value -- what a dot product's band measures -- it stays
    # below 1e-9.
    rng = np.random.default_rng(1)
    base = _bf16(rng.standard_normal(32))
    for dist, own_bound in ((2.0 ** 10, 1e-6), (2.0 ** 16, 1e-4), (2.0 ** 24, 1e-2)):
        row = base.copy()
        row[0] = dist * np.abs(base).max()
        row = _bf16(row)
        r = split_row(row)
        assert np.abs(r).max() <= 1e-9 * np.abs(row).max()
        assert np.abs(r[16:32]).max() <= own_bound * np.abs(row[16:32]).max()


def test_exact_when_the_block_is_representable():
    # a block that is already 16 E2M1 codes times one E4M3 scale: the first
    # component takes it exactly
    x = _bf16(np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 6.0]) * 0.75)
    assert np.abs(split_row(x)).max() == 0.0


# ---- the FP8 weight path's reading of X: eight E4M3 components ----------------

def split_row_e4m3(row):
    """x * 2^sh = sum_c 2^(-4c) e4m3(q_c), q_c the E4M3 rounding of 2^(4c)
    times what components 0..c-1 left; sh puts max|x| in [2^7, 2^8).
    Returns the residual in true units (fp32 arithmetic as on the device)."""
    mx = np.abs(row).max()
    sh = 0 if mx == 0 else 8 - math.frexp(mx)[1]
    r = (row * 2.0 ** sh).astype(np.float32)
    for c in range(8):
        for k in range(len(r)):
            u = float(r[k]) * 2.0 ** (4 * c)
            mag = oracle.e4m3_value(oracle.e4m3_encode(abs(u)))
            v = math.copysign(mag, u)
            r[k] = np.float32(r[k] - np.float32(v * 2.0 ** (-4 * c)))
    return r.astype(np.float64) * 2.0 ** -sh


def test_e4m3_split_residual_negligible():
    rng = np.random.default_rng(7)
    worst = 0.0
    for i in range(20):
        row = _bf16(rng.standard_normal(128) * 2.0 ** rng.integers(-20, 20))
        row[rng.integers(0, 128, 3)] *= 20.0 * (i + 1)
        if i % 5 == 0:
            row[rng.integers(0, 128, 8)] *= 2.0 ** -30  # far below the row max
        res = split_row_e4m3(row)
        worst = max(worst, np.abs(res).max() / np.abs(row).max())
        # its share of a dot product's band with any weights
        w = rng.standard_normal(128)
        assert abs(np.dot(res, w)) <= 1e-4 * 2e-3 * np.sum(np.abs(row * w)) + 1e-300
    assert worst < 1e-9


def test_e4m3_split_exact_for_two_component_values():
    # a bf16 value has 8 significant bits: two E4M3 components (4 bits each)
    # hold it exactly when it is within the E4M3 normal range after the prescale
    row = _bf16(np.array([1.0, -1.5, 3.0 + 2 ** -6, 100.0, -255.0, 2 ** -3 + 2 ** -7] * 2))
    assert np.all(split_row_e4m3(row) == 0.0)
