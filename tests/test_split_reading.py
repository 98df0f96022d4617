"""The decode path's reading of a bf16 activation as eight NVFP4 components
(each component quantizes what the previous ones left: block amax / 6 ->
E4M3 scale in units of 2^(4 - 2c), value / scale -> E2M1 nearest, the
residual updated with the exact product), restated here with the oracle's
E4M3/E2M1 encoders: after eight components the residual of every block is a
tiny fraction of the block's largest value, far inside the GEMM's
2e-3 * sum|x w| band."""
import math

import numpy as np

import oracle


def _bf16(x):
    u = x.astype(np.float32).view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def split_residual(x):
    """Largest |residual| / max|x| after the eight-component split of one
    16-element block (fp32 arithmetic as on the device)."""
    mx = np.abs(x).max()
    _, e = math.frexp(mx)
    sh = 15 - e  # prescale: max|x| * 2^sh in [2^14, 2^15)
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
    return float(np.abs(r).max() / (mx * 2.0 ** sh))


def test_eight_components_leave_a_negligible_residual():
    rng = np.random.default_rng(0)
    worst = 0.0
    for trial in range(200):
        x = rng.standard_normal(16) * 2.0 ** int(rng.integers(-40, 40))
        if trial % 3 == 0:
            x[rng.integers(16)] *= 50.0  # an outlier channel
        if trial % 5 == 0:
            x[:8] = 0.0
        x = _bf16(x)
        if np.abs(x).max() == 0:
            continue
        worst = max(worst, split_residual(x))
    assert worst < 4e-9, worst


def test_exact_when_the_block_is_representable():
    # a block that is already 16 E2M1 codes times one E4M3 scale: the first
    # component takes it exactly
    x = _bf16(np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 6.0]) * 0.75)
    assert split_residual(x) == 0.0
