"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import oracle


def dev_bf16(bits: np.ndarray, ld: int | None = None) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bf16 tensor (optionally with row stride ld)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    if ld is not None and ld != bits.shape[1]:
        big = torch.zeros((bits.shape[0], ld), dtype=torch.bfloat16)
        big[:, : bits.shape[1]] = t
        return big.cuda()[:, : bits.shape[1]]
    return t.cuda()


def dev_nvfp4(codes: np.ndarray, scales: np.ndarray, s: float):
    import nvfp4_weight_quantized_02_gb300 as pkg
    return pkg.NVFP4Tensor(torch.from_numpy(np.ascontiguousarray(codes)).cuda(),
                           torch.from_numpy(np.ascontiguousarray(scales)).cuda(),
                           torch.tensor([s], dtype=torch.float32).cuda())


def num_sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def sample_rows(N: int, seed: int, n_random: int = 128) -> np.ndarray:
    """Rows to check at full size: both ends, rows at the CTA boundaries of a
    one-CTA-per-SM grid, and a seeded random sample."""
    G = min(num_sms(), N)
    rows = set(range(min(N, 48))) | set(range(max(0, N - 48), N))
    for c in range(0, G + 1, max(1, G // 16)):
        b = N * c // G
        rows |= {max(0, b - 1), min(N - 1, b)}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, N, n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def check_within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what: str,
                           tight: bool = True):
    """The acceptance band (oracle.tolerance) on every element and, with
    tight=True, the stricter band of exact products + fp32 sums."""
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    if tight:
        ttol = oracle.tight_tolerance(bound, y_ref)
        tbad = np.argwhere(~(err <= ttol))
        assert tbad.size == 0, (f"{what}: {len(tbad)} elements outside the tight band, first "
                                f"{tbad[:4].tolist()}, err {err[tuple(tbad[0])]:.3e} tight tol "
                                f"{ttol[tuple(tbad[0])]:.3e}")
    tol = oracle.tolerance(bound, y_ref)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{what}: {len(bad)} elements outside tolerance, first {bad[:4].tolist()}, "
                           f"err {err[tuple(bad[0])]:.3e} tol {tol[tuple(bad[0])]:.3e}")
    return float((err / tol).max()) if err.size else 0.0


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def swiglu_decode_reference(gb, ub, codes, scales, ts, M):
    """y = bf16(silu(g) * u) W^T from the oracle, and the extra tolerance for
    elements of h whose fp64 value sits within the kernel's fp32 evaluation
    error of a bf16 rounding boundary (there the kernel may round to the
    neighbouring bf16: one ulp of h times |w|)."""
    g, u = oracle.bf16_to_f64(gb), oracle.bf16_to_f64(ub)
    h = oracle.silu(g) * u
    hb = _bits(torch.from_numpy(h).to(torch.float32).to(torch.bfloat16))
    hq = oracle.bf16_to_f64(hb)
    e = np.floor(np.log2(np.maximum(np.abs(h), 1e-300)))
    ulp = np.exp2(e - 7)
    mid = np.abs(np.abs(h) - (np.abs(hq) + 0.5 * ulp * np.sign(np.abs(h) - np.abs(hq))))
    near = (mid <= 2.0 ** -16 * np.abs(h)) | (np.abs(h) < 2.0 ** -120)
    y_ref, bound = oracle.reference_gemm(hb, M, codes, scales, ts)
    wd = np.abs(oracle.dequant(codes, scales, ts))
    extra = (near * ulp) @ wd.T
    return y_ref, bound, extra


def check_decode_swiglu(y, y_ref, bound, extra, what):
    err = np.abs(y.astype(np.float64) - y_ref)
    tol = oracle.tight_tolerance(bound, y_ref) + extra
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{what}: {len(bad)} outside, first {bad[:4].tolist()}, "
                           f"err {err[tuple(bad[0])]:.3e} tol {tol[tuple(bad[0])]:.3e}")
