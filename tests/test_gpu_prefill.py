"""Prefill path (M > 16) vs the oracle: X quantized on device (bit-exact to
the oracle's quantizer), block-scaled FP4 tensor-core GEMM within the
acceptance band on every checked element; the scale-atom layout checked
against its definition."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import check_within_tolerance, dev_bf16, dev_nvfp4, sample_rows

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def atom_layout(scales: np.ndarray, K: int) -> np.ndarray:
    """Row-major [rows][K/16] scale bytes -> the documented 512-byte atom layout
    (128 rows x 4 blocks per atom; rows padded to a multiple of 256)."""
    rows, KB = scales.shape
    rpad = (rows + 255) // 256 * 256
    out = np.zeros(rpad * KB, np.uint8)
    r = np.arange(rows)[:, None]
    kb = np.arange(KB)[None, :]
    off = ((r // 128) * (K // 64) + kb // 4) * 512 + 16 * (r % 32) + 4 * ((r // 32) % 4) + kb % 4
    out[off] = scales
    return out


def tile_layout(codes: np.ndarray, K: int) -> np.ndarray:
    """Row-major [rows][K/2] code bytes -> the documented 16 KB tile layout
    (128 rows x 128 bytes per tile, 16-byte unit u of row rr stored at unit
    u ^ (rr % 8); tiles along K (padded to 256), then down the rows (padded
    to 256))."""
    rows = codes.shape[0]
    rpad = (rows + 255) // 256 * 256
    nch = (K + 255) // 256
    src = np.zeros((rpad, nch * 128), np.uint8)
    src[:rows, : K // 2] = codes
    t = src.reshape(rpad // 128, 128, nch, 8, 16)       # [rb][rr][c][u][16]
    t = t.transpose(0, 2, 1, 3, 4).copy()                # [rb][c][rr][u][16]
    out = np.empty_like(t)
    rr = np.arange(128)
    for u in range(8):                                   # unit u goes to u ^ (rr % 8)
        out[:, :, rr, u ^ (rr % 8), :] = t[:, :, rr, u, :]
    return out.reshape(-1)


def test_prepare_mma_matches_layout_definition():
    rng = np.random.default_rng(0)
    for rows, K in [(1, 64), (130, 320), (300, 1024), (260, 768)]:
        sc = rng.integers(0, 0x7F, size=(rows, K // 16), dtype=np.uint8)
        cd = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
        t = dev_nvfp4(cd, sc, 1.0)
        p = pkg.prepare_mma(t)
        np.testing.assert_array_equal(p.scales.cpu().numpy(), atom_layout(sc, K))
        np.testing.assert_array_equal(p.codes.cpu().numpy(), tile_layout(cd, K))


def test_quantize_mma_equals_quantize_plus_layout():
    lin = synth.Linear("qm", 300, 1024, 1, 31, x_outlier_frac=0.01)
    xb = lin.act_bf16()
    q = pkg.quantize_mma(dev_bf16(xb))
    torch.cuda.synchronize()
    c, s, ts, _ = oracle.quantize(xb)
    np.testing.assert_array_equal(q.codes.cpu().numpy(), c)
    # compare the bytes of real rows (padding rows are not written)
    r = np.arange(300)[:, None]
    kb = np.arange(64)[None, :]
    off = ((r // 128) * 16 + kb // 4) * 512 + 16 * (r % 32) + 4 * ((r // 32) % 4) + kb % 4
    np.testing.assert_array_equal(q.scales.cpu().numpy()[off], s)
    assert np.float32(q.tensor_scale.item()) == np.float32(ts)


def run_prefill(lin, rows_check=None, cols_check=None, via="gemm"):
    xb = lin.act_bf16()
    wb = lin.weight_bf16()
    w = pkg.quantize(dev_bf16(wb))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if via == "gemm":
        y = pkg.gemm(dev_bf16(xb), w, dev_status=status)
    elif via == "gemm_mma":
        y = pkg.gemm_mma(dev_bf16(xb), pkg.prepare_mma(w), dev_status=status)
    else:  # "gemm_fp4" (whole tiles per CTA) or "gemm_fp4_sk" (stream-K)
        xq = pkg.quantize_mma(dev_bf16(xb), dev_status=status)
        y = pkg.gemm_fp4(xq, pkg.prepare_mma(w), dev_status=status,
                         stream_k=(via == "gemm_fp4_sk"))
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    y = y.float().cpu().numpy()
    rows = np.arange(lin.M) if rows_check is None else rows_check
    cols = np.arange(lin.N) if cols_check is None else cols_check
    _, s_w, _ = oracle.tensor_scale(wb)
    wc, wsc = oracle.quantize_rows(wb[cols], s_w)
    _, s_x, _ = oracle.tensor_scale(xb)
    y_ref, bound = oracle.reference_gemm(xb[rows], lin.M, wc, wsc, s_w, s_x=s_x)
    ratio = check_within_tolerance(y[np.ix_(rows, cols)], y_ref, bound, lin.name, tight=True)
    assert np.isfinite(y).all()
    return ratio


@pytest.mark.parametrize("M,K,N", [(128, 64, 256), (128, 256, 256), (256, 1024, 512),
                                   (128, 320, 256), (200, 320, 312), (17, 128, 40),
                                   (640, 5120, 768), (333, 2048, 1000),
                                   # a second N tile mostly past N; three N tiles of a
                                   # 128-row-block-aligned prepared weight; ragged rows
                                   (130, 512, 200), (256, 768, 576), (300, 4096, 1920),
                                   # more tiles than SMs, a partial last wave
                                   (1280, 256, 4096), (2048, 320, 2600)])
def test_small_shapes_every_element(M, K, N):
    lin = synth.Linear("pf", M, K, N, 77, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                       zero_block_p=0.01, x_outlier_frac=0.01)
    for via in ("gemm_fp4", "gemm_fp4_sk", "gemm", "gemm_mma"):
        run_prefill(lin, via=via)


@pytest.mark.parametrize("lin", synth.workload("prefill_27b"), ids=lambda l: f"{l.K}x{l.N}")
def test_full_size_sampled(lin):
    rows = np.arange(0, lin.M, 32)  # the 64-row sample m = 32 i
    cols = sample_rows(lin.N, seed=lin.K)
    run_prefill(lin, rows_check=rows, cols_check=cols)
    run_prefill(lin, rows_check=rows, cols_check=cols, via="gemm_mma")


@pytest.mark.parametrize("M,K,N", [(256, 1024, 512), (640, 5120, 768)])
def test_repeatable(M, K, N):
    # (640, 5120, 768): 15 tiles of 20 K stages over all SMs, so every tile
    # is summed from the partials of several CTAs
    lin = synth.Linear("rep", M, K, N, 5, w_dist=synth.DIST_STUDENT_T4)
    xb, wb = lin.act_bf16(), lin.weight_bf16()
    w = pkg.quantize(dev_bf16(wb))
    outs = [pkg.gemm(dev_bf16(xb), w).cpu() for _ in range(3)]
    xq, wm = pkg.quantize_mma(dev_bf16(xb)), pkg.prepare_mma(w)
    ws = torch.empty(pkg.imp_nvfp4_gemm_fp4_workspace_size(M, N, K), dtype=torch.uint8,
                     device="cuda")
    sk = [pkg.gemm_fp4(xq, wm, workspace=ws, stream_k=True).cpu() for _ in range(3)]
    fp4 = [pkg.gemm_fp4(xq, wm).cpu() for _ in range(3)]
    for runs in (outs, sk, fp4):
        for o in runs[1:]:
            assert torch.equal(runs[0].view(torch.int16), o.view(torch.int16))
    # whole tiles: the same GEMM whichever form the weight is in
    assert torch.equal(outs[0].view(torch.int16), fp4[0].view(torch.int16))


def test_back_to_back_calls_share_one_workspace():
    """Calls of imp_nvfp4_gemm_mma in a row on one stream and one workspace,
    each with its own X, nothing synchronised between them: X's quantizer,
    its encode pass and the GEMM of a call are chained by programmatic
    dependent launch, so each must wait for its predecessor before touching
    the shared X codes and scales.  Every result equals the same call made
    alone (the arithmetic is deterministic), and the first is checked
    against the oracle."""
    M, K, N = 640, 5120, 768
    lins = [synth.Linear(f"b2b{i}", M, K, N, 90 + i, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                         x_outlier_frac=0.01) for i in range(3)]
    wb = lins[0].weight_bf16()
    wm = pkg.prepare_mma(pkg.quantize(dev_bf16(wb)))
    xs = [dev_bf16(l.act_bf16()) for l in lins]
    ws = torch.empty(pkg.imp_nvfp4_gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in xs]
    for _ in range(2):
        for x, y in zip(xs, ys):
            pkg.gemm_mma(x, wm, y=y, dev_status=status, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for x, y in zip(xs, ys):
        alone = pkg.gemm_mma(x, wm, dev_status=status, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(alone.view(torch.int16), y.view(torch.int16))
    xb = lins[0].act_bf16()
    _, s_w, _ = oracle.tensor_scale(wb)
    cols = np.arange(0, N, 7)
    wc, wsc = oracle.quantize_rows(wb[cols], s_w)
    _, s_x, _ = oracle.tensor_scale(xb)
    rows = np.arange(0, M, 5)
    y_ref, bound = oracle.reference_gemm(xb[rows], M, wc, wsc, s_w, s_x=s_x)
    check_within_tolerance(ys[0].float().cpu().numpy()[np.ix_(rows, cols)], y_ref, bound,
                           "b2b", tight=True)
