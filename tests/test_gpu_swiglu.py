"""Prefill gate/up GEMM with the SwiGLU activation in its epilogue
(imp_nvfp4_gemm_swiglu) vs the oracle's reference_swiglu band on every
checked element; the folded amax of h; the encode-only quantizer fed with it
(bit-identical to the two-pass one); and the whole MLP chain into the down
projection."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import check_within_tolerance, dev_bf16, sample_rows

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def weights(M, K, N, seed):
    lg = synth.Linear(f"gate{seed}", M, K, N, seed, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                      zero_block_p=0.01, x_outlier_frac=0.01)
    lu = synth.Linear(f"up{seed}", M, K, N, seed + 100, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                      zero_block_p=0.01)
    return lg, lu


def run_swiglu(lg, lu):
    xb, gb, ub = lg.act_bf16(), lg.weight_bf16(), lu.weight_bf16()
    wg, wu = pkg.quantize(dev_bf16(gb)), pkg.quantize(dev_bf16(ub))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h, amax = pkg.gemm_swiglu(dev_bf16(xb), pkg.prepare_mma(wg), pkg.prepare_mma(wu), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return xb, gb, ub, h, amax


def check_h(xb, gb, ub, h, rows, cols, M):
    _, sg, _ = oracle.tensor_scale(gb)
    _, su, _ = oracle.tensor_scale(ub)
    gate = (*oracle.quantize_rows(gb[cols], sg), sg)
    up = (*oracle.quantize_rows(ub[cols], su), su)
    _, s_x, _ = oracle.tensor_scale(xb)
    h_ref, tol = oracle.reference_swiglu(xb[rows], M, gate, up, s_x=s_x)
    hg = h.float().cpu().numpy()[np.ix_(rows, cols)].astype(np.float64)
    err = np.abs(hg - h_ref)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{len(bad)} elements outside the band, first {bad[:4].tolist()}, "
                           f"err {err[tuple(bad[0])]:.3e} tol {tol[tuple(bad[0])]:.3e}")


@pytest.mark.parametrize("M,K,N", [(128, 256, 128), (200, 512, 300), (256, 1024, 384),
                                   (33, 320, 130), (640, 5120, 1000), (300, 2048, 2048)])
def test_swiglu_every_element(M, K, N):
    lg, lu = weights(M, K, N, 3)
    xb, gb, ub, h, amax = run_swiglu(lg, lu)
    check_h(xb, gb, ub, h, np.arange(M), np.arange(N), M)
    hb = h.contiguous().view(torch.int16).cpu().numpy().view(np.uint16) & 0x7FFF
    assert int(amax.item()) == int(hb.max())


def test_swiglu_full_size_sampled_and_down_chain():
    """The 27B-class MLP at M = 2048: gate/up 5120 -> 17408 with SwiGLU, h
    quantized from the folded amax, down 17408 -> 5120 on it."""
    lg = [l for l in synth.workload("prefill_27b") if l.K == 5120][0]
    lu = synth.Linear("up_27b", lg.M, lg.K, lg.N, 41, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                      zero_block_p=0.001)
    xb, gb, ub, h, amax = run_swiglu(lg, lu)
    rows = np.arange(0, lg.M, 32)
    cols = sample_rows(lg.N, seed=5)
    check_h(xb, gb, ub, h, rows, cols, lg.M)
    # encode-only quantizer from the folded amax == the two-pass quantizer
    hq = pkg.quantize_mma_amax(h.contiguous(), amax)
    hq2 = pkg.quantize_mma(h.contiguous())
    torch.cuda.synchronize()
    assert torch.equal(hq.codes, hq2.codes) and torch.equal(hq.scales, hq2.scales)
    assert torch.equal(hq.tensor_scale, hq2.tensor_scale)
    # down projection on it, checked against the oracle on h as computed
    ld = [l for l in synth.workload("prefill_27b") if l.K == 17408][0]
    db = ld.weight_bf16()
    wd = pkg.prepare_mma(pkg.quantize(dev_bf16(db)))
    y = pkg.gemm_fp4(hq, wd).float().cpu().numpy()
    hbits = h.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    _, s_h, _ = oracle.tensor_scale(hbits)
    _, s_d, _ = oracle.tensor_scale(db)
    dcols = sample_rows(ld.N, seed=6)
    dc, ds = oracle.quantize_rows(db[dcols], s_d)
    y_ref, bound = oracle.reference_gemm(hbits[rows], ld.M, dc, ds, s_d, s_x=s_h)
    check_within_tolerance(y[np.ix_(rows, dcols)], y_ref, bound, "down after SwiGLU")


def test_swiglu_repeatable_and_rejects_decode_sizes():
    lg, lu = weights(256, 1024, 512, 9)
    outs = [run_swiglu(lg, lu)[3].clone() for _ in range(2)]
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    w = pkg.prepare_mma(pkg.quantize(dev_bf16(lg.weight_bf16())))
    with pytest.raises(pkg.ImpError):
        pkg.gemm_swiglu(dev_bf16(synth.Linear("d", 16, 1024, 512, 1).act_bf16()), w, w)
