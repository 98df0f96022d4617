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
from _gpu import (_bits, check_decode_swiglu, check_within_tolerance, dev_bf16, dev_nvfp4,
                  sample_rows, swiglu_decode_reference)

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


# ---- decode: the down projection with the activation formed in its X split --------

@pytest.mark.parametrize("M,K,N", [(1, 1024, 256), (2, 3072, 1000), (4, 1024, 384),
                                   (16, 2048, 130), (1, 5120, 152 * 128 + 40)])
def test_decode_swiglu_every_element(M, K, N):
    lg = synth.Linear("dg", M, K, 1, 61, x_outlier_frac=0.01)
    lu = synth.Linear("du", M, K, 1, 62)
    ld = synth.Linear("dd", M, K, N, 63, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                      zero_block_p=0.01)
    gb, ub = lg.act_bf16(), lu.act_bf16()
    c, s, ts, _ = oracle.quantize(ld.weight_bf16())
    w = pkg.prepare_mma(dev_nvfp4(c, s, ts))
    assert pkg.imp_nvfp4_gemm_mma_swiglu_plan(M, N, K)[0] == 2
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = pkg.gemm_mma_swiglu(dev_bf16(gb), dev_bf16(ub), w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    y_ref, bound, extra = swiglu_decode_reference(gb, ub, c, s, ts, M)
    check_decode_swiglu(y.float().cpu().numpy(), y_ref, bound, extra, f"decode swiglu {M}x{K}x{N}")


@pytest.mark.parametrize("M", [1, 2, 8])
def test_decode_mlp_27b_sampled(M):
    """A 27B-class decode MLP: gate and up in one grouped call, then the down
    projection on silu(gate) * up; each output against the oracle on the
    inputs it read."""
    L = {l.name: l for l in synth.workload("decode_27b")}
    ws = {}
    for n in ("gate", "up", "down"):
        wb = L[n].weight_bf16()
        ws[n] = (wb, oracle.tensor_scale(wb)[1], pkg.prepare_mma(pkg.quantize(dev_bf16(wb))))
    x = np.concatenate([L["up"].act_bf16()] + [synth.Linear(f"r{i}", 1, 5120, 1, 70 + i).act_bf16()
                                               for i in range(M - 1)])
    g, u = pkg.gemm_grouped(dev_bf16(x), [ws["gate"][2], ws["up"][2]])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = pkg.gemm_mma_swiglu(g, u, ws["down"][2], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for t, n in ((g, "gate"), (u, "up")):
        rows = sample_rows(L[n].N, seed=M + len(n))
        wb, s_w, _ = ws[n]
        c, s = oracle.quantize_rows(wb[rows], s_w)
        y_ref, bound = oracle.reference_gemm(x, M, c, s, s_w)
        check_within_tolerance(t.float().cpu().numpy()[:, rows], y_ref, bound, f"27b {n}")
    rows = sample_rows(L["down"].N, seed=M + 9)
    wb, s_w, _ = ws["down"]
    c, s = oracle.quantize_rows(wb[rows], s_w)
    y_ref, bound, extra = swiglu_decode_reference(_bits(g), _bits(u), c, s, s_w, M)
    check_decode_swiglu(y.float().cpu().numpy()[:, rows], y_ref, bound, extra, "27b down(swiglu)")


def test_decode_swiglu_rejects():
    ld = synth.Linear("rj", 1, 1024, 256, 1)
    c, s, ts, _ = oracle.quantize(ld.weight_bf16())
    w = pkg.prepare_mma(dev_nvfp4(c, s, ts))
    g = dev_bf16(ld.act_bf16())
    with pytest.raises(pkg.ImpError):  # more rows than the decode path holds
        pkg.gemm_mma_swiglu(torch.cat([g] * 17), torch.cat([g] * 17), w)
    assert pkg.imp_nvfp4_gemm_mma_swiglu_plan(1, 256, 512) == (0, None)  # K below 1024
