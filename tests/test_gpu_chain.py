"""Decode chain (imp_nvfp4_gemm_chain): several decode calls in one
persistent launch, each link's X given or the previous link's first output.
Every link's output is checked against the oracle on the X it actually read
(for a chained link: the previous link's bf16 output as the GPU wrote it):
every element for small chains (whole-tile and stream-K links, ragged N,
groups, M = 1 and 2), sampled rows for the 27B-class decode step; the
grouped-call fallback; bitwise repeatability and CUDA-graph replay; argument
checks."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import (_bits, check_decode_swiglu, check_within_tolerance, dev_bf16, dev_nvfp4,
                  num_sms, sample_rows, swiglu_decode_reference)

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def lin(name, M, K, N, seed):
    return synth.Linear(name, M, K, N, seed, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                        zero_block_p=0.01, x_outlier_frac=0.01)


def prepared(l):
    c, s, ts, _ = oracle.quantize(l.weight_bf16())
    return (c, s, ts), pkg.prepare_mma(dev_nvfp4(c, s, ts))


def bits(y):
    return y.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_chain(links, status=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    ys = pkg.gemm_chain(links, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ys


# (M, [(K, [N of each group], X)]) with X "x" (its own), "prev" (the previous
# link's first output) or "same" (the previous link's X: with whole tiles in
# both, the kernel keeps the split X); a link of >= 3/4 as many 128-row tiles
# as SMs runs whole tiles, fewer run stream-K
def chains():
    big = 128 * ((num_sms() * 3 + 3) // 4 + 5)  # whole tiles
    return [
        (1, [(1024, [2048], "x"), (2048, [1024], "prev"), (1024, [300], "prev")]),
        (2, [(1536, [1024, 1024], "x"), (1024, [1536], "prev"), (1536, [130, 7], "prev")]),
        (1, [(1024, [big], "x"), (1024, [1280], "x"), (1280, [1024], "prev"),
             (1024, [big + 72], "prev")]),
        (2, [(2048, [1000, 24, 256], "x"), (1024, [2048], "x")]),
        (2, [(1024, [big], "x"), (1024, [big + 200, 56], "same"), (1024, [1024], "same"),
             (1024, [big], "same")]),
    ]


@pytest.mark.parametrize("case", range(5))
def test_chain_every_element(case):
    M, spec = chains()[case]
    ref, links, xs = [], [], []
    for c, (K, Ns, src) in enumerate(spec):
        ls = [lin(f"c{case}l{c}g{i}", M, K, N, 100 * case + 10 * c + i) for i, N in enumerate(Ns)]
        r, d = zip(*(prepared(l) for l in ls))
        ref.append(r)
        x = None if src == "prev" else xs[-1] if src == "same" else ls[0].act_bf16()
        xs.append(x)
        links.append((list(d), None if x is None else
                      links[-1][1] if src == "same" else dev_bf16(x)))
    assert pkg.imp_nvfp4_gemm_chain_plan(M, pkg.ChainLinks(
        [([pkg.ImpNvfp4Group(w.c_struct(), 0, 0) for w in d], x is not None and 16 or None, 0)
         for d, x in links])) == 1
    ys = run_chain(links)
    for c in range(len(spec)):
        x = xs[c] if xs[c] is not None else bits(ys[c - 1][0])
        for y, (cc, s, ts) in zip(ys[c], ref[c]):
            y_ref, bound = oracle.reference_gemm(x, M, cc, s, ts)
            check_within_tolerance(y.float().cpu().numpy(), y_ref, bound, f"chain {case} link {c}")


def test_chain_27b_decode_step_sampled():
    """The 27B-class decode step as one chain: up and gate read x, down reads
    gate's output, the LM head reads down's output."""
    L = {l.name: l for l in synth.workload("decode_27b")}
    names = ["up", "gate", "down", "lm_head"]
    ws, refs = {}, {}
    for n in names:
        wb = L[n].weight_bf16()
        ws[n] = pkg.prepare_mma(pkg.quantize(dev_bf16(wb)))
        refs[n] = (wb, oracle.tensor_scale(wb)[1])
    x = L["up"].act_bf16()
    xd = dev_bf16(x)
    links = [([ws["up"]], xd), ([ws["gate"]], xd), ([ws["down"]], None), ([ws["lm_head"]], None)]
    ys = run_chain(links)
    xin = {"up": x, "gate": x, "down": bits(ys[1][0]), "lm_head": bits(ys[2][0])}
    for c, n in enumerate(names):
        wb, ts = refs[n]
        rows = sample_rows(L[n].N, seed=c + 7)
        cc, s = oracle.quantize_rows(wb[rows], ts)
        y_ref, bound = oracle.reference_gemm(xin[n], 1, cc, s, ts)
        check_within_tolerance(ys[c][0].float().cpu().numpy()[:, rows], y_ref, bound, f"27b {n}")


def test_chain_repeatable_and_graph_replay():
    M, spec = chains()[2]
    links = []
    for c, (K, Ns, src) in enumerate(spec):
        d = [prepared(lin(f"r{c}g{i}", M, K, N, 7 * c + i))[1] for i, N in enumerate(Ns)]
        links.append((d, None if src == "prev" else
                      dev_bf16(lin(f"x{c}", M, K, 1, 3 + c).act_bf16())))
    a = [[y.clone() for y in yl] for yl in run_chain(links)]
    b = run_chain(links)
    for ya, yb in zip(a, b):
        for u, v in zip(ya, yb):
            assert torch.equal(u.view(torch.int16), v.view(torch.int16))
    # captured once, replayed on a new X (copied into the captured input)
    ys = [[torch.empty_like(y) for y in yl] for yl in a]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_bytes = pkg.imp_nvfp4_gemm_chain_workspace_size(M, pkg.ChainLinks(
        [([pkg.ImpNvfp4Group(w.c_struct(), 0, 0) for w in d], None if x is None else 16, 0)
         for d, x in links]))
    work = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pkg.gemm_chain(links, ys=ys, dev_status=status, workspace=work, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkg.gemm_chain(links, ys=ys, dev_status=status, workspace=work)
    x0 = links[0][1]
    for seed in (11, 12):
        x0.copy_(dev_bf16(lin("new", M, x0.shape[1], 1, seed).act_bf16()))
        g.replay()
        torch.cuda.synchronize()
        e = run_chain(links)
        for ya, yb in zip(ys, e):
            for u, v in zip(ya, yb):
                assert torch.equal(u.view(torch.int16), v.view(torch.int16))
    assert int(status.item()) == 0


def test_chain_fallback_for_more_rows():
    """M = 4: no persistent plan; the links run as grouped calls in order."""
    M = 4
    l0, l1 = lin("f0", M, 1024, 1024, 1), lin("f1", M, 1024, 512, 2)
    (r0, d0), (r1, d1) = prepared(l0), prepared(l1)
    links = [([d0], dev_bf16(l0.act_bf16())), ([d1], None)]
    cl = pkg.ChainLinks([([pkg.ImpNvfp4Group(d0.c_struct(), 0, 0)], 16, 0),
                         ([pkg.ImpNvfp4Group(d1.c_struct(), 0, 0)], None, 0)])
    assert pkg.imp_nvfp4_gemm_chain_plan(M, cl) == 0
    ys = run_chain(links)
    y_ref, bound = oracle.reference_gemm(l0.act_bf16(), M, *r0)
    check_within_tolerance(ys[0][0].float().cpu().numpy(), y_ref, bound, "fallback link 0")
    y_ref, bound = oracle.reference_gemm(bits(ys[0][0]), M, *r1)
    check_within_tolerance(ys[1][0].float().cpu().numpy(), y_ref, bound, "fallback link 1")


def test_chain_rejects():
    M = 1
    d0 = prepared(lin("a", M, 1024, 1024, 1))[1]
    d1 = prepared(lin("b", M, 2048, 512, 2))[1]
    x = dev_bf16(lin("a", M, 1024, 1024, 1).act_bf16())
    y = torch.empty((1, 1024), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    lone = pkg.ChainLinks([([pkg.ImpNvfp4Group(d0.c_struct(), y.data_ptr(), 1024)], None, 0)])
    assert pkg.imp_nvfp4_gemm_chain(M, lone, None, ws.data_ptr(), ws.numel(), None) == \
        pkg.IMP_ERR_INVALID_ARG  # link 0 with no X
    with pytest.raises(pkg.ImpError):  # chained X of the wrong length (1024 outputs, K 2048)
        pkg.gemm_chain([([d0], x), ([d1], None)])
    with pytest.raises(pkg.ImpError):  # two links writing one buffer
        pkg.gemm_chain([([d0], x), ([d0], x)], ys=[[y], [y]])
    with pytest.raises(pkg.ImpError):  # an output over an explicit X
        pkg.gemm_chain([([d0], x)], ys=[[x]])


@pytest.mark.parametrize("case", [0, 4])
def test_chain_back_to_back_launches(case):
    """Ten launches queued back to back on one workspace (each may start
    while the previous one drains): no wait gives up and every launch writes
    the same bits.  Case 4 keeps the split X between calls, whose barrier
    phases must stay in step from launch to launch."""
    M, spec = chains()[case]
    links, xs = [], []
    for c, (K, Ns, src) in enumerate(spec):
        d = [prepared(lin(f"b{case}{c}g{i}", M, K, N, 31 * c + i))[1] for i, N in enumerate(Ns)]
        x = None if src == "prev" else xs[-1] if src == "same" else \
            dev_bf16(lin(f"bx{c}", M, K, 1, 5 + c).act_bf16())
        xs.append(x)
        links.append((d, x))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = [[y.clone() for y in yl] for yl in run_chain(links)]
    ys = [[torch.empty_like(y) for y in yl] for yl in ref]
    ws_bytes = pkg.imp_nvfp4_gemm_chain_workspace_size(M, pkg.ChainLinks(
        [([pkg.ImpNvfp4Group(w.c_struct(), 0, 0) for w in d], None if x is None else 16, 0)
         for d, x in links]))
    work = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for _ in range(10):
        pkg.gemm_chain(links, ys=ys, dev_status=status, workspace=work)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for ya, yb in zip(ref, ys):
        for u, v in zip(ya, yb):
            assert torch.equal(u.view(torch.int16), v.view(torch.int16))


@pytest.mark.parametrize("M", [1, 2, 4])
def test_chain_decode_mlp_swiglu(M):
    """A decode MLP as one chain: gate and up grouped on x, down on
    silu(gate) * up (x_swiglu), then a projection of down's output.  M = 4
    runs the links one call after another (the same results are required)."""
    K, F = 1024, 2048
    lg, lu = lin("mg", M, K, F, 81), lin("mu", M, K, F, 82)
    ld, lo = lin("md", M, F, K, 83), lin("mo", M, K, 300, 84)
    (rg, dg), (ru, du), (rd, dd), (ro, do) = (prepared(l) for l in (lg, lu, ld, lo))
    x = lg.act_bf16()
    links = [([dg, du], dev_bf16(x)), ([dd], "swiglu"), ([do], None)]
    cl = pkg.ChainLinks([([pkg.ImpNvfp4Group(w.c_struct(), 0, 0) for w in ws],
                          None if isinstance(xx, str) or xx is None else 16, 0,
                          1 if xx == "swiglu" else 0) for ws, xx in links])
    assert pkg.imp_nvfp4_gemm_chain_plan(M, cl) == (1 if M <= 2 else 0)
    ys = run_chain(links)
    for y, r in zip(ys[0], (rg, ru)):
        y_ref, bound = oracle.reference_gemm(x, M, *r)
        check_within_tolerance(y.float().cpu().numpy(), y_ref, bound, "gate/up")
    y_ref, bound, extra = swiglu_decode_reference(_bits(ys[0][0]), _bits(ys[0][1]), *rd, M)
    check_decode_swiglu(ys[1][0].float().cpu().numpy(), y_ref, bound, extra, "down on silu(g) u")
    y_ref, bound = oracle.reference_gemm(_bits(ys[1][0]), M, *ro)
    check_within_tolerance(ys[2][0].float().cpu().numpy(), y_ref, bound, "after down")
