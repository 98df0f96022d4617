"""Grouped decode GEMV (imp_nvfp4_gemm_grouped) vs the oracle: each weight's
output within the band on every element (small layers) or sampled columns
(27B-class gate/up), ragged groups, the per-group fallback for more rows of
X, bitwise repeatability, and a decode layer captured once as a CUDA graph
and replayed on new inputs (bitwise equal to the eager calls)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import check_within_tolerance, dev_bf16, dev_nvfp4, sample_rows

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def layer(name):
    return {l.name: l for l in synth.workload(name)}


def prepared(lin):
    c, s, ts, _ = oracle.quantize(lin.weight_bf16())
    return (c, s, ts), pkg.prepare_mma(dev_nvfp4(c, s, ts))


def run_grouped(x_bits, ws, status=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    ys = pkg.gemm_grouped(dev_bf16(x_bits), ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return [y.float().cpu().numpy() for y in ys]


@pytest.mark.parametrize("names", [("q", "k", "v"), ("gate", "up")])
def test_0p6b_groups_every_element(names):
    L = layer("decode_0p6b")
    lins = [L[n] for n in names]
    K = lins[0].K
    assert pkg.imp_nvfp4_gemm_grouped_plan(1, K, [l.N for l in lins]) == (1, "gemv_f4r_kernel")
    ref, dev = zip(*(prepared(l) for l in lins))
    x = lins[0].act_bf16()
    for y, (c, s, ts), l in zip(run_grouped(x, list(dev)), ref, lins):
        y_ref, bound = oracle.reference_gemm(x, 1, c, s, ts)
        check_within_tolerance(y, y_ref, bound, f"grouped {l.name}")


@pytest.mark.parametrize("M,K,Ns", [(1, 1024, [100, 28, 1]), (2, 1024, [130, 256, 7, 300]),
                                    (1, 2048, [1000, 24]), (2, 3072, [384]),
                                    # per-group fallback: more rows of X than one split holds
                                    (3, 1024, [200, 129]), (16, 1024, [128, 300])])
def test_ragged_groups_every_element(M, K, Ns):
    lins = [synth.Linear(f"g{i}", M, K, N, 50 + i, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                         zero_block_p=0.01, x_outlier_frac=0.01) for i, N in enumerate(Ns)]
    ref, dev = zip(*(prepared(l) for l in lins))
    x = lins[0].act_bf16()
    for y, (c, s, ts), l in zip(run_grouped(x, list(dev)), ref, lins):
        y_ref, bound = oracle.reference_gemm(x, M, c, s, ts)
        check_within_tolerance(y, y_ref, bound, f"ragged {l.name}")


@pytest.mark.parametrize("M", [1, 2])
def test_27b_gate_up_sampled(M):
    L = layer("decode_27b")
    lins = [L["gate"], L["up"]]
    K = lins[0].K
    assert pkg.imp_nvfp4_gemm_grouped_plan(M, K, [l.N for l in lins])[0] == 2
    ws, refs = [], []
    for l in lins:
        wb = l.weight_bf16()
        w = pkg.quantize(dev_bf16(wb))
        ws.append(pkg.prepare_mma(w))
        refs.append((wb, oracle.tensor_scale(wb)[1]))
    x = np.concatenate([lins[0].act_bf16()] * M) if M > 1 else lins[0].act_bf16()
    if M > 1:  # a second, different row
        x[1] = synth.Linear("row2", 1, K, 1, 99).act_bf16()[0]
    for y, (wb, ts), l in zip(run_grouped(x, ws), refs, lins):
        rows = sample_rows(l.N, seed=l.N + M)
        c, s = oracle.quantize_rows(wb[rows], ts)
        y_ref, bound = oracle.reference_gemm(x, M, c, s, ts)
        check_within_tolerance(y[:, rows], y_ref, bound, f"27b grouped {l.name}")


def test_grouped_repeatable():
    L = layer("decode_0p6b")
    lins = [L["q"], L["k"], L["v"]]
    dev = [prepared(l)[1] for l in lins]
    x = dev_bf16(lins[0].act_bf16())
    runs = [[y.clone() for y in pkg.gemm_grouped(x, dev)] for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layer_graph_replay_matches_eager():
    """A 0.6B-class decode layer (q/k/v grouped, o, gate/up grouped, down: 4
    kernels) captured once and replayed on new inputs."""
    L = layer("decode_0p6b")
    dev = {n: prepared(L[n])[1] for n in L}
    dev_stream = torch.cuda.Stream()
    x_in = torch.empty((1, 1024), dtype=torch.bfloat16, device="cuda")
    o_in = torch.empty((1, 2048), dtype=torch.bfloat16, device="cuda")
    d_in = torch.empty((1, 3072), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsz = max(pkg.imp_nvfp4_gemm_grouped_workspace_size(1, 1024, [2048, 1024, 1024]),
              pkg.imp_nvfp4_gemm_grouped_workspace_size(1, 1024, [3072, 3072]),
              pkg.imp_nvfp4_gemm_workspace_size(1, 1024, 2048),
              pkg.imp_nvfp4_gemm_workspace_size(1, 1024, 3072))
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    outs = {n: torch.empty((1, L[n].N), dtype=torch.bfloat16, device="cuda") for n in L}

    def step(stream):
        pkg.gemm_grouped(x_in, [dev["q"], dev["k"], dev["v"]],
                         ys=[outs["q"], outs["k"], outs["v"]], dev_status=status, stream=stream,
                         workspace=ws)
        pkg.gemm_mma(o_in, dev["o"], y=outs["o"], dev_status=status, stream=stream, workspace=ws)
        pkg.gemm_grouped(x_in, [dev["gate"], dev["up"]], ys=[outs["gate"], outs["up"]],
                         dev_status=status, stream=stream, workspace=ws)
        pkg.gemm_mma(d_in, dev["down"], y=outs["down"], dev_status=status, stream=stream,
                     workspace=ws)

    def inputs(seed):
        return [dev_bf16(synth.Linear(f"in{seed}_{K}", 1, K, 1, seed).act_bf16())
                for K in (1024, 2048, 3072)]

    # eager results for two input sets
    eager = []
    for seed in (11, 12):
        a, b, c = inputs(seed)
        x_in.copy_(a), o_in.copy_(b), d_in.copy_(c)
        step(torch.cuda.current_stream())
        torch.cuda.synchronize()
        eager.append({n: outs[n].clone() for n in outs})
    # capture once (after a warm-up call on the capture stream), replay on each input set
    dev_stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(dev_stream):
        step(dev_stream)
    torch.cuda.current_stream().wait_stream(dev_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=dev_stream):
        step(dev_stream)
    for seed, ref in zip((11, 12), eager):
        a, b, c = inputs(seed)
        x_in.copy_(a), o_in.copy_(b), d_in.copy_(c)
        for n in outs:
            outs[n].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for n in outs:
            assert torch.equal(outs[n].view(torch.int16), ref[n].view(torch.int16)), n


def test_graph_replay_split_tiles():
    """Replays of a captured call whose tiles are split between CTAs (the
    per-tile counters are left at zero by each launch, so a replay of the
    same launch parameters counts afresh)."""
    lin = synth.Linear("sk", 4, 5120, 5120, 21, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02)
    w = prepared(lin)[1]
    x_in = dev_bf16(lin.act_bf16())
    y = torch.empty((4, 5120), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(pkg.imp_nvfp4_gemm_workspace_size(4, 5120, 5120), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkg.gemm_mma(x_in, w, y=y, stream=s, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkg.gemm_mma(x_in, w, y=y, stream=s, workspace=ws)
    for _ in range(3):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
