"""GPU quantizer vs the oracle: codes, scale bytes and tensor scale must be
bit-exact (memcmp), on the hand-worked blocks, every workload tensor (full
size; the largest checked on sampled rows against the oracle's whole-tensor
scale) and edge shapes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _golden import all_cases
from _gpu import dev_bf16, sample_rows

pkg = pytest.importorskip("nvfp4_weight_quantized_02_gb300")
pytestmark = pytest.mark.gpu


def gpu_quantize(bits, ld=None):
    x = dev_bf16(bits, ld)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = pkg.quantize(x, dev_status=status)
    torch.cuda.synchronize()
    return (q.codes.cpu().numpy(), q.scales.cpu().numpy(), float(q.tensor_scale.item()),
            int(status.item()))


def assert_same(gpu, ref, what):
    gc, gs, gts = gpu[:3]
    rc, rs, rts = ref[:3]
    assert np.float32(gts) == np.float32(rts), f"{what}: tensor scale {gts!r} vs {rts!r}"
    bad_s = np.argwhere(gs != rs)
    assert bad_s.size == 0, f"{what}: scale bytes differ at {bad_s[:4].tolist()}"
    bad_c = np.argwhere(gc != rc)
    assert bad_c.size == 0, f"{what}: code bytes differ at {bad_c[:4].tolist()}"


@pytest.mark.parametrize("case", all_cases(), ids=lambda c: c["name"])
def test_golden_blocks(case):
    g = gpu_quantize(case["X"])
    assert g[3] == 0
    assert_same(g, (case["codes_arr"], case["scales_arr"], case["tensor_scale"]), case["name"])


SMALL = [(w, l) for w in ["single_1k", "decode_0p6b"] for l in synth.workload(w)]


@pytest.mark.parametrize("lin", [l for _, l in SMALL], ids=lambda l: f"{l.name}_{l.K}x{l.N}")
def test_workload_weights_and_activations_exact(lin):
    for bits in (lin.weight_bf16(), lin.act_bf16()):
        g = gpu_quantize(bits)
        c, s, ts, _ = oracle.quantize(bits)
        assert_same(g, (c, s, ts), lin.name)


BIG = synth.workload("decode_27b") + synth.workload("prefill_27b")[:1]


@pytest.mark.parametrize("lin", BIG, ids=lambda l: f"{l.name}_M{l.M}_{l.K}x{l.N}")
def test_full_size_weights_sampled(lin):
    bits = lin.weight_bf16()
    g = gpu_quantize(bits)
    _, ts, bad = oracle.tensor_scale(bits)
    assert not bad and np.float32(g[2]) == np.float32(ts)
    rows = sample_rows(lin.N, seed=lin.N)
    c, s = oracle.quantize_rows(bits[rows], ts)
    assert_same((g[0][rows], g[1][rows], g[2]), (c, s, ts), lin.name)


def test_prefill_activation_full_size_sampled():
    lin = synth.workload("prefill_27b")[1]  # X 2048 x 17408 with outlier channels
    bits = lin.act_bf16()
    g = gpu_quantize(bits)
    _, ts, _ = oracle.tensor_scale(bits)
    rows = np.arange(0, lin.M, 32)
    c, s = oracle.quantize_rows(bits[rows], ts)
    assert_same((g[0][rows], g[1][rows], g[2]), (c, s, ts), "prefill X")


@pytest.mark.parametrize("rows,K,ld", [(1, 16, 16), (3, 48, 56), (7, 80, 80), (1000, 1040, 1048),
                                       (33, 4096, 4096), (2, 17408, 17416)])
def test_edge_shapes(rows, K, ld):
    lin = synth.Linear("edge", 1, K, rows, 99, w_dist=synth.DIST_STUDENT_T4, w_scale=0.3,
                       zero_block_p=0.05)
    bits = lin.weight_bf16()
    g = gpu_quantize(bits, ld)
    c, s, ts, _ = oracle.quantize(bits)
    assert_same(g, (c, s, ts), f"{rows}x{K} ld {ld}")


def test_random_bit_patterns_exact():
    # Every finite bf16 pattern class: subnormals, huge values, both signs, zeros.
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=(512, 256), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] = 0x3F80  # drop Inf/NaN
    for scale_row in (None, 7):
        b = bits.copy()
        if scale_row is not None:
            b[scale_row] = np.where(rng.random(256) < 0.5, 0x0001, 0x8000)  # tiny subnormals, -0
        g = gpu_quantize(b)
        c, s, ts, _ = oracle.quantize(b)
        assert_same(g, (c, s, ts), "random patterns")
    # a tensor whose magnitudes are all bf16 subnormals
    sub = rng.integers(0, 0x80, size=(64, 64), dtype=np.uint16) | (rng.integers(0, 2, (64, 64)).astype(np.uint16) << 15)
    g = gpu_quantize(sub)
    assert_same(g, oracle.quantize(sub)[:3], "subnormal tensor")


def test_nonfinite_input_sets_status():
    bits = synth.workload("single_1k")[0].weight_bf16(0, 64)
    bits[5, 7] = 0x7FC0
    assert gpu_quantize(bits)[3] & pkg.IMP_DEV_NONFINITE_INPUT
    bits[5, 7] = 0xFF80
    assert gpu_quantize(bits)[3] & pkg.IMP_DEV_NONFINITE_INPUT


def test_zero_tensor_and_empty():
    g = gpu_quantize(np.zeros((5, 64), np.uint16))
    assert g[2] == 0.0 and not g[0].any() and not g[1].any()
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q = pkg.quantize(x)
    torch.cuda.synchronize()
    assert q.tensor_scale.item() == 0.0


def test_repeatable():
    bits = synth.workload("decode_0p6b")[6].weight_bf16()
    a, b = gpu_quantize(bits), gpu_quantize(bits)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]
