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


def _near_boundary_tensor(seed, n_blocks=512):
    """Rows of 16-element blocks whose elements x make x / d land within
    2^-20 (relative) of an E2M1 rounding boundary without being on it, plus
    exact ties -- the cases a quotient computed as x * (1/d) could round
    differently from the division.  Found by search on the CPU: the tensor
    scale is fixed by one element g; each block's amax a sets d."""
    rng = np.random.default_rng(seed)
    g = np.float32(1992.0)  # exact in bf16; s = g / 2688 has a full 24-bit mantissa
    s = np.float32(g / np.float32(2688.0))
    bounds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    blocks = []
    while len(blocks) < n_blocks:
        a = np.float32(torch.tensor(float(rng.uniform(0.05, 1.9) * float(g) / 6)).bfloat16().float().item())
        u = np.float32(np.float32(a / np.float32(6.0)) / s)
        sb = torch.tensor([float(u)]).to(torch.float8_e4m3fn).float().item()
        d = np.float32(np.float32(sb) * s)
        xs = []
        for t in bounds:
            target = t * float(d)
            b = torch.tensor([target]).bfloat16()
            for cand in (b.float().item(), torch.nextafter(b.float(), torch.tensor([0.0])).bfloat16().float().item(),
                         torch.nextafter(b.float(), torch.tensor([1e30])).bfloat16().float().item()):
                rel = abs(cand / float(d) - t) / t
                if rel < 2.0 ** -20 and cand <= float(a):
                    xs.append(cand)
        if xs:
            row = [float(a)] + xs[:15]
            row += [0.0] * (16 - len(row))
            blocks.append(row)
    x = np.array(blocks, np.float32).reshape(-1, 32 * 16)[: n_blocks // 32]
    x[0, 1] = g
    x *= np.where(rng.random(x.shape) < 0.5, -1.0, 1.0).astype(np.float32)
    return torch.from_numpy(x).bfloat16().view(torch.int16).numpy().view(np.uint16)


def test_quotients_next_to_rounding_boundaries():
    bits = _near_boundary_tensor(0)
    got = gpu_quantize(bits)
    assert got[3] == 0
    assert_same(got, oracle.quantize(bits), "near-boundary quotients")
