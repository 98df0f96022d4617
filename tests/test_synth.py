"""The seeded input generator: determinism, row-subset regeneration and the
distributions each workload recipe states."""
import numpy as np

import synth


def _f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def test_rows_are_independent_of_slicing():
    lin = synth.workload("decode_27b")[2]
    full = lin.weight_bf16(0, 64)
    part = lin.weight_bf16(17, 5)
    np.testing.assert_array_equal(full[17:22], part)


def test_student_t_weight_recipe():
    lin = synth.workload("decode_27b")[0]
    w = _f32(lin.weight_bf16(0, 4096))
    assert abs(w.std() - 0.02) < 0.002
    blocks = w.reshape(4096, -1, 16)
    zero = np.all(blocks == 0, axis=2).mean()
    assert 0.0006 < zero < 0.0014
    # heavy tails: kurtosis of t(4) is infinite; the sample's is well above 3
    k = ((w - w.mean()) ** 4).mean() / w.var() ** 2
    assert k > 6


def test_outlier_channels():
    lin = synth.workload("prefill_27b")[1]
    mask = lin.outlier_mask()
    assert mask.sum() == round(0.01 * lin.K)
    x = _f32(lin.act_bf16(0, 256))
    ratio = np.abs(x[:, mask == 1]).mean() / np.abs(x[:, mask == 0]).mean()
    assert 15 < ratio < 25


def test_gaussian_recipes_and_shapes():
    lins = synth.workload("decode_0p6b")
    assert [(l.K, l.N) for l in lins] == [(1024, 2048), (1024, 1024), (1024, 1024), (2048, 1024),
                                          (1024, 3072), (1024, 3072), (3072, 1024)]
    w = _f32(lins[0].weight_bf16(0, 512))
    assert abs(w.std() - 0.02) < 0.001 and abs(w.mean()) < 0.001
    x = _f32(lins[0].act_bf16())
    assert x.shape == (1, 1024) and 0.9 < x.std() < 1.1
    assert sum(l.weight_bytes for l in lins) == 8847360 + 7 * 4


def test_workload_table():
    assert [l.M for l in synth.workload("skinny_27b")] == [2, 2, 4, 4, 8, 8, 16, 16]
    p = synth.workload("prefill_27b")
    assert [(l.M, l.K, l.N) for l in p] == [(2048, 5120, 17408), (2048, 17408, 5120)]
    assert synth.workload("decode_27b")[3].weight_bytes == 437575680 + 4
