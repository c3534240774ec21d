"""The seeded generators against their published definition (SplitMix64, Box-Muller)."""
import math

import numpy as np
import torch

from mxfp8_activation_quant_gb300 import synth


def test_splitmix64_published_first_output():
    # SplitMix64 seeded with 0: first output 0xE220A8397B1DCDAF (the reference value that
    # accompanies the published algorithm's C implementation)
    assert synth.splitmix64_sequence(0, 1)[0] == 0xE220A8397B1DCDAF


def test_torch_hash_matches_python_ints():
    key = synth.stream_key(7, 3)
    idx = torch.arange(1000, dtype=torch.int64)
    got = synth.hash64(key, idx).numpy().view(np.uint64)
    want = np.array([synth.mix64_int(key + (i + 1) * synth.GOLDEN) for i in range(1000)], np.uint64)
    assert np.array_equal(got, want)
    # the same stream as a SplitMix64 sequence seeded with the key
    assert synth.splitmix64_sequence(key, 5) == [int(v) for v in want[:5]]


def test_normals_have_unit_moments():
    z = synth.normal(synth.stream_key(0, 1), torch.arange(1 << 18, dtype=torch.int64))
    assert abs(float(z.mean())) < 0.01
    assert abs(float(z.std()) - 1.0) < 0.01
    u = synth.uniform(synth.stream_key(0, 2), torch.arange(1 << 16, dtype=torch.int64))
    assert float(u.min()) > 0.0 and float(u.max()) < 1.0


def test_row_subset_equals_full_draw():
    full = synth.quantizer_input(0, 40, K=256)
    rows = torch.tensor([0, 5, 39])
    sub = synth.quantizer_input(0, 40, K=256, rows=rows)
    assert torch.equal(full[rows].view(torch.int16), sub.view(torch.int16))
    o_full = synth.o_proj_activation(0, 3)
    o_sub = synth.o_proj_activation(0, 3, rows=torch.tensor([2]))
    assert torch.equal(o_full[2:3].view(torch.int16), o_sub.view(torch.int16))


def test_quantizer_input_special_classes_present():
    x = synth.bf16_bits(synth.quantizer_input(0, 64, K=8192)).astype(np.int64)
    g = x.reshape(-1, 32)
    exp = (g >> 7) & 0xFF
    all_zero = np.all((g & 0x7FFF) == 0, axis=1)
    all_sub = np.all(exp == 0, axis=1) & ~all_zero
    big = np.any((g & 0x7FFF) >= 0x7F00, axis=1)
    assert all_zero.mean() > 0.005 and all_sub.mean() > 0.005 and big.mean() > 0.005
    assert not np.any(exp == 0xFF)   # finite only


def test_rmsnorm_inputs_shape_and_outliers():
    x = synth.rmsnorm_input(0, 4)
    ch = synth.rmsnorm_outlier_channels(0)
    assert x.shape == (4, 5120) and len(ch) == 5
    ratio = x.float()[:, ch].abs().mean() / x.float().abs().mean()
    assert ratio > 10
    g = synth.rmsnorm_gamma(0)
    assert abs(float(g.float().mean()) - 1.0) < 0.01
