"""The seeded input generator: determinism, slicing, distribution, rounding,
and (on a GPU) bit-identity of the CUDA copy with the numpy one."""
import numpy as np
import pytest

import synth


def test_deterministic_and_sliceable():
    a = synth.normal_bf16_bits(0, 3, 0, 10000, 0.0, 1.0)
    b = synth.normal_bf16_bits(0, 3, 0, 10000, 0.0, 1.0)
    np.testing.assert_array_equal(a, b)
    c = synth.normal_bf16_bits(0, 3, 1234, 500, 0.0, 1.0)
    np.testing.assert_array_equal(a[1234:1734], c)
    full = synth.tensor_bits(0, "x", (5, 7, 11), synth.X_DIST)
    rows = synth.tensor_bits(0, "x", (5, 7, 11), synth.X_DIST, rows=[3, 1])
    np.testing.assert_array_equal(rows, full[[3, 1]])
    assert not np.array_equal(synth.normal_bf16_bits(1, 3, 0, 100, 0, 1), a[:100])
    assert not np.array_equal(synth.normal_bf16_bits(0, 4, 0, 100, 0, 1), a[:100])


def test_distribution_moments():
    v = synth.bf16_bits_to_f64(synth.normal_bf16_bits(0, 0, 0, 1 << 20, 0.0, 1.0))
    assert abs(v.mean()) < 5e-3
    assert abs(v.std() - 1.0) < 5e-3
    assert np.abs(v).max() <= np.sqrt(3.0) * 2 + 1e-2        # Irwin-Hall(4) support
    w = synth.bf16_bits_to_f64(synth.normal_bf16_bits(0, 2, 0, 1 << 18, 0.0, 0.02))
    assert abs(w.std() - 0.02) < 2e-4
    g = synth.bf16_bits_to_f64(synth.normal_bf16_bits(0, 1, 0, 1 << 18, 1.0, 0.1))
    assert abs(g.mean() - 1.0) < 2e-3 and abs(g.std() - 0.1) < 2e-3


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    f = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 10
    ours = synth.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


@pytest.mark.gpu
def test_cuda_generator_bit_identical(gpu_available):
    import torch
    for (seed, name, start, n, dist) in [(0, "x", 0, 100003, synth.X_DIST),
                                         (0, "w_q_b", 777777, 65536, synth.WEIGHT_DIST),
                                         (5, "w_q_a_norm", 3, 1536, synth.GAIN_DIST)]:
        ref = synth.normal_bf16_bits(seed, synth.STREAMS[name], start, n, *dist)
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_bf16_cuda(t.data_ptr(), n, seed, synth.STREAMS[name], start, *dist,
                                    torch.cuda.current_stream().cuda_stream)
        got = t.view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(got, ref)
