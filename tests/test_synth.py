"""The seeded input generator: determinism, slicing, distribution, rounding,
and (on a GPU) bit-identity of the CUDA copy with the numpy one."""
import math

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
    assert abs(np.mean(v ** 4) / np.var(v) ** 2 - 3.0) < 0.03    # normal kurtosis
    # normal tails: P(|z| > k) = erfc(k / sqrt 2) for k = 3, 4 (binomial sampling error
    # about 5e-5 and 8e-6 at 2^20 draws)
    assert abs(np.mean(np.abs(v) > 3.0) - math.erfc(3.0 / math.sqrt(2.0))) < 3e-4
    assert abs(np.mean(np.abs(v) > 4.0) - math.erfc(4.0 / math.sqrt(2.0))) < 4e-5
    assert np.abs(v).max() < math.sqrt(-2.0 * math.log(2.0 ** -53)) + 0.05   # u1 >= 2^-53
    w = synth.bf16_bits_to_f64(synth.normal_bf16_bits(0, 2, 0, 1 << 18, 0.0, 0.02))
    assert abs(w.std() - 0.02) < 2e-4
    g = synth.bf16_bits_to_f64(synth.normal_bf16_bits(0, 1, 0, 1 << 18, 1.0, 0.1))
    assert abs(g.mean() - 1.0) < 2e-3 and abs(g.std() - 0.1) < 2e-3


def test_box_muller_series_match_library_log_and_cos():
    """The generator's ln and cos power series against numpy's log and cos:
    the same two draws through z = sqrt(-2 ln u1) cos(2 pi u2) with the
    library functions give the same bf16 value, but for rare cases one unit
    apart where float64 z lands next to a rounding boundary."""
    n, start, seed, stream = 200000, 12345, 0, 3
    key = np.uint64(synth.stream_key(seed, stream))
    c2 = (np.arange(start, start + n, dtype=np.uint64)) * np.uint64(2)
    r1 = synth._splitmix64(key + c2 * np.uint64(synth.GAMMA)) >> np.uint64(11)
    r2 = synth._splitmix64(key + (c2 + np.uint64(1)) * np.uint64(synth.GAMMA)) >> np.uint64(11)
    u1 = (r1 + np.uint64(1)).astype(np.float64) * 2.0 ** -53
    u2 = r2.astype(np.float64) * 2.0 ** -53
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    for mean, std in [(0.0, 1.0), (0.0, 0.02), (1.0, 0.1)]:
        ref = synth.f32_to_bf16_bits((z * std + mean).astype(np.float32)).astype(np.int64)
        got = synth.normal_bf16_bits(seed, stream, start, n, mean, std).astype(np.int64)
        diff = np.abs(got - ref)
        assert diff.max() <= 1 and np.count_nonzero(diff) <= 2, (mean, std, np.count_nonzero(diff))


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
