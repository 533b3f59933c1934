"""The seeded input generator (host side)."""
import numpy as np

import synth_inputs as S


def test_splitmix64_published_outputs():
    # First outputs of SplitMix64 seeded with 0 (the reference C implementation's).
    assert S.splitmix64_sequence(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_vector_mix_equals_scalar_mix():
    z = [0, 1, S.GAMMA, S.MASK64, 0x0123456789ABCDEF]
    assert S.mix64(np.array(z, np.uint64)).tolist() == [S.mix64_int(x) for x in z]


def test_normal_moments_and_bounds():
    key = S.stream_key(11, S.ARRAY_GRAD, 3)
    x = S.normal_f32(key, np.arange(2_000_000), 1.0).astype(np.float64)
    assert abs(x.mean()) < 3e-3
    assert abs(x.std() - 1.0) < 3e-3
    assert np.abs(x).max() <= 6.0
    # kurtosis of Irwin-Hall(12) is 3 - 1.2/12 = 2.9
    k = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert abs(k - 2.9) < 0.02


def test_uniform_range_and_mean():
    v = S.adam_v_f32(4, np.arange(1_000_000))
    assert v.min() >= 0 and v.max() < 1e-6
    assert abs(v.mean() - 5e-7) < 3e-9


def test_keyed_by_logical_index():
    idx = np.array([5, 0, 123456789, 17], np.int64)
    full = S.master_f32(9, np.arange(20))
    assert np.array_equal(S.master_f32(9, idx[[1, 0, 3]]), full[[0, 5, 17]])
    big = S.master_f32(9, idx)
    assert big[2] == S.master_f32(9, np.array([123456789]))[0]


def test_streams_differ():
    idx = np.arange(1000)
    a = S.grad_f32(1, 0, idx)
    assert not np.array_equal(a, S.grad_f32(1, 1, idx))
    assert not np.array_equal(a, S.grad_f32(2, 0, idx))
    assert not np.array_equal(S.master_f32(1, idx), S.adam_m_f32(1, idx))


def test_bf16_grads_are_truncations():
    x = S.grad_f32(3, 2, np.arange(1000))
    b = S.grad_bf16_bits(3, 2, np.arange(1000))
    assert np.array_equal(b.astype(np.uint32), x.view(np.uint32) >> 16)
