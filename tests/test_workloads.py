"""Pins for the seeded input generator (CPU only)."""
import numpy as np
import pytest
from scipy import stats

import workloads as W


def test_splitmix64_published_sequence():
    # splitmix64 started from state 1234567 (the sequence printed with Vigna's
    # public reference implementation)
    got = [int(x) for x in W._raw(np.uint64(1234567), 0, 5)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_normal_is_counter_based_and_standard():
    a = W.normal_fp16(0, 1, (3_000_001,))
    b = W.normal_fp16(0, 1, (1001,))
    assert np.array_equal(a[:1001], b)           # prefix property across chunk sizes
    x = a.astype(np.float64)
    assert abs(x.mean()) < 3e-3 and abs(x.std() - 1) < 3e-3
    assert stats.kstest(x[:200_000], "norm").pvalue > 1e-3
    assert not np.array_equal(W.normal_fp16(0, 0, (64,)), W.normal_fp16(0, 1, (64,)))
    assert not np.array_equal(W.normal_fp16(0, 0, (64,)), W.normal_fp16(1, 0, (64,)))


def test_uniform_int_and_permutation():
    u = W.uniform_int(0, 3, 100_000, 128, 2048)
    assert u.min() == 128 and u.max() == 2048
    p = W.permutation(0, 4, 5000)
    assert np.array_equal(np.sort(p), np.arange(5000))


def test_decode_layout_tables():
    lens = np.array([0, 1, 16, 17, 2048], np.int32)
    t, nb = W.decode_layout(lens, 16, 128, seed=0)
    pages = [0, 1, 1, 2, 128]
    assert nb == sum(pages)
    used = np.concatenate([t[n, :p] for n, p in enumerate(pages)])
    assert np.array_equal(np.sort(used), np.arange(nb))
    for n, p in enumerate(pages):
        assert np.all(t[n, p:] == -1)
    with pytest.raises(ValueError):
        W.decode_layout(np.array([2049], np.int32), 16, 128)


def test_config_sizes():
    assert W.PREFILL_LONG.flops() == 2 * 2 * 32 * 8192 ** 2 * 128
    assert W.PREFILL_LONG_FULL.flops() == 2 * W.PREFILL_LONG.flops()
    assert W.PREFILL_QWEN.flops() == pytest.approx(1.718e10, rel=1e-3)
    lens = np.full(8, 32768, np.int32)
    assert int(lens.sum()) * 8 * 128 * 2 * 2 == 1073741824
    mix = W.uniform_int(0, 3, 256, 128, 2048)
    assert 250_000 < mix.sum() < 310_000
