"""The device's own log / exp / tanh / Gumbel transform / BF16 rounding are
bit-identical to the oracle's independent C implementation."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _dev(api, fn, x: np.ndarray) -> np.ndarray:
    y = api.markov_device_math(fn, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _same(a, b):
    an, bn = np.isnan(a), np.isnan(b)
    assert np.array_equal(an, bn)
    assert np.array_equal(a[~an].view(np.uint32), b[~bn].view(np.uint32))


def test_log_bit_identical(gpu_lib):
    x = np.arange(0, 1 << 32, 509, dtype=np.uint64).astype(np.uint32).view(np.float32)
    _same(_dev(gpu_lib, 0, x), oracle.log(x))


def test_exp_bit_identical(gpu_lib):
    x = np.arange(0, 1 << 32, 509, dtype=np.uint64).astype(np.uint32).view(np.float32)
    _same(_dev(gpu_lib, 1, x), oracle.exp(x))


def test_tanh_bit_identical(gpu_lib):
    x = np.arange(0, 1 << 32, 509, dtype=np.uint64).astype(np.uint32).view(np.float32)
    _same(_dev(gpu_lib, 2, x), oracle.tanh(x))


def test_gumbel_transform_exhaustive(gpu_lib):
    # every u the hash can produce: (m + 1/2) 2^-23, m < 2^23
    m = np.arange(1 << 23, dtype=np.float64)
    u = ((m + 0.5) * 2.0**-23).astype(np.float32)
    _same(_dev(gpu_lib, 3, u), -oracle.log(-oracle.log(u)))


def test_bf16_rounding_bit_identical(gpu_lib):
    rng = np.random.default_rng(1)
    x = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32).view(np.float32)
    y = _dev(gpu_lib, 4, x).view(np.uint32)
    ref = oracle.bf16_rne(x).astype(np.uint32)
    nan = np.isnan(x)
    assert np.array_equal(y[~nan], ref[~nan])
    assert np.all((y[nan] & 0x7FFF) > 0x7F80)


def test_packed_bf16_rounding_bit_identical(gpu_lib):
    # the epilogue's packed conversion: same bits as the oracle's rounding
    # for every non-NaN input, some NaN for a NaN
    rng = np.random.default_rng(2)
    x = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -1.0, 2.0**-133, -(2.0**-149),
                        3.3895314e38, 3.4e38, -3.4e38, 1.00390625, 1.01171875],
                       dtype=np.float32)
    x = np.concatenate([x, special])
    y = _dev(gpu_lib, 5, x).view(np.uint32)
    ref = oracle.bf16_rne(x).astype(np.uint32)
    nan = np.isnan(x)
    assert np.array_equal(y[~nan], ref[~nan])
    assert np.all((y[nan] & 0x7FFF) > 0x7F80)
