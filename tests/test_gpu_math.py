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


def _uniform_of_mantissa(m: np.ndarray) -> np.ndarray:
    return ((m.astype(np.float64) + 0.5) * 2.0**-23).astype(np.float32)


def test_gumbel_noise_bounds_exhaustive(gpu_lib):
    # the tcgen05 chain prunes Gumbel rows with one noise byte per (id, row):
    # for every u the hash can give, the byte's lower and upper ends must
    # bracket the exact noise the oracle computes, and the byte must not
    # saturate (a saturated byte would not be a bound)
    m = np.arange(1 << 23, dtype=np.uint32)
    q = _dev(gpu_lib, 6, m.view(np.float32))
    assert q.min() > 0.0 and q.max() < 255.0
    assert np.array_equal(q, np.round(q))
    lo = _dev(gpu_lib, 8, q)
    hi = _dev(gpu_lib, 7, q)
    u = _uniform_of_mantissa(m)
    g = -oracle.log(-oracle.log(u))
    assert np.all(lo <= g), float(np.max(lo - g))
    assert np.all(g <= hi), float(np.max(g - hi))
    # the byte is a useful bound: its upper end within a byte step of g
    assert float(np.max(hi - g)) < 1.0 / 12.0 + 0.02


def _key_triples(rng, n):
    l = np.concatenate([
        rng.standard_normal(n).astype(np.float32) * np.float32(3.0),
        rng.standard_normal(n).astype(np.float32) * np.float32(300.0),
        (rng.standard_normal(n) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1e-45, -1e-45, 1e-38, -1e-38, 3.3e38, -3.3e38, np.inf, -np.inf,
                  64.0, -64.0], dtype=np.float32)])
    Ts = np.array([0.05, 0.6, 1.0, 3.0], dtype=np.float32)
    T = np.concatenate([Ts[rng.integers(0, 4, l.size - n)],
                        np.exp(rng.uniform(-4.0, 2.5, n)).astype(np.float32)])
    rng.shuffle(T)
    m = rng.integers(0, 1 << 23, l.size, dtype=np.uint32)
    return l, T, m


def test_gumbel_key_bounds_bracket_the_exact_key(gpu_lib):
    # key_lower <= fp32(l / T) + gumbel(u) <= key_upper for logits of every
    # scale (BF16 and fp32 caches, overflowing quotients, infinities) and
    # temperatures 0.05 .. 12; the device's exact key equals the oracle's
    rng = np.random.default_rng(7)
    l, T, m = _key_triples(rng, 1 << 20)
    x = np.empty(3 * l.size, dtype=np.float32)
    x[0::3], x[1::3], x[2::3] = l, T, m.view(np.float32)
    y = _dev(gpu_lib, 9, x)
    lo, hi, ex = y[0::3], y[1::3], y[2::3]
    with np.errstate(over="ignore", invalid="ignore"):
        q = np.where(T == np.float32(1.0), l, l / T).astype(np.float32)
        key = (q + (-oracle.log(-oracle.log(_uniform_of_mantissa(m))))).astype(np.float32)
    _same(ex, key)
    lo = np.where(np.isnan(lo), -np.inf, lo)
    hi = np.where(np.isnan(hi), np.inf, hi)
    assert np.all(lo <= key), int(np.sum(~(lo <= key)))
    assert np.all(key <= hi), int(np.sum(~(key <= hi)))


def _weights(api, d: np.ndarray) -> np.ndarray:
    lo = _dev(api, 10, d).view(np.uint32).astype(np.uint64)
    hi = _dev(api, 11, d).view(np.uint32).astype(np.uint64)
    return lo | (hi << np.uint64(32))


def _oracle_weights(d: np.ndarray) -> np.ndarray:
    # the oracle's inverse-CDF weight: its exp, an exact fp32 scale by 2^40,
    # then truncation to an unsigned integer
    e = oracle.exp(d).astype(np.float32) * np.float32(2.0 ** 40)
    return e.astype(np.uint64)


def test_cdf_weight_matches_the_oracle(gpu_lib):
    # (1) every 257th fp32 in [-40, 0] (bit patterns of -0 .. -40), (2) every
    # fp32 around the -28 cut, (3) the d = fp32(x / T) - M of every finite
    # BF16 logit x for several temperatures and maxima M >= every x / T
    neg40 = int(np.float32(-40.0).view(np.uint32))
    d1 = np.arange(0x80000000, neg40 + 1, 257, dtype=np.uint64).astype(np.uint32).view(np.float32)
    c = int(np.float32(-28.0).view(np.uint32))
    d2 = np.arange(c - (1 << 18), c + (1 << 18), dtype=np.uint64).astype(np.uint32).view(np.float32)
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    x = x[np.isfinite(x)]
    d3 = []
    for T in (0.37, 0.5, 0.7, 0.8, 1.0, 1.2, 3.0):
        q = (x / np.float32(T)).astype(np.float32)
        for M in (q.max(), np.float32(0.0) + q.max() * np.float32(0.5), np.float32(12.5),
                  np.float32(30.0)):
            d = (q - np.float32(M)).astype(np.float32)
            d3.append(d[d <= 0])
    d = np.concatenate([d1, d2, np.float32([-np.inf, -0.0, 0.0, -27.7, -27.73, -28.0])] + d3)
    assert np.all((d <= 0) | np.isneginf(d))
    got, want = _weights(gpu_lib, d), _oracle_weights(d)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (d[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_temperature_division_is_ieee(gpu_lib):
    # fp32(l / T) for every finite BF16 logit, powers of two from 2^-126 to
    # 2^127 (the product path) and other temperatures (the division path),
    # against numpy's IEEE float32 division
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    x = x[np.isfinite(x)]
    p2 = [np.float32(2.0) ** np.float32(k) for k in range(-126, 128, 7)] + [np.float32(0.5), np.float32(1.0)]
    other = [np.float32(v) for v in (0.7, 0.8, 1.2, 3.0, 1e-30)]
    pairs = []
    for T in p2 + other:
        pairs.append(np.stack([x, np.full_like(x, T)], axis=1))
    xt = np.concatenate(pairs).astype(np.float32).reshape(-1)
    y = _dev(gpu_lib, 12, xt).reshape(-1, 2)
    l, T = xt.reshape(-1, 2)[:, 0], xt.reshape(-1, 2)[:, 1]
    with np.errstate(all="ignore"):
        want = (l / T).astype(np.float32)
    _same(y[:, 0], want)
    is_p2 = np.isin(T, np.float32(p2))
    assert np.array_equal(y[:, 1] == 1.0, is_p2)
