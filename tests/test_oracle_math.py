"""Pins of the oracle's scalar pieces against things other than itself:
torch's BF16 conversion, float64 libm (numpy), published splitmix64 vectors,
an independent big-integer splitmix64, and closed forms of the Gumbel law."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1


# ---------------------------------------------------------------- BF16 RNE

def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _check_bf16(bits_u32: np.ndarray):
    x = bits_u32.view(np.float32)
    ours = oracle.bf16_rne(x)
    ref = _torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(oracle.bits_to_f32(ours[nan])))


def test_bf16_rne_all_low_halves():
    # Rounding depends on the low 16 bits and the kept LSB: every low half
    # against a spread of high halves (both signs, both LSB parities,
    # subnormals, the overflow edge, inf/NaN).
    lows = np.arange(1 << 16, dtype=np.uint32)
    highs = np.array([0x0000, 0x0001, 0x0080, 0x3F80, 0x3F81, 0x4080, 0x42F6, 0x7F7F,
                      0x7F7E, 0x7F80, 0x7FC0, 0x8000, 0x8001, 0xBF80, 0xC2F7, 0xFF7F,
                      0xFF80, 0xFFC0], dtype=np.uint32)
    _check_bf16(((highs[:, None] << 16) | lows[None, :]).ravel())


def test_bf16_rne_all_high_halves():
    highs = np.arange(1 << 16, dtype=np.uint32)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000],
                    dtype=np.uint32)
    _check_bf16(((highs[:, None] << 16) | lows[None, :]).ravel())


def test_bf16_rne_random_patterns():
    rng = np.random.default_rng(7)
    _check_bf16(rng.integers(0, 1 << 32, size=4_000_000, dtype=np.uint64).astype(np.uint32))


def test_bf16_add_matches_torch_bf16_add():
    # s = bf16(f32(base) + f32(bias)) is torch's BF16 addition.
    rng = np.random.default_rng(3)
    a = torch.from_numpy((rng.standard_normal(1_000_000) * 3).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy((rng.standard_normal(1_000_000) * 0.01).astype(np.float32)).to(torch.bfloat16)
    ref = (a + b).view(torch.int16).numpy().view(np.uint16)
    ab = oracle.bf16_bits(a)
    bb = oracle.bf16_bits(b)
    lib = oracle.lib()
    ours = np.array([lib.orc_logit(int(x), int(y), 0, 1.0, 0, 1.0, 1.0)
                     for x, y in zip(ab[:20000], bb[:20000])], dtype=np.uint16)
    assert np.array_equal(ours, ref[:20000])


# ------------------------------------------------------------- own math

def _ulp_err(y32: np.ndarray, ref64: np.ndarray) -> np.ndarray:
    sp = np.spacing(np.abs(ref64.astype(np.float32))).astype(np.float64)
    return np.abs(y32.astype(np.float64) - ref64) / sp


def test_log_accuracy():
    x = np.arange(0x00800000, 0x7F800000, 211, dtype=np.uint32).view(np.float32)
    assert _ulp_err(oracle.log(x), np.log(x.astype(np.float64))).max() <= 2.0
    # the noise's domains: u in [2^-24, 1) and w = -log u in (0, 17)
    u = np.arange(np.float32(2.0**-24).view(np.uint32), np.float32(1.0).view(np.uint32), 41,
                  dtype=np.uint32).view(np.float32)
    assert _ulp_err(oracle.log(u), np.log(u.astype(np.float64))).max() <= 2.0
    assert oracle.log(np.float32([1.0]))[0] == 0.0


def test_log_special_values():
    x = np.float32([0.0, -0.0, -1.0, np.inf, np.nan, 1e-45, 2.0**-149])
    y = oracle.log(x)
    assert y[0] == -np.inf and y[1] == -np.inf and np.isnan(y[2]) and y[3] == np.inf
    assert np.isnan(y[4])
    assert abs(y[5] - np.log(np.float64(np.float32(1e-45)))) < 1e-4


def test_exp_accuracy():
    neg = np.arange(0x80000001, np.float32(-87.0).view(np.uint32), 401, dtype=np.uint32)
    pos = np.arange(0x00000001, np.float32(88.72).view(np.uint32), 401, dtype=np.uint32)
    x = np.concatenate([neg, pos]).view(np.float32)
    assert _ulp_err(oracle.exp(x), np.exp(x.astype(np.float64))).max() <= 1.0
    y = oracle.exp(np.float32([0.0, -0.0, -88.0, 89.0, -np.inf, np.inf, np.nan]))
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == 0.0 and y[3] == np.inf
    assert y[4] == 0.0 and y[5] == np.inf and np.isnan(y[6])


def test_tanh_accuracy_and_symmetry():
    x = np.arange(0x00000001, np.float32(20.0).view(np.uint32), 257, dtype=np.uint32).view(np.float32)
    x = np.concatenate([x, -x])
    y = oracle.tanh(x)
    assert _ulp_err(y, np.tanh(x.astype(np.float64))).max() <= 2.0
    n = len(x) // 2
    assert np.array_equal(y[:n], -y[n:])
    z = oracle.tanh(np.float32([0.0, np.inf, -np.inf, 40.0, np.nan]))
    assert z[0] == 0.0 and z[1] == 1.0 and z[2] == -1.0 and z[3] == 1.0 and np.isnan(z[4])


# ----------------------------------------------------------- splitmix64

def _py_splitmix64(x: int) -> int:
    """Independent big-integer splitmix64, from the published definition."""
    z = (x + 0x9E3779B97F4A7C15) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_splitmix64_published_vectors():
    with open(os.path.join(GOLDEN, "splitmix64_vectors.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            state, n = int(parts[0]), int(parts[1])
            want = [int(p, 0) for p in parts[2:2 + n]]
            got = []
            for _ in range(n):
                # the generator's k-th output is sm(state + (k-1) gamma)
                got.append(int(oracle.splitmix64(np.array([state], dtype=np.uint64))[0]))
                state = (state + 0x9E3779B97F4A7C15) & M64
            assert got == want


def test_splitmix64_matches_bigint():
    rng = np.random.default_rng(11)
    x = rng.integers(0, 2**63, size=2000, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    y = oracle.splitmix64(x)
    assert all(int(b) == _py_splitmix64(int(a)) for a, b in zip(x, y))


def test_row_step_hash_composition():
    for seed in (0, 1, 2**63 + 5, M64, 123456789):
        for row in (0, 1, 7, 63):
            for step in (0, 1, 7, 15):
                want = _py_splitmix64(_py_splitmix64(_py_splitmix64(seed) ^ row) ^ step)
                assert oracle.row_step_hash(seed, row, step) == want
                cdf = _py_splitmix64(want ^ (1 << 63))
                assert oracle.cdf_hash(seed, row, step) == cdf


def test_uniform_is_exact_top_23_bits():
    for h in (0, 1, (1 << 41) - 1, 1 << 41, M64, 0x123456789ABCDEF0):
        m = h >> 41
        assert oracle.uniform(h) == (m + 0.5) * 2.0**-23
    assert oracle.uniform(0) == 2.0**-24
    assert oracle.uniform(M64) == 1 - 2.0**-24


def test_gumbel_noise_is_hash_then_two_logs():
    seed, row, step = 99, 3, 5
    g = oracle.gumbel(seed, row, step, 1000, 64)
    hrs = _py_splitmix64(_py_splitmix64(_py_splitmix64(seed) ^ row) ^ step)
    for j in range(64):
        u = ((_py_splitmix64(hrs ^ (1000 + j)) >> 41) + 0.5) * 2.0**-23
        ref = -np.log(-np.log(u))
        assert abs(float(g[j]) - ref) <= 4e-6 * max(1.0, abs(ref))


def test_gumbel_moments():
    # Gumbel(0,1): mean = Euler-Mascheroni gamma, variance = pi^2 / 6.
    g = np.concatenate([oracle.gumbel(s, r, i, 0, 500_000).astype(np.float64)
                        for s, r, i in ((1, 0, 0), (2, 3, 1), (3, 1, 7), (2**40, 6, 2))])
    assert abs(g.mean() - 0.5772156649015329) < 6e-3
    assert abs(g.var() - np.pi**2 / 6) < 2e-2


def test_uniform_histogram():
    from scipy.stats import chisquare
    seed, row, step = 5, 2, 3
    hrs = oracle.row_step_hash(seed, row, step)
    v = np.arange(400_000, dtype=np.uint64)
    h = oracle.splitmix64(np.uint64(hrs) ^ v)
    u = ((h >> np.uint64(41)).astype(np.float64) + 0.5) * 2.0**-23
    counts, _ = np.histogram(u, bins=64, range=(0.0, 1.0))
    assert chisquare(counts).pvalue > 1e-4
