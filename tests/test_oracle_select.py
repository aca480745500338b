"""Pins of the oracle's selection rules: brute force at tiny V against
numpy.argmax (which takes the first maximum and the first NaN, the
torch.argmax order), the sampling law by chi-square against fp64
softmax(l / T) in both modes, and exact inverse-CDF cases whose answer an
independent big-integer computation gives."""
import numpy as np
import pytest
from scipy.stats import chisquare

import oracle
from oracle import GUMBEL, INVCDF

M64 = (1 << 64) - 1


def _py_sm(x: int) -> int:
    z = (x + 0x9E3779B97F4A7C15) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def _bits(vals) -> np.ndarray:
    return oracle.bf16_rne(np.asarray(vals, dtype=np.float32))


def _np_first_argmax_with_nan(keys: np.ndarray) -> int:
    keys = np.where(keys == 0.0, 0.0, keys)  # -0 == +0
    return int(np.argmax(keys))


def _edge_rows(rng, V):
    pool = np.float32([0.0, -0.0, 1.0, 1.0, -1.0, 2.5, 2.5, np.inf, -np.inf, np.nan, 7.0])
    for _ in range(300):
        row = rng.standard_normal(V).astype(np.float32) * 2
        k = rng.integers(0, 4)
        for _ in range(k):
            row[rng.integers(0, V)] = pool[rng.integers(0, len(pool))]
        if rng.random() < 0.3:  # exact ties at the maximum
            m = row[~np.isnan(row)].max() if (~np.isnan(row)).any() else 0.0
            row[rng.integers(0, V, size=2)] = m
        yield row


@pytest.mark.parametrize("V", [16, 32])
def test_greedy_bruteforce(V):
    rng = np.random.default_rng(V)
    for row in _edge_rows(rng, V):
        l = _bits(row)
        lf = oracle.bits_to_f32(l)
        tok, _, _ = oracle.select(l, 0.0, GUMBEL, 1, 0, 0)
        assert tok == _np_first_argmax_with_nan(lf)
        tok2, _, _ = oracle.select(l, 0.0, INVCDF, 1, 0, 0)
        assert tok2 == tok


@pytest.mark.parametrize("V", [16, 32])
def test_gumbel_bruteforce(V):
    rng = np.random.default_rng(100 + V)
    for n, row in enumerate(_edge_rows(rng, V)):
        l = _bits(row)
        T = float(np.float32(rng.choice([0.6, 1.0, 1.5])))
        seed, b, i = int(rng.integers(0, 2**62)), n % 8, n % 5
        g = oracle.gumbel(seed, b, i, 0, V)
        keys = (oracle.bits_to_f32(l) / np.float32(T)).astype(np.float32) + g
        tok, k1, k2 = oracle.select(l, T, GUMBEL, seed, b, i)
        assert tok == _np_first_argmax_with_nan(keys.astype(np.float32))
        if not np.isnan(keys).any():
            srt = np.sort(keys)[::-1]
            assert k1 == srt[0] and k2 == srt[1]


def test_nan_rule_lowest_nan_in_every_mode():
    row = np.float32([1.0, 3.0, np.nan, 9.0, np.nan, -np.inf])
    l = _bits(row)
    for T in (0.0, 0.7, 1.0):
        for mode in (GUMBEL, INVCDF):
            assert oracle.select(l, T, mode, 5, 0, 0)[0] == 2


def test_negative_and_nan_temperature_are_greedy():
    l = _bits([1.0, 5.0, 5.0, 2.0])
    for T in (-1.0, float("nan"), 0.0):
        for mode in (GUMBEL, INVCDF):
            assert oracle.select(l, T, mode, 9, 1, 1)[0] == 1


def test_invcdf_infinities():
    l = _bits([1.0, np.inf, 2.0, np.inf])
    assert oracle.select(l, 0.8, INVCDF, 3, 0, 0)[0] == 1
    l = _bits([-np.inf] * 5)
    assert oracle.select(l, 0.8, INVCDF, 3, 0, 0)[0] == 0


def test_invcdf_exact_integer_cases():
    # Logits in {M, -inf} give weights exactly 2^40 and 0: the token is the
    # (floor(t / 2^40))-th maximal id, with t = mulhi64(H, S) and H the
    # salted row-step hash; computed here with Python integers.
    rng = np.random.default_rng(5)
    for trial in range(200):
        V = int(rng.integers(2, 40))
        mask = rng.random(V) < 0.5
        mask[rng.integers(0, V)] = True
        M = float(rng.choice([0.0, 1.5, -3.0, 12.0]))
        row = np.where(mask, M, -np.inf).astype(np.float32)
        seed, b, i = int(rng.integers(0, 2**63)), trial % 7, trial % 3
        T = 1.0
        H = _py_sm(_py_sm(_py_sm(_py_sm(seed) ^ b) ^ i) ^ (1 << 63))
        ids = np.flatnonzero(mask)
        S = len(ids) << 40
        t = (H * S) >> 64
        want = int(ids[t >> 40])
        assert oracle.select(_bits(row), T, INVCDF, seed, b, i)[0] == want


def _law_case(V, T, mode, n_draws, seed0):
    rng = np.random.default_rng(seed0)
    logits = (rng.standard_normal(V) * 1.5).astype(np.float32)
    l = _bits(logits)
    rows = n_draws
    base = np.broadcast_to(l, (rows, 1, V)).copy()
    head = np.zeros((V, 8), dtype=np.uint16)      # zero head: bias = 0, l = base
    embed = np.zeros((V, 8), dtype=np.uint16)
    anchor = np.zeros(rows, dtype=np.int32)
    temp = np.full(rows, T, dtype=np.float32)
    seeds = np.arange(rows, dtype=np.int64) * 7919 + seed0
    idx = np.arange(rows, dtype=np.int64)
    toks, _ = oracle.chain(base, head, embed, anchor, temp, seeds, idx, mode, nthreads=1)
    counts = np.bincount(toks[:, 0], minlength=V)
    x = oracle.bits_to_f32(l).astype(np.float64) / np.float64(np.float32(T))
    p = np.exp(x - x.max())
    p /= p.sum()
    return counts, p


@pytest.mark.parametrize("mode", [GUMBEL, INVCDF])
@pytest.mark.parametrize("V,T", [(16, 0.6), (16, 1.0), (64, 1.5), (64, 1.0)])
def test_sampling_law_chi_square(mode, V, T):
    counts, p = _law_case(V, T, mode, 200_000, 17 + V + int(T * 10))
    expected = p * counts.sum()
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    assert chisquare(obs, exp).pvalue > 1e-4


def test_sampling_law_detects_wrong_temperature():
    # Power check: the same counts against the law at another temperature fail.
    counts, _ = _law_case(16, 0.6, GUMBEL, 200_000, 33)
    rng = np.random.default_rng(33)
    logits = (rng.standard_normal(16) * 1.5).astype(np.float32)
    x = oracle.bits_to_f32(_bits(logits)).astype(np.float64) * 0.6  # l * T instead of l / T
    p = np.exp(x - x.max())
    p /= p.sum()
    assert chisquare(counts, p * counts.sum()).pvalue < 1e-6
