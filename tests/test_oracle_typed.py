"""Pins of the oracle's fp32 base-logit and fp32 cache variants (the
sharded_markov page's chain takes BF16 or fp32 for both: set-up and _kernel
compile it per base and cache dtype; the module docstring's
cache_round(base + bf16(head . embed)) rounds to the cache's dtype).

  * with a BF16 base and a BF16 cache the typed logit, selection and chain
    are the pinned BF16 ones, bit for bit;
  * an fp32 cache without a transform holds exactly f32(base) + f32(bias):
    numpy's IEEE fp32 sum of the two, brute force over a small chain;
  * with a transform, the fp32 cache holds the fp32 steps of the transform
    (numpy fp32 products around the oracle's pinned tanh);
  * an fp32 base with BF16-representable values gives the BF16 chain;
  * the tokens are the selection applied to the chain's own fp32 cache."""
import numpy as np
import pytest
import torch

import oracle
from oracle import GUMBEL, INVCDF
from draft_token_markov_gb300 import workloads as W


def _weights(w):
    head, embed = W.make_weights(w)
    return oracle.bf16_bits(head), oracle.bf16_bits(embed)


def _args(c):
    return (c["anchor"].numpy(), c["temperature"].numpy(), c["seeds"].numpy(),
            c["row_state_idx"].numpy())


def test_typed_logit_equals_bf16_logit_for_a_bf16_cache():
    rng = np.random.default_rng(5)
    base = oracle.bf16_rne(rng.normal(0, 4, 4000).astype(np.float32))
    bias = oracle.bf16_rne(rng.normal(0, 0.5, 4000).astype(np.float32))
    base[:3] = [0x7F80, 0xFF80, 0x7FC0]        # +inf, -inf, NaN
    for mult, cap in ((1.0, None), (0.5, None), (1.0, 30.0), (0.7, 12.0)):
        for b, s in zip(base, bias):
            want = oracle.bits_to_f32(np.array([oracle.logit(int(b), int(s), mult, cap)],
                                               dtype=np.uint16))[0]
            got = np.float32(oracle.logit_typed(float(oracle.bits_to_f32(np.array([b]))[0]),
                                                int(s), False, mult, cap))
            assert (np.isnan(want) and np.isnan(got)) or want == got


def test_fp32_cache_is_the_fp32_sum_without_rounding():
    rng = np.random.default_rng(6)
    base = rng.normal(0, 4, 3000).astype(np.float32)
    bias = oracle.bf16_rne(rng.normal(0, 0.5, 3000).astype(np.float32))
    want = base + oracle.bits_to_f32(bias)                       # IEEE fp32 sums
    got = np.array([oracle.logit_typed(float(b), int(s), True) for b, s in zip(base, bias)],
                   dtype=np.float32)
    assert np.array_equal(got, want)
    # and a BF16 cache rounds that same sum once
    got16 = np.array([oracle.logit_typed(float(b), int(s), False) for b, s in zip(base, bias)],
                     dtype=np.float32)
    assert np.array_equal(got16, oracle.bits_to_f32(oracle.bf16_rne(want)))


def test_fp32_cache_transform_steps():
    rng = np.random.default_rng(7)
    base = rng.normal(0, 20, 2000).astype(np.float32)
    bias = oracle.bf16_rne(rng.normal(0, 0.5, 2000).astype(np.float32))
    mult, cap = 0.75, 30.0
    s = base + oracle.bits_to_f32(bias)
    y = (s * np.float32(mult)).astype(np.float32)
    inv = np.float32(1.0) / np.float32(cap)
    want = (np.float32(cap) * oracle.tanh((y * inv).astype(np.float32))).astype(np.float32)
    got = np.array([oracle.logit_typed(float(b), int(t), True, mult, cap)
                    for b, t in zip(base, bias)], dtype=np.float32)
    assert np.array_equal(got, want)
    got_m = np.array([oracle.logit_typed(float(b), int(t), True, mult, None)
                      for b, t in zip(base, bias)], dtype=np.float32)
    assert np.array_equal(got_m, y)


@pytest.mark.parametrize("mode", [GUMBEL, INVCDF])
def test_typed_chain_with_bf16_dtypes_is_the_bf16_chain(mode):
    w = W.small(700, 32, 3, 4, mode, seed=61, padding_rows=(1,), spikes=3)
    hb, eb = _weights(w)
    c = W.make_call(w)
    base = oracle.bf16_bits(c["base"])
    t0, c0 = oracle.chain(base, hb, eb, *_args(c), mode, mult=0.5, cap=20.0)
    t1, c1 = oracle.chain_typed(base, hb, eb, *_args(c), mode, mult=0.5, cap=20.0)
    assert np.array_equal(t0, t1) and np.array_equal(c0, c1)
    # an fp32 base holding the same (BF16-representable) values: same chain
    t2, c2 = oracle.chain_typed(oracle.bits_to_f32(base), hb, eb, *_args(c), mode, mult=0.5,
                                cap=20.0)
    assert np.array_equal(t0, t2) and np.array_equal(c0, c2)


@pytest.mark.parametrize("mode", [GUMBEL, INVCDF])
def test_fp32_cache_chain_brute_force(mode):
    w = W.small(600, 32, 3, 3, mode, seed=62, padding_rows=(2,), spikes=2,
                temperatures=(0.0, 0.8, 1.0))
    hb, eb = _weights(w)
    c = W.make_call(w, base_f32=True)
    base = c["base"].numpy()
    anchor, temp, seeds, idx = _args(c)
    toks, cache = oracle.chain_typed(base, hb, eb, anchor, temp, seeds, idx, mode, cache_f32=True)
    R, N, V = base.shape
    for b in range(R):
        if idx[b] < 0:
            assert np.all(toks[b] == -1) and np.all(np.isnan(cache[b]))
            continue
        p = int(anchor[b])
        for i in range(N):
            bias = oracle.bias_all(hb, eb, p)
            want = base[b, i] + oracle.bits_to_f32(bias)
            assert np.array_equal(cache[b, i], want)
            tok, _, _ = oracle.select_f(cache[b, i], float(temp[b]), mode, int(seeds[b]), b, i)
            assert tok == toks[b, i]
            p = int(toks[b, i])


def test_select_f_on_bf16_values_is_select_on_bits():
    rng = np.random.default_rng(8)
    bits = oracle.bf16_rne(rng.normal(0, 3, 500).astype(np.float32))
    vals = oracle.bits_to_f32(bits)
    for mode in (GUMBEL, INVCDF):
        for T in (0.0, 0.7, 1.0):
            a = oracle.select(bits, T, mode, 99, 1, 2)
            b = oracle.select_f(vals, T, mode, 99, 1, 2)
            assert a[0] == b[0]
