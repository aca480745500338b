"""Pins of the oracle's chain: a closed-form chain whose tokens are known in
advance, the bias against an fp64 dot product, the soft cap against an fp64
30 tanh(x / 30), greedy T = 0 against argmax of the written cache, padding
rows inert, and restarting a row mid-chain."""
import numpy as np
import pytest
import torch

import oracle
from oracle import GUMBEL, INVCDF
from draft_token_markov_gb300 import workloads as W


def _bf16(x) -> np.ndarray:
    return oracle.bf16_rne(np.asarray(x, dtype=np.float32))


def _f32(bits) -> np.ndarray:
    return oracle.bits_to_f32(bits)


def _inputs(w: W.Workload):
    head, embed = W.make_weights(w)
    c = W.make_call(w)
    return (oracle.bf16_bits(c["base"]), oracle.bf16_bits(head), oracle.bf16_bits(embed),
            c["anchor"].numpy(), c["temperature"].numpy(), c["seeds"].numpy(),
            c["row_state_idx"].numpy())


def _closed_form_weights(V, r, c):
    head = np.zeros((V, r), dtype=np.float32)
    embed = np.zeros((V, r), dtype=np.float32)
    for v in range(V):
        head[v, v % r] = c
        embed[v, (v + 1) % r] = c
    return _bf16(head), _bf16(embed)


@pytest.mark.parametrize("V,r", [(64, 8), (96, 16), (256, 64)])
def test_closed_form_chain_greedy(V, r):
    # head[v] = c e_{v mod r}, embed[p] = c e_{(p+1) mod r}: bias[v] = c^2
    # exactly when v = p + 1 (mod r), else 0.  With zero base logits and
    # T = 0 the lowest such id wins, so the tokens walk (anchor+1), (anchor+2),
    # ... mod r: each token is the next position's previous token.
    N, rows = 7, 5
    head, embed = _closed_form_weights(V, r, 0.5)
    base = np.zeros((rows, N, V), dtype=np.uint16)
    anchor = np.array([0, 3, V - 1, r - 1, 17], dtype=np.int32)
    toks, cache = oracle.chain(base, head, embed, anchor, np.zeros(rows, np.float32),
                               np.arange(rows), np.arange(rows), GUMBEL)
    for b in range(rows):
        want = [(int(anchor[b]) + 1 + i) % r for i in range(N)]
        assert toks[b].tolist() == want
        for i in range(N):
            p = int(anchor[b]) if i == 0 else want[i - 1]
            hit = (np.arange(V) % r) == ((p + 1) % r)
            assert np.all(_f32(cache[b, i])[hit] == 0.25)
            assert np.all(_f32(cache[b, i])[~hit] == 0.0)


def test_closed_form_chain_gumbel_class():
    # With bias 64 on the class v = p + 1 (mod r) and zero elsewhere, the
    # Gumbel draw (noise < 17) always stays in that class; which member it
    # takes is random.
    V, r, N, rows = 256, 16, 6, 4
    head, embed = _closed_form_weights(V, r, 8.0)
    base = np.zeros((rows, N, V), dtype=np.uint16)
    anchor = np.array([5, 200, 0, 15], dtype=np.int32)
    toks, _ = oracle.chain(base, head, embed, anchor, np.full(rows, 1.0, np.float32),
                           np.arange(rows) + 11, np.arange(rows), GUMBEL)
    for b in range(rows):
        p = int(anchor[b])
        for i in range(N):
            assert toks[b, i] % r == (p + 1) % r
            p = int(toks[b, i])
    assert len(set(toks.ravel().tolist())) > N  # members vary


def test_bias_matches_fp64_dot_except_near_ties():
    rng = np.random.default_rng(2)
    V, r = 4000, 256
    head = _bf16(rng.standard_normal((V, r)) * 0.02)
    embed = _bf16(rng.standard_normal((8, r)) * 0.02)
    h64 = _f32(head).astype(np.float64)
    e64 = _f32(embed).astype(np.float64)
    mism = 0
    for p in range(8):
        ours = oracle.bias_all(head, embed, p)
        exact = h64 @ e64[p]
        ref = _bf16(exact.astype(np.float32))
        diff = ours != ref
        if diff.any():
            # only where the exact sum sits within fp32 accumulation error of a
            # BF16 rounding midpoint, and then by one BF16 ulp
            o = _f32(ours[diff]).astype(np.float64)
            rf = _f32(ref[diff]).astype(np.float64)
            mid = (o + rf) / 2
            bound = r * 2.0**-24 * np.abs(h64 * e64[p]).sum(axis=1)[diff] + 1e-30
            assert np.all(np.abs(exact[diff] - mid) <= bound)
            ulp = np.abs(ours[diff].astype(np.int32) - ref[diff].astype(np.int32))
            assert np.all(ulp == 1)
            mism += int(diff.sum())
    assert mism <= V * 8 * 0.001


def test_soft_cap_matches_fp64_except_near_ties():
    # l = bf16(30 tanh(0.5 s / 30)) for every finite BF16 s in [-2^9, 2^9].
    s_all = np.arange(0, 1 << 16, dtype=np.uint16)
    sf = _f32(s_all)
    keep = np.isfinite(sf) & (np.abs(sf) <= 512)
    s_bits = s_all[keep]
    ours = np.array([oracle.logit(int(b), 0, mult=0.5, cap=30.0) for b in s_bits],
                    dtype=np.uint16)
    x64 = _f32(s_bits).astype(np.float64)
    y64 = 30.0 * np.tanh(0.5 * x64 / 30.0)
    ref = torch.from_numpy(y64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    diff = ours != ref
    # halving a BF16 subnormal lands exactly on a rounding midpoint: those
    # are ties by construction; among normal values mismatches are rare
    assert (diff & (np.abs(x64) >= 2.0**-120)).sum() <= 8
    if diff.any():
        o = _f32(ours[diff]).astype(np.float64)
        rf = _f32(ref[diff]).astype(np.float64)
        mid = (o + rf) / 2
        assert np.all(np.abs(y64[diff] - mid) <= 1e-6 * np.abs(mid))


def test_multiplier_only_transform():
    rng = np.random.default_rng(9)
    s = _bf16(rng.standard_normal(5000) * 4)
    ours = np.array([oracle.logit(int(b), 0, mult=0.5) for b in s], dtype=np.uint16)
    assert np.array_equal(ours, _bf16(_f32(s) * np.float32(0.5)))
    same = np.array([oracle.logit(int(b), 0, mult=1.0) for b in s], dtype=np.uint16)
    assert np.array_equal(same, s)


def test_greedy_rows_pick_argmax_of_written_cache():
    w = W.small(777, 32, 5, 4, GUMBEL, seed=3, temperatures=(0.0,), spikes=2)
    base, head, embed, anchor, temp, seeds, idx = _inputs(w)
    toks, cache = oracle.chain(base, head, embed, anchor, temp, seeds, idx, GUMBEL)
    for b in range(w.rows):
        for i in range(w.steps):
            lf = _f32(cache[b, i])
            assert toks[b, i] == int(np.argmax(np.where(lf == 0, 0.0, lf)))


def test_padding_rows_are_inert():
    w = W.small(300, 16, 6, 3, INVCDF, seed=4, padding_rows=(1, 4))
    base, head, embed, anchor, temp, seeds, idx = _inputs(w)
    toks0 = np.full((6, 3), -7, dtype=np.int64)
    cache0 = np.full((6, 3, 300), 0xABCD, dtype=np.uint16)
    toks, cache = oracle.chain(base, head, embed, anchor, temp, seeds, idx, INVCDF,
                               tokens=toks0.copy(), cache=cache0.copy())
    for b in (1, 4):
        assert np.all(toks[b] == -7) and np.all(cache[b] == 0xABCD)
    for b in (0, 2, 3, 5):
        assert np.all(toks[b] >= 0) and not np.any(cache[b] == 0xABCD)


@pytest.mark.parametrize("mode", [GUMBEL, INVCDF])
def test_restart_mid_chain_reproduces_tail(mode):
    w = W.small(500, 32, 4, 6, mode, seed=5, temperatures=(0.0, 0.7, 1.0))
    base, head, embed, anchor, temp, seeds, idx = _inputs(w)
    toks, cache = oracle.chain(base, head, embed, anchor, temp, seeds, idx, mode)
    for k in range(1, 6):
        ss = np.full(4, k, dtype=np.int32)
        sp = toks[:, k - 1].copy()
        t2, c2 = oracle.chain(base, head, embed, anchor, temp, seeds, idx, mode,
                              start_step=ss, start_prev=sp)
        assert np.array_equal(t2[:, k:], toks[:, k:])
        assert np.array_equal(c2[:, k:], cache[:, k:])


def test_noise_independent_of_chain():
    # Changing the base logits and the head changes the chain but never the
    # noise: the Gumbel key of the drawn token is its logit / T plus the
    # noise of (seed, row, step, token) alone.
    w = W.small(400, 16, 2, 4, GUMBEL, seed=6, temperatures=(1.0,))
    base, head, embed, anchor, temp, seeds, idx = _inputs(w)
    for variant in range(2):
        if variant:
            head = _bf16(_f32(head) * 2)
            base = _bf16(_f32(base) + 1)
        toks, cache = oracle.chain(base, head, embed, anchor, temp, seeds, idx, GUMBEL)
        for b in range(2):
            for i in range(4):
                g = oracle.gumbel(int(seeds[b]), b, i, 0, 400)
                keys = _f32(cache[b, i]) / np.float32(temp[b]) + g
                assert toks[b, i] == int(np.argmax(keys))


def test_tiny_workload_golden():
    # Regression against the stored output of the committed golden script.
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny_chain.txt")
    want = [int(t) for t in open(path).read().split("tokens:")[1].split()]
    base, head, embed, anchor, temp, seeds, idx = _inputs(W.TINY)
    toks, _ = oracle.chain(base, head, embed, anchor, temp, seeds, idx, W.TINY.mode)
    assert toks.ravel().tolist() == want
