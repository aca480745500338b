"""Parity of the fp32 base-logit and fp32 cache variants (the
sharded_markov page's chain compiled per base and cache dtype, BF16 or
fp32; cache_round rounds each logit to the cache's dtype) against the
oracle's typed chain, through the C ABI, on the tcgen05 chain, the simple
persistent chain (up to 8 rows) and the per-position kernels (more rows), both modes,
ragged vocabulary tails (V a multiple of 16, not of 128), padding rows and, for the batch path, a soft cap."""
import numpy as np
import pytest
import torch

from draft_token_markov_gb300 import workloads as W
from tests import gpu_util as U
from tests.acceptance import check_typed

pytestmark = pytest.mark.gpu

AUTO, CHAIN, BATCH, SIMPLE = 0, 1, 2, 3
SENT_F32_BITS = 0x7FABCDEF          # a NaN pattern the kernels never write


def _run_typed(api, w, inp, path, cache_f32):
    h, e, _, _ = U.weights(w)
    head, embed = h.cuda(), e.cuda()
    plan = api.Plan(w.vocab, w.rank, w.steps, max(w.rows, 1))
    try:
        plan.set_path(path)
        d = U.to_dev(inp)
        toks = torch.full((w.rows, w.steps), U.SENT_T, dtype=torch.int64, device="cuda")
        if cache_f32:
            cache = torch.full((w.rows, w.steps, w.vocab), SENT_F32_BITS, dtype=torch.int32,
                               device="cuda").view(torch.float32)
        else:
            cache = torch.full((w.rows, w.steps, w.vocab), U.SENT_C - 65536, dtype=torch.int16,
                               device="cuda").view(torch.bfloat16)
        api.markov_chain_sample(plan, d["base"], head, embed, d["anchor"], d["temperature"],
                                d["seeds"], d["row_state_idx"], w.mode, w.mult, w.cap, toks,
                                cache)
        assert api.markov_plan_status(plan) == 0
        t = toks.cpu().numpy()
        c = (cache.cpu().numpy() if cache_f32
             else cache.view(torch.int16).cpu().numpy().view(np.uint16))
        return t, c
    finally:
        plan.close()


CASES = [
    # (name, workload, path)
    ("tcgen05 chain", lambda mode: W.small(12000, 256, 8, 4, mode, seed=70, padding_rows=(2, 5),
                                           spikes=4, temperatures=(0.0, 0.6, 1.0)), CHAIN),
    ("tcgen05 chain, rank 128, capped", lambda mode: W.small(6000, 128, 4, 3, mode, seed=76,
                                                             spikes=2, mult=0.5, cap=30.0), CHAIN),
    ("chain", lambda mode: W.small(5008, 128, 6, 4, mode, seed=71, padding_rows=(1,), spikes=3,
                                   temperatures=(0.0, 0.7, 1.0)), SIMPLE),
    ("auto", lambda mode: W.small(4096, 64, 3, 3, mode, seed=72, spikes=2), AUTO),
    ("batch", lambda mode: W.small(3008, 64, 12, 3, mode, seed=73, padding_rows=(4, 9),
                                   spikes=2, mult=0.5, cap=30.0,
                                   temperatures=(0.0, 0.8, 1.0)), BATCH),
    # 13 rows: two tcgen05 chain slices in Gumbel mode, the per-position
    # kernels (16-row groups) in inverse-CDF mode
    ("auto, 13 rows", lambda mode: W.small(8192, 256, 13, 3, mode, seed=74, padding_rows=(6,),
                                           spikes=2, temperatures=(0.0, 0.6, 1.0)), AUTO),
]


@pytest.mark.parametrize("base_f32,cache_f32", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("mode", [W.GUMBEL, W.INVCDF])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_typed_variants_match_the_oracle(gpu_lib, base_f32, cache_f32, mode, case):
    name, mk, path = CASES[case]
    w = mk(mode)
    inp = W.make_call(w, base_f32=base_f32)
    toks, cache = _run_typed(gpu_lib, w, inp, path, cache_f32)
    _, _, hb, eb = U.weights(w)
    rep = check_typed(inp, hb, eb, w.mode, w.mult, w.cap, toks, cache, cache_f32, U.SENT_T,
                      SENT_F32_BITS if cache_f32 else U.SENT_C, nthreads=U.NTHREADS)
    assert rep.ok(), (name, rep.summary())


def test_bf16_through_the_typed_entry_equals_the_bf16_call(gpu_lib):
    w = W.small(4112, 128, 5, 3, W.GUMBEL, seed=74, padding_rows=(2,), spikes=2)
    inp = W.make_call(w)
    a = _run_typed(gpu_lib, w, inp, SIMPLE, False)
    b = U.run(gpu_lib, w, inp, SIMPLE)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("base_f32,cache_f32", [(True, True), (False, True)])
def test_typed_full_deepseek_shape(gpu_lib, base_f32, cache_f32):
    # the DeepSeek-V4.1-shaped chain (V=129280, r=256, 8 rows, 2 padding,
    # N=8, Gumbel) with an fp32 cache on the tcgen05 chain; the record logs
    # how often the fp32-cache rule needed a bias beyond one ulp
    from tests import acceptance as A
    w = W.DEEPSEEK
    inp = W.make_call(w, base_f32=base_f32)
    toks, cache = _run_typed(gpu_lib, w, inp, CHAIN, cache_f32)
    _, _, hb, eb = U.weights(w)
    rep = check_typed(inp, hb, eb, w.mode, w.mult, w.cap, toks, cache, cache_f32, U.SENT_T,
                      SENT_F32_BITS, nthreads=U.NTHREADS)
    A.log(f"deepseek {'f32' if base_f32 else 'bf16'} base, f32 cache (chain path)", rep)
    assert rep.ok(), rep.summary()


def test_typed_rule_needs_no_wide_bias_without_cancellation(gpu_lib):
    # head and embed with non-negative entries: no dot product cancels, so
    # every fp32 cache element is the oracle's or its bias one ulp away
    w = W.small(12000, 256, 8, 3, W.GUMBEL, seed=77, padding_rows=(5,),
                temperatures=(0.0, 0.6, 1.0))
    h, e, _, _ = U.weights(w)
    h, e = h.float().abs().to(torch.bfloat16), e.float().abs().to(torch.bfloat16)
    import oracle
    hb, eb = oracle.bf16_bits(h), oracle.bf16_bits(e)
    inp = W.make_call(w)
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    try:
        plan.set_path(CHAIN)
        d = U.to_dev(inp)
        toks = torch.full((w.rows, w.steps), U.SENT_T, dtype=torch.int64, device="cuda")
        cache = torch.full((w.rows, w.steps, w.vocab), SENT_F32_BITS, dtype=torch.int32,
                           device="cuda").view(torch.float32)
        gpu_lib.markov_chain_sample(plan, d["base"], h.cuda(), e.cuda(), d["anchor"],
                                    d["temperature"], d["seeds"], d["row_state_idx"], w.mode,
                                    w.mult, w.cap, toks, cache)
        assert gpu_lib.markov_plan_status(plan) == 0
        t, c = toks.cpu().numpy(), cache.cpu().numpy()
    finally:
        plan.close()
    rep = check_typed(inp, hb, eb, w.mode, w.mult, w.cap, t, c, True, U.SENT_T, SENT_F32_BITS,
                      nthreads=U.NTHREADS)
    assert rep.ok(), rep.summary()
    assert rep.cache_bias_wide == 0, rep.summary()
