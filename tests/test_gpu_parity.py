"""Parity of the CUDA path (chain and batch) with the oracle under the
acceptance rule: small shapes spanning several tiles with ragged per-warp and
per-CTA tails, edge cases, and the five full workloads."""
import numpy as np
import pytest
import torch

import oracle
from draft_token_markov_gb300 import workloads as W
from tests import gpu_util as U
from tests import acceptance as A
from tests.acceptance import check_typed

pytestmark = pytest.mark.gpu

AUTO, CHAIN, BATCH, SIMPLE = 0, 1, 2, 3
PATH_NAMES = {AUTO: "auto", CHAIN: "chain", BATCH: "batch", SIMPLE: "simple"}

SMALL = [
    W.small(16, 64, 1, 1, W.GUMBEL, seed=1, temperatures=(1.0,)),
    W.small(272, 64, 3, 4, W.GUMBEL, seed=2),
    W.small(4144, 128, 8, 5, W.GUMBEL, seed=3, padding_rows=(1, 6), spikes=4),
    W.small(12000, 256, 5, 3, W.INVCDF, seed=4, mult=0.5, cap=30.0, tie_row=1, nan_row=2,
            temperatures=(0.7, 1.0)),
    W.small(2048, 64, 8, 16, W.INVCDF, seed=5, temperatures=(0.0,)),
    W.small(3008, 256, 8, 3, W.GUMBEL, seed=6, mult=1.5, temperatures=(0.0, 0.6, 1.0)),
    W.small(5000 - 8, 128, 7, 6, W.INVCDF, seed=7, temperatures=(0.0, 0.5, 1.2),
            padding_rows=(0,)),
]


def _ids(ws):
    return [w.name.replace(" ", "_") for w in ws]


@pytest.mark.parametrize("path", [CHAIN, SIMPLE, BATCH])
@pytest.mark.parametrize("w", SMALL, ids=_ids(SMALL))
def test_small_parity(gpu_lib, w, path):
    inp = W.make_call(w)
    toks, cache = U.run(gpu_lib, w, inp, path)
    rep = U.check(w, inp, toks, cache)
    assert rep.ok(), rep.summary()


BATCHES = [
    W.small(3008, 256, 20, 3, W.GUMBEL, seed=8, padding_rows=(3, 19)),
    W.small(1024, 128, 70, 2, W.INVCDF, seed=9, temperatures=(0.0, 0.8, 1.0)),
    W.small(512, 64, 256, 2, W.GUMBEL, seed=10),
    # two 64-row groups of the tcgen05 logits kernel, CTAs with a full tile
    # pair and a ragged last tile (16400 = 128 x 128 + 16), every temperature
    W.small(16400, 256, 100, 3, W.INVCDF, seed=11, padding_rows=(5, 64, 99),
            temperatures=(0.0, 0.5, 0.8, 1.0, 1.2), spikes=2),
    W.small(8192, 128, 130, 2, W.GUMBEL, seed=12, padding_rows=(0, 127),
            temperatures=(0.0, 0.7, 1.0)),
]


@pytest.mark.parametrize("w", BATCHES, ids=_ids(BATCHES))
def test_batch_rows_parity(gpu_lib, w):
    inp = W.make_call(w)
    toks, cache = U.run(gpu_lib, w, inp, AUTO)
    rep = U.check(w, inp, toks, cache)
    assert rep.ok(), rep.summary()


@pytest.mark.parametrize("rows", [9, 16, 21, 24])
def test_chain_row_slices(gpu_lib, rows):
    # between the chain limit and 24 rows, in Gumbel mode, the automatic path
    # runs the tcgen05 chain once per 8-row slice; the noise hash takes the
    # call's row index, so the slices sample what one call would
    w = W.small(8192, 256, rows, 6, W.GUMBEL, seed=80 + rows, padding_rows=(3, rows - 1),
                spikes=4, temperatures=(0.0, 0.6, 1.0))
    inp = W.make_call(w)
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    try:
        toks, cache = U.run(gpu_lib, w, inp, AUTO, plan=plan)
        assert plan.query(gpu_lib.Q_LAST_PATH) == CHAIN
        assert plan.query(gpu_lib.Q_LAST_LAUNCHES) == (rows + 7) // 8
        rep = U.check(w, inp, toks, cache)
        assert rep.ok(), rep.summary()
        # the same call with the noise forked takes the per-position kernels
        toks2, cache2 = U.run(gpu_lib, w, inp, AUTO, plan=plan, fork=True)
        assert plan.query(gpu_lib.Q_LAST_PATH) == BATCH
        rep = U.check(w, inp, toks2, cache2)
        assert rep.ok(), rep.summary()
        # inverse-CDF calls of this size take the per-position kernels
        wc = w.with_(mode=W.INVCDF)
        toks3, cache3 = U.run(gpu_lib, wc, inp, AUTO, plan=plan)
        assert plan.query(gpu_lib.Q_LAST_PATH) == BATCH
        rep = U.check(wc, inp, toks3, cache3)
        assert rep.ok(), rep.summary()
    finally:
        plan.close()


def test_batch_calls_share_one_plan(gpu_lib):
    # the per-position path keeps per-row winner words and done counters in
    # the plan; each call must leave them cleared for the next, whatever its
    # row count or mode
    V, r = 4096, 128
    plan = gpu_lib.Plan(V, r, 4, 70)
    try:
        for k, (rows, mode) in enumerate([(70, W.INVCDF), (20, W.GUMBEL), (70, W.GUMBEL),
                                          (33, W.INVCDF), (70, W.INVCDF)]):
            w = W.small(V, r, rows, 4, mode, seed=60 + k, padding_rows=(1,),
                        temperatures=(0.0, 0.7, 1.0))
            inp = W.make_call(w)
            toks, cache = U.run(gpu_lib, w, inp, BATCH, plan=plan)
            assert plan.query(gpu_lib.Q_LAST_PATH) == BATCH
            # inverse CDF: logits + sum kernels per position; Gumbel: the noise
            # kernel, then one logits kernel per position
            assert plan.query(gpu_lib.Q_LAST_LAUNCHES) == (8 if mode == W.INVCDF else 1 + 4)
            rep = U.check(w, inp, toks, cache)
            assert rep.ok(), (k, rep.summary())
    finally:
        plan.close()


def test_forced_chain_refuses_large_batch(gpu_lib):
    w = BATCHES[0]
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    plan.set_path(CHAIN)
    with pytest.raises(gpu_lib.MarkovError) as e:
        U.run(gpu_lib, w, W.make_call(w), CHAIN, plan=plan)
    assert e.value.code == 2


@pytest.mark.parametrize("path", [CHAIN, SIMPLE, BATCH])
def test_max_vocab_and_steps(gpu_lib, path):
    w = W.small(262144, 64, 2, 16, W.GUMBEL, seed=11, temperatures=(0.0, 1.0))
    inp = W.make_call(w)
    toks, cache = U.run(gpu_lib, w, inp, path)
    rep = U.check(w, inp, toks, cache)
    assert rep.ok(), rep.summary()


@pytest.mark.parametrize("path", [CHAIN, SIMPLE, BATCH])
def test_infinities_and_empty_rows(gpu_lib, path):
    # row 0: every logit -inf (inverse CDF takes id 0); row 1: +inf at two
    # ids (the lowest wins); row 2: a NaN after a +inf (NaN first); row 3:
    # padding.  No soft cap, so infinities pass through.
    w = W.small(1024, 64, 4, 2, W.INVCDF, seed=12, temperatures=(1.0,), padding_rows=(3,))
    inp = W.make_call(w)
    base = inp["base"].float()
    base[0] = float("-inf")
    base[1, :, 700] = float("inf")
    base[1, :, 300] = float("inf")
    base[2, :, 50] = float("inf")
    base[2, :, 900] = float("nan")
    inp["base"] = base.to(torch.bfloat16)
    toks, cache = U.run(gpu_lib, w, inp, path)
    rep = U.check(w, inp, toks, cache)
    assert rep.ok(), rep.summary()
    assert toks[0].tolist() == [0, 0]
    assert toks[1].tolist() == [300, 300]
    assert toks[2].tolist() == [900, 900]
    for mode_w in (w.with_(mode=W.GUMBEL),):
        toks, cache = U.run(gpu_lib, mode_w, inp, path)
        assert U.check(mode_w, inp, toks, cache).ok()
        assert toks[1].tolist() == [300, 300] and toks[2].tolist() == [900, 900]


def test_closed_form_chain_on_gpu(gpu_lib):
    # head[v] = c e_{v mod r}, embed[p] = c e_{(p+1) mod r}, zero base, T = 0:
    # the tokens walk (anchor + 1 + i) mod r.
    V, r, N = 512, 64, 8
    head = torch.zeros(V, r)
    embed = torch.zeros(V, r)
    for v in range(V):
        head[v, v % r] = 0.5
        embed[v, (v + 1) % r] = 0.5
    w = W.small(V, r, 3, N, W.GUMBEL, seed=13, temperatures=(0.0,))
    inp = W.make_call(w)
    inp["base"] = torch.zeros_like(inp["base"])
    for path in (CHAIN, SIMPLE, BATCH):
        toks, _ = U.run(gpu_lib, w, inp, path, head=head.to(torch.bfloat16).cuda(),
                        embed=embed.to(torch.bfloat16).cuda())
        for b in range(3):
            a = int(inp["anchor"][b])
            assert toks[b].tolist() == [(a + 1 + i) % r for i in range(N)]


def test_forked_noise_and_repeat_are_identical(gpu_lib):
    w = SMALL[2]
    inp = W.make_call(w)
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    a = U.run(gpu_lib, w, inp, CHAIN, plan=plan)
    b = U.run(gpu_lib, w, inp, CHAIN, plan=plan, fork=True)
    c = U.run(gpu_lib, w, inp, CHAIN, plan=plan)
    for x, y in ((a, b), (a, c)):
        assert np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1])
    plan.close()


def test_repeated_calls_are_deterministic(gpu_lib):
    w = W.DEEPSEEK.with_(vocab=16384)
    inp = W.make_call(w)
    h, e = W.make_weights(w)
    head, embed = h.cuda(), e.cuda()
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    ref = U.run(gpu_lib, w, inp, CHAIN, plan=plan, head=head, embed=embed)
    for _ in range(20):
        out = U.run(gpu_lib, w, inp, CHAIN, plan=plan, head=head, embed=embed)
        assert np.array_equal(out[0], ref[0]) and np.array_equal(out[1], ref[1])
    plan.close()


@pytest.mark.parametrize("name,path", [("tiny", AUTO), ("deepseek", AUTO), ("softcap", AUTO),
                                       ("batch", AUTO), ("deepseek", SIMPLE),
                                       ("softcap", SIMPLE)])
def test_full_workload_parity(gpu_lib, name, path):
    w = W.BY_NAME[name]
    inp = W.make_call(w)
    toks, cache = U.run(gpu_lib, w, inp, path)
    rep = U.check(w, inp, toks, cache)
    A.log(f"{name} ({PATH_NAMES[path]} path)", rep)
    assert rep.ok(), rep.summary()


def test_latency_workload_calls(gpu_lib):
    # the latency workload's calls differ in seed and anchor: 125 of its 1000
    # calls (every 8th), each checked against the oracle
    w = W.LATENCY
    h, e = W.make_weights(w)
    head, embed = h.cuda(), e.cuda()
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    total = A.Report()
    try:
        for call in range(0, 1000, 8):
            inp = W.make_call(w, call)
            toks, cache = U.run(gpu_lib, w, inp, AUTO, plan=plan, head=head, embed=embed)
            total.merge(U.check(w, inp, toks, cache), tag=f"call {call}")
    finally:
        plan.close()
    A.log("latency (125 calls, auto path)", total)
    assert total.positions == 125 * w.steps
    assert total.ok(), total.summary()


def test_tcgen05_chain_takes_the_chain_workloads(gpu_lib):
    # the head of every chain workload fits on chip: the chain path runs the
    # tcgen05 kernel and reports the whole head resident
    for name in ("tiny", "deepseek", "latency", "softcap"):
        w = W.BY_NAME[name]
        plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
        assert plan.query(gpu_lib.Q_RESIDENT_HEAD_BYTES) == w.vocab * w.rank * 2
        inp = W.make_call(w)
        U.run(gpu_lib, w, inp, AUTO, plan=plan)
        assert plan.query(gpu_lib.Q_LAST_PATH) == CHAIN
        assert plan.query(gpu_lib.Q_LAST_LAUNCHES) == 1
        plan.close()


# Inverse-CDF calls of at most 4 rows, where the two row halves of the
# tcgen05 chain's epilogue warps take each accumulator's tiles in turn:
# vocabularies with 5 to 11 tiles per CTA (odd and even counts per
# accumulator, ragged last tiles), every rank, greedy and sampling rows, a
# padding row, the soft cap with a tie and a NaN row; and 5 rows, where the
# halves split the rows again.
TURNS = [
    W.small(107088, 64, 1, 3, W.INVCDF, seed=13, temperatures=(0.7,)),
    W.small(107088, 128, 2, 2, W.INVCDF, seed=14, temperatures=(0.0, 0.6)),
    W.small(129264, 256, 3, 2, W.INVCDF, seed=15, mult=0.5, cap=30.0, tie_row=1, nan_row=2,
            temperatures=(0.7, 1.0)),
    W.small(200016, 128, 4, 2, W.INVCDF, seed=16, padding_rows=(2,), temperatures=(0.5, 1.2)),
    W.small(107088, 128, 5, 2, W.INVCDF, seed=17, temperatures=(0.0, 0.7, 1.0)),
]


@pytest.mark.parametrize("w", TURNS, ids=_ids(TURNS))
def test_inverse_cdf_epilogue_turns(gpu_lib, w):
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    try:
        inp = W.make_call(w)
        toks, cache = U.run(gpu_lib, w, inp, CHAIN, plan=plan)
        assert plan.query(gpu_lib.Q_LAST_PATH) == CHAIN
        rep = U.check(w, inp, toks, cache)
        assert rep.ok(), rep.summary()
    finally:
        plan.close()


def test_bad_arguments_launch_nothing(gpu_lib):
    w = W.TINY
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, 4)
    inp = U.to_dev(W.make_call(w))
    h, e, _, _ = U.weights(w)
    toks, cache = U.sentinel_outputs(1, w.steps, w.vocab)
    L = gpu_lib.lib()
    def call(**kw):
        args = dict(base=inp["base"].data_ptr(), s0=w.steps * w.vocab, s1=w.vocab,
                    head=h.cuda().data_ptr(), embed=e.cuda().data_ptr(),
                    anchor=inp["anchor"].data_ptr(), T=inp["temperature"].data_ptr(),
                    seeds=inp["seeds"].data_ptr(), idx=inp["row_state_idx"].data_ptr(), rows=1,
                    mode=0, mult=1.0, cap=-1.0, toks=toks.data_ptr(), ts0=w.steps,
                    cache=cache.data_ptr(), cs0=w.steps * w.vocab, cs1=w.vocab)
        args.update(kw)
        return L.markov_chain_sample(plan.handle, *args.values(), None)
    assert call(rows=0) == 1
    assert call(rows=5) == 1
    assert call(mode=3) == 1
    assert call(s1=w.vocab - 1) == 1
    assert call(cs1=w.vocab + 1) == 1          # 16-byte row stride of the cache
    assert call(cache=cache.data_ptr() + 2) == 1
    assert call(mult=float("inf")) == 1
    torch.cuda.synchronize()
    assert np.all(toks.cpu().numpy() == U.SENT_T)
    assert call() == 0
    assert gpu_lib.markov_plan_status(plan) == 0
    plan.close()


@pytest.mark.parametrize("path", [CHAIN, BATCH, SIMPLE])
def test_infinite_keys_take_the_lowest_id(gpu_lib, path):
    # inverse CDF at T = 0.5: row 0 has two +inf base logits; row 1 has finite
    # logits near the BF16 maximum whose key l / T overflows to +inf, the
    # largest of them not at the lowest id; row 3 is all -inf (token 0).
    # +inf keys decide the token directly: the lowest id with a +inf key.
    w = W.small(4096, 128, 4, 3, W.INVCDF, seed=90, temperatures=(0.5,))
    inp = W.make_call(w)
    base = inp["base"].float()
    for i in range(w.steps):
        base[0, i, [100, 3000]] = float("inf")
        base[1, i, 500] = 2.9e38
        base[1, i, 2000] = 2.5e38
        base[1, i, 510] = 3.3e38      # same vocab block as 500, larger logit
        base[3, i, :] = float("-inf")
    inp["base"] = base.to(torch.bfloat16)
    toks, cache = U.run(gpu_lib, w, inp, path)
    rep = U.check(w, inp, toks, cache)
    assert rep.ok(), rep.summary()
    assert toks[0].tolist() == [100] * w.steps
    assert toks[1].tolist() == [500] * w.steps
    assert toks[3].tolist() == [0] * w.steps


@pytest.mark.parametrize("path", [AUTO, BATCH])
def test_gumbel_nan_and_tie_rows_above_the_chain_limit(gpu_lib, path):
    # 12 rows in Gumbel mode: the automatic path runs two chain slices, the
    # forced one the per-position kernels (16-row groups); a NaN row takes
    # its lowest NaN id, a tie row's equal maxima the lowest id, and +inf
    # logits win over finite ones
    w = W.small(4096, 128, 12, 4, W.GUMBEL, seed=91, tie_row=3, nan_row=5, padding_rows=(7,),
                temperatures=(0.0, 0.8, 1.0))
    inp = W.make_call(w)
    base = inp["base"].float()
    for i in range(w.steps):
        base[9, i, [40, 2900]] = float("inf")
    inp["base"] = base.to(torch.bfloat16)
    toks, cache = U.run(gpu_lib, w, inp, path)
    rep = U.check(w, inp, toks, cache)
    assert rep.ok(), rep.summary()
    assert toks[9].tolist() == [40] * w.steps


@pytest.mark.parametrize("path", [CHAIN, SIMPLE, BATCH])
@pytest.mark.parametrize("base_f32", [False, True], ids=["bf16 base", "f32 base"])
def test_odd_base_strides(gpu_lib, path, base_f32):
    # base logits as a view with odd row and position strides (elements):
    # the per-position kernels' paired base loads need even strides and
    # take single-element loads here; every path must read the same values
    w = W.small(4096, 128, 5, 3, W.GUMBEL, seed=92, padding_rows=(2,),
                temperatures=(0.0, 0.7, 1.0))
    if path == BATCH:
        w = w.with_(rows=12, padding_rows=(2, 9))
    inp = W.make_call(w, base_f32=base_f32)
    R, N, V = w.rows, w.steps, w.vocab
    big = torch.zeros((R, N, V + 3), dtype=inp["base"].dtype, device="cuda")
    big[:, :, 1:V + 1] = inp["base"].cuda()
    view = big[:, :, 1:V + 1]
    assert view.stride(1) % 2 == 1 and view.stride(0) % 2 == 1
    h, e, hb, eb = U.weights(w)
    plan = gpu_lib.Plan(V, w.rank, N, R)
    try:
        plan.set_path(path)
        d = U.to_dev(inp)
        toks, cache = U.sentinel_outputs(R, N, V)
        gpu_lib.markov_chain_sample(plan, view, h.cuda(), e.cuda(), d["anchor"], d["temperature"],
                                    d["seeds"], d["row_state_idx"], w.mode, w.mult, w.cap, toks,
                                    cache)
        assert gpu_lib.markov_plan_status(plan) == 0
        t = toks.cpu().numpy()
        c = cache.view(torch.int16).cpu().numpy().view(np.uint16)
    finally:
        plan.close()
    if base_f32:
        rep = check_typed(inp, hb, eb, w.mode, w.mult, w.cap, t, c, False, U.SENT_T, U.SENT_C,
                          nthreads=U.NTHREADS)
    else:
        rep = U.check(w, inp, t, c)
    assert rep.ok(), rep.summary()
