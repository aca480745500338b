"""The vocabulary-sharded chain (sharded_markov page, module docstring and
"Per call" diagram) with its ranks emulated on one GPU, through the C ABI:
every rank's tokens and full-vocabulary cache against the oracle's
(unsharded) chain, and bit for bit against the single-GPU simple chain,
which computes the same bias tiles."""
import numpy as np
import pytest
import torch

from draft_token_markov_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

SIMPLE = 3


def _shards(head, world):
    # each rank's head rows in an allocation of its own
    V = head.shape[0]
    return [head[k * V // world:(k + 1) * V // world].clone().cuda() for k in range(world)]


def _run_sharded(api, w, inp, world, timeout_ms=0):
    h, e, _, _ = U.weights(w)
    heads = _shards(h, world)
    embed = e.cuda()
    d = U.to_dev(inp)
    plan = api.ShardPlan(w.vocab, w.rank, w.steps, max(w.rows, 1), world, timeout_ms=timeout_ms)
    try:
        outs = [U.sentinel_outputs(w.rows, w.steps, w.vocab) for _ in range(world)]
        toks = [o[0] for o in outs]
        caches = [o[1] for o in outs]
        api.markov_chain_sample_sharded(plan, d["base"], heads, embed, d["anchor"],
                                        d["temperature"], d["seeds"], d["row_state_idx"],
                                        w.mult, w.cap, toks, caches)
        st = api.markov_shard_plan_status(plan)
        assert st == 0, f"device status {st}"
        return [(t.cpu().numpy(), c.view(torch.int16).cpu().numpy().view(np.uint16))
                for t, c in zip(toks, caches)]
    finally:
        plan.close()


CASES = [
    # (workload, worlds)
    (W.small(12288, 256, 8, 4, W.GUMBEL, seed=81, padding_rows=(2, 5), spikes=4,
             temperatures=(0.0, 0.6, 1.0)), (1, 2, 4, 8)),
    (W.small(8192, 128, 5, 3, W.GUMBEL, seed=82, spikes=2, mult=0.5, cap=30.0), (2, 8)),
    (W.small(4096, 64, 3, 5, W.GUMBEL, seed=83, padding_rows=(1,)), (4,)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_sharded_ranks_match_the_oracle(gpu_lib, case):
    w, worlds = CASES[case]
    inp = W.make_call(w)
    ref = U.run(gpu_lib, w, inp, SIMPLE)
    rep = U.check(w, inp, *ref)
    assert rep.ok(), rep.summary()
    for world in worlds:
        outs = _run_sharded(gpu_lib, w, inp, world)
        for k, (t, c) in enumerate(outs):
            # the same bias tiles as the simple chain: bit-identical outputs
            assert np.array_equal(t, ref[0]), (world, k)
            assert np.array_equal(c, ref[1]), (world, k)


def test_sharded_deepseek_shape_on_eight_ranks(gpu_lib):
    # the DeepSeek-V4.1-shaped chain (V=129280, r=256, 8 rows, 2 padding,
    # N=8) on 8 ranks of 16160 ids each; every rank's outputs against the
    # oracle through the acceptance rule
    from tests import acceptance as A
    w = W.DEEPSEEK
    inp = W.make_call(w)
    outs = _run_sharded(gpu_lib, w, inp, 8)
    for k, (t, c) in enumerate(outs):
        if k > 0:
            assert np.array_equal(t, outs[0][0]) and np.array_equal(c, outs[0][1]), k
    rep = U.check(w, inp, *outs[0])
    A.log("deepseek, 8 sharded ranks (rank 0; ranks 1-7 equal)", rep)
    assert rep.ok(), rep.summary()


def test_sharded_repeated_calls_share_one_plan(gpu_lib):
    # the epoch tags move with every call: a plan serves many calls
    w = W.small(6144, 128, 4, 3, W.GUMBEL, seed=84, temperatures=(0.6, 1.0))
    h, e, _, _ = U.weights(w)
    heads = _shards(h, 4)
    embed = e.cuda()
    plan = gpu_lib.ShardPlan(w.vocab, w.rank, w.steps, w.rows, 4)
    try:
        for call in range(5):
            inp = W.make_call(w, call)
            d = U.to_dev(inp)
            toks, caches = gpu_lib.markov_chain_sample_sharded(
                plan, d["base"], heads, embed, d["anchor"], d["temperature"], d["seeds"],
                d["row_state_idx"], w.mult, w.cap)
            assert gpu_lib.markov_shard_plan_status(plan) == 0
            ref = U.run(gpu_lib, w, inp, SIMPLE)
            for t, c in zip(toks, caches):
                assert np.array_equal(t.cpu().numpy(), ref[0])
                assert np.array_equal(c.view(torch.int16).cpu().numpy().view(np.uint16), ref[1])
    finally:
        plan.close()


def test_sharded_bad_anchor_writes_nothing(gpu_lib):
    w = W.small(4096, 64, 2, 3, W.GUMBEL, seed=85)
    inp = W.make_call(w)
    inp["anchor"][1] = w.vocab + 5          # outside the vocabulary
    h, e, _, _ = U.weights(w)
    heads = _shards(h, 2)
    d = U.to_dev(inp)
    plan = gpu_lib.ShardPlan(w.vocab, w.rank, w.steps, w.rows, 2)
    try:
        outs = [U.sentinel_outputs(w.rows, w.steps, w.vocab) for _ in range(2)]
        gpu_lib.markov_chain_sample_sharded(plan, d["base"], heads, e.cuda(), d["anchor"],
                                            d["temperature"], d["seeds"], d["row_state_idx"],
                                            w.mult, w.cap, [o[0] for o in outs],
                                            [o[1] for o in outs])
        assert gpu_lib.markov_shard_plan_status(plan) == 1      # MARKOV_EINVAL
        for t, c in outs:
            assert (t.cpu().numpy() == U.SENT_T).all()
            assert (c.view(torch.int16).cpu().numpy().view(np.uint16) == U.SENT_C).all()
        # the status read cleared it: the next call on the same plan runs
        inp2 = W.make_call(w)
        d2 = U.to_dev(inp2)
        toks, caches = gpu_lib.markov_chain_sample_sharded(
            plan, d2["base"], heads, e.cuda(), d2["anchor"], d2["temperature"], d2["seeds"],
            d2["row_state_idx"], w.mult, w.cap)
        assert gpu_lib.markov_shard_plan_status(plan) == 0
        ref = U.run(gpu_lib, w, inp2, SIMPLE)
        for t, c in zip(toks, caches):
            assert np.array_equal(t.cpu().numpy(), ref[0])
            assert np.array_equal(c.view(torch.int16).cpu().numpy().view(np.uint16), ref[1])
    finally:
        plan.close()


def test_sharded_plan_rejects_bad_arguments(gpu_lib):
    import ctypes
    from draft_token_markov_gb300 import api
    L = api.lib()
    h = ctypes.c_void_p()
    for vocab, rank, steps, rows, world in ((4096, 64, 4, 8, 3),      # world not 1/2/4/8
                                            (4104, 64, 4, 8, 2),      # V / world not tile-aligned
                                            (4096, 96, 4, 8, 2),      # rank
                                            (4096, 64, 17, 8, 2),     # steps
                                            (4096, 64, 4, 9, 2)):     # rows above the MMA columns
        d = api._Desc(vocab, rank, steps, rows, torch.cuda.current_device(), 0)
        assert L.markov_shard_plan_create(ctypes.byref(d), world, ctypes.byref(h)) == 1
