"""CUDA-graph capture of a whole draft step (the speculator's FULL graph
mode, the sharded_markov page's module docstring): markov_chain_sample on a
plan is captured once into a torch CUDA graph and replayed on new inputs
copied into the captured buffers.  Each replay must give exactly what an
eager call gives on the same inputs (same kernels), and the plan's
cross-call state (call counter, exchange words of both call parities) must
stay consistent over replays."""
import numpy as np
import pytest
import torch

from draft_token_markov_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _eager(api, w, inp, head, embed, plan):
    d = U.to_dev(inp)
    toks, cache = U.sentinel_outputs(w.rows, w.steps, w.vocab)
    api.markov_chain_sample(plan, d["base"], head, embed, d["anchor"], d["temperature"],
                            d["seeds"], d["row_state_idx"], w.mode, w.mult, w.cap, toks, cache)
    assert api.markov_plan_status(plan) == 0
    return toks.cpu().numpy(), cache.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("rows", [8, 20, 40], ids=["chain", "chain-slices", "per-position"])
@pytest.mark.parametrize("mode", [W.GUMBEL, W.INVCDF])
def test_graph_replays_equal_eager_calls(gpu_lib, mode, rows):
    # 8 rows take the chain kernel; 20 rows three chain launches (8-row
    # slices) in Gumbel mode and the per-position kernels in inverse-CDF
    # mode; 40 rows the per-position kernels, whose launches after the first
    # are programmatic dependent launches (graph edges of that kind once
    # captured)
    api = gpu_lib
    w = W.small(129280, 256, rows, 8, mode, seed=41, padding_rows=(2, 5), spikes=8,
                temperatures=(0.0, 0.6, 1.0))
    h, e = W.make_weights(w)
    head, embed = h.cuda(), e.cuda()
    calls = [W.make_call(w.with_(gen_seed=w.gen_seed + k)) for k in range(3)]
    plan = api.Plan(w.vocab, w.rank, w.steps, w.rows)
    try:
        # static buffers the graph reads and writes
        st = U.to_dev(calls[0])
        toks, cache = U.sentinel_outputs(w.rows, w.steps, w.vocab)
        api.markov_chain_sample(plan, st["base"], head, embed, st["anchor"], st["temperature"],
                                st["seeds"], st["row_state_idx"], w.mode, w.mult, w.cap, toks,
                                cache)                                  # warm-up (maps, plan)
        assert api.markov_plan_status(plan) == 0
        side = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                api.markov_chain_sample(plan, st["base"], head, embed, st["anchor"],
                                        st["temperature"], st["seeds"], st["row_state_idx"],
                                        w.mode, w.mult, w.cap, toks, cache)
        torch.cuda.synchronize()
        for inp in calls:
            for k, v in inp.items():
                st[k].copy_(v.cuda())
            g.replay()
            torch.cuda.synchronize()
            assert api.markov_plan_status(plan) == 0
            got = (toks.cpu().numpy(), cache.view(torch.int16).cpu().numpy())
            ref = _eager(api, w, inp, head, embed, plan)
            assert np.array_equal(got[0], ref[0])
            assert np.array_equal(got[1], ref[1])
    finally:
        plan.close()
