"""Host-resident inputs and tokens (include/markov.h, markov_chain_sample):
pinned CPU tensors for the base logits, anchors, temperatures, seeds,
row_state_idx and draft_tokens, read and written by the kernels over the
host link, give the same outputs bit for bit as device-resident ones, on
every path."""
import numpy as np
import pytest
import torch

from draft_token_markov_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

AUTO, CHAIN, BATCH, SIMPLE = 0, 1, 2, 3

CASES = [
    ("tcgen05 chain", W.small(12000, 256, 8, 4, W.GUMBEL, seed=91, padding_rows=(2,), spikes=3,
                              temperatures=(0.0, 0.6, 1.0)), CHAIN, False),
    ("tcgen05 chain, inverse CDF, capped", W.small(8192, 128, 4, 3, W.INVCDF, seed=92, spikes=2,
                                                   mult=0.5, cap=30.0), CHAIN, False),
    ("simple chain", W.small(5008, 128, 6, 4, W.GUMBEL, seed=93, padding_rows=(1,)), SIMPLE, False),
    ("batch, inverse CDF", W.small(4096, 256, 40, 3, W.INVCDF, seed=94, padding_rows=(3, 17),
                                   temperatures=(0.0, 0.8, 1.0)), BATCH, False),
    ("batch, Gumbel, fp32 base", W.small(3008, 64, 12, 3, W.GUMBEL, seed=95, padding_rows=(4,)),
     BATCH, True),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_host_resident_inputs_match_device_inputs(gpu_lib, case):
    name, w, path, base_f32 = CASES[case]
    inp = W.make_call(w, base_f32=base_f32)
    h, e, _, _ = U.weights(w)
    head, embed = h.cuda(), e.cuda()
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    try:
        plan.set_path(path)
        outs = []
        for where in ("device", "host"):
            src = ({k: v.cuda() for k, v in inp.items()} if where == "device"
                   else {k: v.pin_memory() for k, v in inp.items()})
            toks = torch.full((w.rows, w.steps), U.SENT_T, dtype=torch.int64)
            toks = toks.cuda() if where == "device" else toks.pin_memory()
            cache = torch.full((w.rows, w.steps, w.vocab), U.SENT_C - 65536, dtype=torch.int16,
                               device="cuda").view(torch.bfloat16)
            gpu_lib.markov_chain_sample(plan, src["base"], head, embed, src["anchor"],
                                        src["temperature"], src["seeds"], src["row_state_idx"],
                                        w.mode, w.mult, w.cap, toks, cache)
            assert gpu_lib.markov_plan_status(plan) == 0
            outs.append((toks.cpu().numpy().copy(),
                         cache.view(torch.int16).cpu().numpy().view(np.uint16)))
        assert np.array_equal(outs[0][0], outs[1][0]), name
        assert np.array_equal(outs[0][1], outs[1][1]), name
        if not base_f32:
            rep = U.check(w, inp, *outs[1])
            assert rep.ok(), (name, rep.summary())
    finally:
        plan.close()


def test_pageable_cpu_tensors_are_refused(gpu_lib):
    w = W.small(4096, 64, 2, 2, W.GUMBEL, seed=96)
    inp = W.make_call(w)
    h, e, _, _ = U.weights(w)
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    try:
        d = {k: v.cuda() for k, v in inp.items()}
        with pytest.raises(TypeError):
            gpu_lib.markov_chain_sample(plan, inp["base"], h.cuda(), e.cuda(), d["anchor"],
                                        d["temperature"], d["seeds"], d["row_state_idx"],
                                        w.mode, w.mult, w.cap)
    finally:
        plan.close()
