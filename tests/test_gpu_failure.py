"""Failure detection on the GPU without faulting it: the kernels' bounded
waits give up and report MARKOV_ETIMEOUT, and a status planted on the host
(as a failing kernel would record it) makes the next call return without
writing outputs, after which the plan works again."""
import time

import numpy as np
import pytest
import torch

from draft_token_markov_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

ETIMEOUT = 4


@pytest.mark.parametrize("which", [0, 1], ids=["grid_barrier", "mbarrier"])
def test_bounded_wait_gives_up(gpu_lib, which):
    t0 = time.perf_counter()
    st = gpu_lib.markov_selftest_wait(which, 2000)
    el = time.perf_counter() - t0
    assert st == ETIMEOUT
    assert el < 5.0
    # the context is still usable: a normal call after it passes parity
    w = W.TINY
    inp = W.make_call(w)
    toks, cache = U.run(gpu_lib, w, inp)
    rep = U.check(w, inp, toks, cache)
    assert rep.ok(), rep.summary()


def test_planted_status_aborts_the_next_call(gpu_lib):
    w = W.TINY.with_(rows=2, temperatures=(0.0, 1.0))
    h, e, _, _ = U.weights(w)
    head, embed = h.cuda(), e.cuda()
    inp = W.make_call(w)
    d = U.to_dev(inp)
    plan = gpu_lib.Plan(w.vocab, w.rank, w.steps, w.rows)
    try:
        gpu_lib.markov_plan_inject_status(plan, ETIMEOUT, 0x1234)
        toks, cache = U.sentinel_outputs(w.rows, w.steps, w.vocab)
        gpu_lib.markov_chain_sample(plan, d["base"], head, embed, d["anchor"], d["temperature"],
                                    d["seeds"], d["row_state_idx"], w.mode, w.mult, w.cap,
                                    toks, cache)
        assert gpu_lib.markov_plan_status(plan) == ETIMEOUT
        # no output was written
        assert (toks.cpu().numpy() == U.SENT_T).all()
        c = cache.view(torch.int16).cpu().numpy().view(np.uint16)
        assert (c == U.SENT_C).all()
        # the status was cleared: the same plan computes the call again
        toks2, cache2 = U.run(gpu_lib, w, inp, plan=plan)
        rep = U.check(w, inp, toks2, cache2)
        assert rep.ok(), rep.summary()
    finally:
        plan.close()


def test_inject_status_rejects_ok(gpu_lib):
    plan = gpu_lib.Plan(4096, 64, 4, 1)
    try:
        with pytest.raises(gpu_lib.MarkovError):
            gpu_lib.markov_plan_inject_status(plan, 0)
    finally:
        plan.close()
