"""One whole draft step as a serving loop runs it (sharded_markov page, module
docstring: the backbone produces the base logits of the N draft positions,
then the chain draws the tokens; fork_noise / join_noise: the Gumbel noise
is drawn on a side stream meanwhile).

A synthetic draft LM head computes the base logits on the main stream
(hidden [rows * N, H] times lm_head [V, H] transposed: a plain library GEMM,
not part of the sampling path) while markov_noise_fork draws the noise on
the plan's side stream; markov_noise_join and markov_chain_sample follow.
The whole step is captured in one CUDA graph.  Replays on new inputs must
equal eager steps bit for bit, and every step's tokens and cache must pass
the oracle acceptance check on the base logits the GEMM produced."""
import numpy as np
import pytest
import torch

from draft_token_markov_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

H = 512   # hidden size of the synthetic draft model


def _inputs(w, k):
    call = W.make_call(w.with_(gen_seed=w.gen_seed + k))
    g = torch.Generator().manual_seed(500 + k)
    hidden = torch.randn(w.rows * w.steps, H, generator=g).to(torch.bfloat16)
    return call, hidden


@pytest.mark.parametrize("rows", [8, 20], ids=["chain", "per-position"])
def test_draft_step_with_lm_head_in_one_graph(gpu_lib, rows):
    api = gpu_lib
    w = W.small(16384, 256, rows, 8, W.GUMBEL, seed=71, padding_rows=(2,), spikes=4,
                temperatures=(0.0, 0.6, 1.0))
    V, N = w.vocab, w.steps
    h, e = W.make_weights(w)
    head, embed = h.cuda(), e.cuda()
    lm_head = (torch.randn(V, H, generator=torch.Generator().manual_seed(77)) * 0.08) \
        .to(torch.bfloat16).cuda()
    plan = api.Plan(V, w.rank, N, rows)
    try:
        call0, hid0 = _inputs(w, 0)
        st = U.to_dev({k: v for k, v in call0.items() if k != "base"})
        hidden = hid0.cuda()
        base = torch.empty((rows * N, V), dtype=torch.bfloat16, device="cuda")
        toks, cache = U.sentinel_outputs(rows, N, V)

        def step(stream):
            api.markov_noise_fork(plan, st["seeds"], st["temperature"], st["row_state_idx"],
                                  stream)
            torch.matmul(hidden, lm_head.t(), out=base)
            api.markov_noise_join(plan, stream)
            api.markov_chain_sample(plan, base.view(rows, N, V), head, embed, st["anchor"],
                                    st["temperature"], st["seeds"], st["row_state_idx"],
                                    w.mode, w.mult, w.cap, toks, cache, stream)

        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            step(s)                                          # warm-up (plan, GEMM handles)
        torch.cuda.synchronize()
        assert api.markov_plan_status(plan) == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                step(s)
        torch.cuda.synchronize()

        for k in range(3):
            call, hid = _inputs(w, k)
            for key in st:
                st[key].copy_(call[key].cuda())
            hidden.copy_(hid.cuda())
            toks.fill_(U.SENT_T)
            g.replay()
            torch.cuda.synchronize()
            assert api.markov_plan_status(plan) == 0
            got_t = toks.cpu().numpy()
            got_c = cache.view(torch.int16).cpu().numpy().view(np.uint16)
            # the base logits this step sampled from, as the GEMM wrote them
            inp = dict(call, base=base.view(rows, N, V).cpu())
            rep = U.check(w, inp, got_t, got_c)
            assert rep.ok(), (k, rep.summary())
            # an eager step on the same inputs gives the same bits
            toks.fill_(U.SENT_T)
            with torch.cuda.stream(s):
                step(s)
            torch.cuda.synchronize()
            assert np.array_equal(toks.cpu().numpy(), got_t)
            assert np.array_equal(cache.view(torch.int16).cpu().numpy().view(np.uint16), got_c)
        assert plan.query(api.Q_LAST_PATH) == (1 if rows <= 8 else 2)
    finally:
        plan.close()
