"""Helpers for the GPU tests: run the CUDA path through the C ABI on a
workload and collect its outputs as numpy arrays."""
from __future__ import annotations

import functools
import os

import numpy as np
import torch

import oracle
from draft_token_markov_gb300 import workloads as W

SENT_T = -7
SENT_C = 0xABCD
NTHREADS = os.cpu_count() or 1


@functools.lru_cache(maxsize=4)
def weights(w: W.Workload):
    head, embed = W.make_weights(w)
    return head, embed, oracle.bf16_bits(head), oracle.bf16_bits(embed)


def to_dev(inp: dict) -> dict:
    return {k: v.cuda() for k, v in inp.items()}


def sentinel_outputs(R, N, V):
    toks = torch.full((R, N), SENT_T, dtype=torch.int64, device="cuda")
    cache = torch.full((R, N, V), SENT_C - 65536, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return toks, cache


def run(api, w: W.Workload, inp: dict, path: int = 0, plan=None, fork: bool = False,
        head=None, embed=None):
    if head is None:
        h, e, _, _ = weights(w)
        head, embed = h.cuda(), e.cuda()
    own = plan is None
    if own:
        plan = api.Plan(w.vocab, w.rank, w.steps, max(w.rows, 1))
    plan.set_path(path)
    d = to_dev(inp)
    toks, cache = sentinel_outputs(w.rows, w.steps, w.vocab)
    if fork:
        api.markov_noise_fork(plan, d["seeds"], d["temperature"], d["row_state_idx"])
    api.markov_chain_sample(plan, d["base"], head, embed, d["anchor"], d["temperature"],
                            d["seeds"], d["row_state_idx"], w.mode, w.mult, w.cap, toks, cache)
    st = api.markov_plan_status(plan)
    assert st == 0, f"device status {st}"
    out = (toks.cpu().numpy(), cache.view(torch.int16).cpu().numpy().view(np.uint16))
    if own:
        plan.close()
    return out


def check(w: W.Workload, inp: dict, toks, cache):
    from tests.acceptance import check as _check
    _, _, hb, eb = weights(w)
    return _check(inp, hb, eb, w.mode, w.mult, w.cap, toks, cache, SENT_T, SENT_C,
                  nthreads=NTHREADS)
