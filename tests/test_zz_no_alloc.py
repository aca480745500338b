"""markov_chain_sample_static: the entry point for callers that cannot
allocate device memory (code inside a CUDA graph capture that forbids
allocation, servers drawing every byte from their own pool).  It keeps its
scratch in a static device array instead of a plan.

Called through the C ABI and compared, on two calls in a row, with the
existing entry point's simple chain path, which runs the same kernels: the
outputs must be identical.  Both outputs also pass the oracle's acceptance
check.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from draft_token_markov_gb300 import workloads as W
from tests import acceptance as A
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

SIMPLE = 3


def _static_fn(api):
    L = api.lib()
    f = L.markov_chain_sample_static
    c = ctypes
    P, i32, i64, f32 = c.c_void_p, c.c_int32, c.c_int64, c.c_float
    f.restype = i32
    f.argtypes = [i32, i32, i32, P, i64, i64, P, P, P, P, P, P, i32, i32, f32, f32, P, i64, P,
                  i64, i64, P]
    return f


def _run_static(api, w, inp, head, embed):
    f = _static_fn(api)
    d = U.to_dev(inp)
    toks, cache = U.sentinel_outputs(w.rows, w.steps, w.vocab)
    cap = -1.0 if w.cap is None else float(w.cap)
    st = f(w.vocab, w.rank, w.steps, d["base"].data_ptr(), d["base"].stride(0),
           d["base"].stride(1), head.data_ptr(), embed.data_ptr(), d["anchor"].data_ptr(),
           d["temperature"].data_ptr(), d["seeds"].data_ptr(), d["row_state_idx"].data_ptr(),
           w.rows, w.mode, float(w.mult), cap, toks.data_ptr(), toks.stride(0), cache.data_ptr(),
           cache.stride(0), cache.stride(1), torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"status {st}"
    torch.cuda.synchronize()
    return toks.cpu().numpy(), cache.view(torch.int16).cpu().numpy().view(np.uint16)


def test_static_scratch_entry_point_matches_plan_path(gpu_lib):
    cases = [W.small(4144, 128, 8, 5, W.GUMBEL, seed=31, padding_rows=(1, 6), spikes=4),
             W.small(12000, 256, 5, 3, W.INVCDF, seed=32, mult=0.5, cap=30.0, tie_row=1,
                     nan_row=2, temperatures=(0.7, 1.0))]
    for w in cases:                                   # two calls in a row
        h, e = W.make_weights(w)
        head, embed = h.cuda(), e.cuda()
        inp = W.make_call(w)
        got = _run_static(gpu_lib, w, inp, head, embed)
        ref = U.run(gpu_lib, w, inp, SIMPLE, head=head, embed=embed)
        assert np.array_equal(got[0], ref[0])
        assert np.array_equal(got[1], ref[1])
        rep = U.check(w, inp, *got)
        assert rep.ok(), rep.summary()


def test_static_scratch_inverse_cdf_above_the_noise_limit(gpu_lib):
    # inverse-CDF calls draw no Gumbel noise, so the noise bound does not
    # apply to them: 8 rows x 16 positions x 262144 ids is accepted
    w = W.small(262144, 64, 8, 16, W.INVCDF, seed=34, padding_rows=(5,),
                temperatures=(0.0, 0.8, 1.0))
    h, e = W.make_weights(w)
    inp = W.make_call(w)
    got = _run_static(gpu_lib, w, inp, h.cuda(), e.cuda())
    rep = U.check(w, inp, *got)
    A.log("allocation-free entry, inverse CDF V=262144 rows=8 N=16", rep)
    assert rep.ok(), rep.summary()


def test_static_scratch_rejects_sizes_beyond_its_limit(gpu_lib):
    f = _static_fn(gpu_lib)
    w = W.small(262144, 64, 8, 16, W.GUMBEL, seed=33)   # 8 * 16 * 262144 noise values: too many
    h, e = W.make_weights(w)
    inp = U.to_dev(W.make_call(w))
    toks, cache = U.sentinel_outputs(w.rows, w.steps, w.vocab)
    st = f(w.vocab, w.rank, w.steps, inp["base"].data_ptr(), inp["base"].stride(0),
           inp["base"].stride(1), h.cuda().data_ptr(), e.cuda().data_ptr(),
           inp["anchor"].data_ptr(), inp["temperature"].data_ptr(), inp["seeds"].data_ptr(),
           inp["row_state_idx"].data_ptr(), w.rows, w.mode, 1.0, -1.0, toks.data_ptr(),
           toks.stride(0), cache.data_ptr(), cache.stride(0), cache.stride(1), None)
    assert st == 2
    torch.cuda.synchronize()
    assert np.all(toks.cpu().numpy() == U.SENT_T)
