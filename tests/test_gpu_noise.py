"""The noise kernel is bit-identical to the oracle's noise, and depends on
(seed, row, position, id) only."""
import numpy as np
import pytest
import torch

import oracle
from draft_token_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noise(api, inp, N, V):
    out = api.markov_gumbel_noise(inp["seeds"].cuda(), inp["temperature"].cuda(),
                                  inp["row_state_idx"].cuda(), N, V)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("w", [W.TINY, W.small(4112, 64, 6, 5, seed=1, padding_rows=(1, 4),
                                               temperatures=(0.0, 0.5, 1.0)),
                               W.DEEPSEEK.with_(rows=3, padding_rows=(1,))])
def test_noise_matches_oracle(gpu_lib, w):
    inp = W.make_call(w)
    R, N, V = w.rows, w.steps, w.vocab
    got = _noise(gpu_lib, inp, N, V)
    T = inp["temperature"].numpy()
    idx = inp["row_state_idx"].numpy()
    seeds = inp["seeds"].numpy()
    for b in range(R):
        for i in range(N):
            row = got[b * N + i]
            if idx[b] < 0 or not T[b] > 0:
                assert np.all(np.isnan(row)), "rows without sampling are not written"
                continue
            ref = oracle.gumbel(int(seeds[b]), b, i, 0, V)
            assert np.array_equal(row.view(np.uint32), ref.view(np.uint32))


def test_noise_depends_on_position_only(gpu_lib):
    inp = W.make_call(W.TINY)
    a = _noise(gpu_lib, inp, 4, 4096)
    inp2 = dict(inp)
    inp2["base"] = inp["base"] * 2   # not an input of the noise at all
    b = _noise(gpu_lib, inp2, 4, 4096)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
