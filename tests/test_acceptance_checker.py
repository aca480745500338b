"""The acceptance checker must accept the oracle's own outputs and reject
planted mistakes (CPU only: the "GPU" outputs here are the oracle's, edited)."""
import numpy as np

import oracle
from draft_token_markov_gb300 import workloads as W
from tests.acceptance import check

SENT_T, SENT_C = -7, 0xABCD


def _run(w):
    head, embed = W.make_weights(w)
    inp = W.make_call(w)
    hb, eb = oracle.bf16_bits(head), oracle.bf16_bits(embed)
    toks = np.full((w.rows, w.steps), SENT_T, dtype=np.int64)
    cache = np.full((w.rows, w.steps, w.vocab), SENT_C, dtype=np.uint16)
    toks, cache = oracle.chain(oracle.bf16_bits(inp["base"]), hb, eb, inp["anchor"].numpy(),
                               inp["temperature"].numpy(), inp["seeds"].numpy(),
                               inp["row_state_idx"].numpy(), w.mode, w.mult, w.cap,
                               tokens=toks, cache=cache)
    return inp, hb, eb, toks, cache


def _chk(w, inp, hb, eb, toks, cache):
    return check(inp, hb, eb, w.mode, w.mult, w.cap, toks, cache, SENT_T, SENT_C)


def test_checker_accepts_oracle_and_rejects_mistakes():
    w = W.small(512, 32, 4, 3, W.GUMBEL, seed=21, padding_rows=(2,), temperatures=(0.0, 1.0))
    inp, hb, eb, toks, cache = _run(w)
    assert _chk(w, inp, hb, eb, toks, cache).ok()
    # a wrong token with an identical cache
    t2 = toks.copy()
    t2[0, 1] = (t2[0, 1] + 1) % 512
    assert not _chk(w, inp, hb, eb, t2, cache).ok()
    # a cache element 2 ulps away
    c2 = cache.copy()
    c2[1, 0, 5] = int(c2[1, 0, 5]) + 2
    assert not _chk(w, inp, hb, eb, toks, c2).ok()
    # a padding row written
    c3 = cache.copy()
    c3[2, 0, 0] = 0
    assert not _chk(w, inp, hb, eb, toks, c3).ok()
    # a 1-ulp cache difference far below the winner is accepted
    c4 = cache.copy()
    row = oracle.bits_to_f32(c4[3, 2])
    j = int(np.argmin(row))
    c4[3, 2, j] = int(c4[3, 2, j]) + (1 if c4[3, 2, j] < 0x8000 else -1)
    rep = _chk(w, inp, hb, eb, toks, c4)
    assert rep.ok() and rep.cache_ulp_diffs == 1


def test_checker_inverse_cdf_softcap():
    w = W.small(400, 64, 3, 4, W.INVCDF, seed=22, mult=0.5, cap=30.0, tie_row=1, nan_row=2,
                temperatures=(0.7, 1.0))
    inp, hb, eb, toks, cache = _run(w)
    assert _chk(w, inp, hb, eb, toks, cache).ok()
    t2 = toks.copy()
    t2[0, 3] = (t2[0, 3] + 3) % 400
    assert not _chk(w, inp, hb, eb, t2, cache).ok()


def test_checker_bias_ulp_rule():
    # A cache element equal to the epilogue of the oracle's bias moved by one
    # BF16 ulp is accepted at any distance; 3 ulps away otherwise is not.
    from tests.acceptance import bf16_nudges
    w = W.small(256, 32, 1, 1, W.GUMBEL, seed=23, temperatures=(1.0,))
    inp, hb, eb, toks, cache = _run(w)
    base = oracle.bf16_bits(inp["base"])
    p = int(inp["anchor"][0])
    planted = 0
    for v in range(256):
        bias = oracle.bias_one(hb, eb, v, p)
        for nb in bf16_nudges(bias)[::2]:
            l = oracle.lib().orc_logit(int(base[0, 0, v]), int(nb), 0, 1.0, 0, 1.0, 1.0)
            if l != cache[0, 0, v] and v != toks[0, 0]:
                c2 = cache.copy()
                c2[0, 0, v] = l
                rep = _chk(w, inp, hb, eb, toks, c2)
                assert rep.ok(), rep.summary()
                planted += 1
                break
        if planted >= 3:
            break
    assert planted >= 1
    c3 = cache.copy()
    v = (int(toks[0, 0]) + 1) % 256
    c3[0, 0, v] = int(c3[0, 0, v]) + (3 if c3[0, 0, v] < 0x7000 else -3)
    assert not _chk(w, inp, hb, eb, toks, c3).ok()


def test_typed_checker_accepts_oracle_and_rejects_mistakes():
    from tests.acceptance import check_typed
    sent_bits = 0x7FABCDEF
    for base_f32, cache_f32 in ((True, True), (False, True), (True, False)):
        w = W.small(512, 32, 3, 3, W.GUMBEL, seed=22, padding_rows=(1,),
                    temperatures=(0.0, 1.0))
        head, embed = W.make_weights(w)
        inp = W.make_call(w, base_f32=base_f32)
        hb, eb = oracle.bf16_bits(head), oracle.bf16_bits(embed)
        base = inp["base"].numpy() if base_f32 else oracle.bf16_bits(inp["base"])
        toks = np.full((w.rows, w.steps), SENT_T, dtype=np.int64)
        if cache_f32:
            cache = np.full((w.rows, w.steps, w.vocab), sent_bits, dtype=np.uint32).view(np.float32)
        else:
            cache = np.full((w.rows, w.steps, w.vocab), SENT_C, dtype=np.uint16)
        toks, cache = oracle.chain_typed(base, hb, eb, inp["anchor"].numpy(),
                                         inp["temperature"].numpy(), inp["seeds"].numpy(),
                                         inp["row_state_idx"].numpy(), w.mode,
                                         cache_f32=cache_f32, tokens=toks, cache=cache)
        sent = sent_bits if cache_f32 else SENT_C

        def chk(t, c):
            return check_typed(inp, hb, eb, w.mode, 1.0, None, t, c, cache_f32, SENT_T, sent)

        assert chk(toks, cache).ok()
        t2 = toks.copy()
        t2[0, 1] = (t2[0, 1] + 1) % 512
        assert not chk(t2, cache).ok()
        c2 = cache.copy()
        if cache_f32:
            c2[2, 0, 5] = c2[2, 0, 5] + np.float32(0.25)       # far beyond any bias change
        else:
            c2[2, 0, 5] = int(c2[2, 0, 5]) + 2
        assert not chk(toks, c2).ok()
        c3 = cache.copy()
        c3[1, 0, 0] = c3[2, 0, 0]                               # a padding row written
        assert not chk(toks, c3).ok()


def test_no_vacuous_report_asserts():
    # asserting a report's bound ok method (no call) is always true: every use
    # must call it, and a report has no truth value of its own
    import pathlib
    import re
    root = pathlib.Path(__file__).resolve().parent.parent
    files = list((root / "tests").glob("*.py")) + [root / "__graft_entry__.py"]
    bad = []
    for f in files:
        for n, line in enumerate(f.read_text().splitlines(), 1):
            if re.search(r"\.ok\b(?!\s*\()", line) and "def ok" not in line:
                bad.append(f"{f.name}:{n}")
    assert not bad, bad
    from tests.acceptance import Report
    try:
        bool(Report())
    except TypeError:
        pass
    else:
        raise AssertionError("a Report must not have a truth value")


def test_typed_relaxation_is_one_ulp_without_cancellation():
    # the fp32-cache rule's wider bias set comes from cancellation only: for
    # dot products whose terms all have one sign it is the oracle's bias one
    # ulp either way, and under cancellation it can be wider
    from tests.acceptance import _bias_candidates, bf16_nudges
    rng = np.random.default_rng(3)
    r = 256
    h = oracle.bf16_rne(np.abs(rng.standard_normal((64, r))).astype(np.float32) * 0.02)
    e = oracle.bf16_rne(np.abs(rng.standard_normal((4, r))).astype(np.float32) * 0.02)
    for v in range(64):
        for p in range(4):
            nb = set(bf16_nudges(oracle.bias_one(h, e, v, p)))
            assert _bias_candidates(h, e, v, p) == nb, (v, p)
    # cancellation: a row and its negation plus a tiny term
    hc = np.concatenate([h[:1, : r // 2], h[:1, : r // 2]], axis=1).copy()
    ec = np.concatenate([e[:1, : r // 2], e[:1, : r // 2] ^ np.uint16(0x8000)], axis=1).copy()
    hc[0, 0] = oracle.bf16_rne(np.array([1e-4], np.float32))[0]
    wide = _bias_candidates(hc, ec, 0, 0)
    assert len(wide) > 3
