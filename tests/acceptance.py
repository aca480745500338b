"""The acceptance rule, checked against the oracle.

  * cache: every element of every live row within 1 BF16 ulp of the oracle
    (ordered-integer distance, +0 == -0), NaN only where the oracle has NaN;
    an element further away must be exactly what the oracle's epilogue gives
    with its BF16 bias moved by one ulp (the licensed difference: the bias
    reduction order may change the bias's last bit).  That case arises under
    cancellation, base ~ -bias, where one bias ulp is many ulps of the sum;
  * always: the oracle's selection applied to the GPU's own cache row gives
    the GPU's token, bit for bit;
  * tokens: equal to the oracle's, except where the GPU's cache row differs
    from the oracle's and (Gumbel / greedy) the GPU's token is a contender:
    nudging each of the two ids' bias by one BF16 ulp either way can bring
    its key up to the oracle winner's key; (inverse CDF) the GPU token is
    what the oracle's selection gives on the GPU's cache.  An excused
    position is reported, and that row's later positions are compared with
    the oracle rerun from the next position with the GPU's token as the
    previous token;
  * padding rows: both outputs still hold the caller's sentinel.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
from oracle import GUMBEL, INVCDF


def ordered_bf16(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def is_nan_bf16(bits: np.ndarray) -> np.ndarray:
    return (bits & 0x7FFF) > 0x7F80


def bf16_nudges(bits: int) -> list[int]:
    """The BF16 value one ulp below, itself, one ulp above (finite inputs)."""
    o = int(ordered_bf16(np.array([bits], dtype=np.uint16))[0])
    out = []
    for d in (-1, 0, 1):
        q = o + d
        out.append((q if q >= 0 else (0x8000 | (-q))) & 0xFFFF)
    return out


@dataclass
class Report:
    """What one check saw.  Besides pass / fail it counts the licensed
    deviations so that they can be reported: cache elements 1 ulp from the
    oracle (cache_1ulp), elements explained only by the oracle's bias moved
    one BF16 ulp (cache_bias_ulp), for fp32 caches elements explained only by
    a bias further inside the fp32 summation bound (cache_bias_wide), and
    every excused token with the oracle's winner / runner-up key margin.
    min_margin is the smallest oracle margin k1 - k2 over all positions whose
    winner a finite key decides (where = (row, position))."""
    positions: int = 0
    cache_elems: int = 0
    cache_ulp_diffs: int = 0
    cache_bias_ulp: int = 0
    cache_bias_wide: int = 0
    excused: list = field(default_factory=list)
    failures: list = field(default_factory=list)
    min_margin: float = float("inf")
    min_margin_at: tuple = ()
    margins_below_1e_3: int = 0

    def ok(self) -> bool:
        return not self.failures

    def __bool__(self):
        raise TypeError("a Report has no truth value: use report.ok()")

    def note_margin(self, b: int, i: int, k1: float, k2: float) -> None:
        m = float(k1) - float(k2)
        if not np.isfinite(m):
            return
        if m < 1e-3:
            self.margins_below_1e_3 += 1
        if m < self.min_margin:
            self.min_margin, self.min_margin_at = m, (b, i)

    def merge(self, other: "Report", tag=None) -> "Report":
        """Fold another check's counts into this one (several calls of one
        workload); `tag` prefixes the other's excused cases and failures."""
        self.positions += other.positions
        self.cache_elems += other.cache_elems
        self.cache_ulp_diffs += other.cache_ulp_diffs
        self.cache_bias_ulp += other.cache_bias_ulp
        self.cache_bias_wide += other.cache_bias_wide
        pre = () if tag is None else (tag,)
        self.excused += [pre + tuple(e) for e in other.excused]
        self.failures += [pre + tuple(f) for f in other.failures]
        self.margins_below_1e_3 += other.margins_below_1e_3
        if other.min_margin < self.min_margin:
            self.min_margin, self.min_margin_at = other.min_margin, pre + tuple(other.min_margin_at)
        return self

    def record(self) -> dict:
        return {"ok": self.ok(), "positions": self.positions, "cache_elems": self.cache_elems,
                "cache_1ulp": self.cache_ulp_diffs, "cache_bias_ulp": self.cache_bias_ulp,
                "cache_bias_wide": self.cache_bias_wide, "excused": len(self.excused),
                "excused_cases": [list(e) for e in self.excused[:20]],
                "min_margin": self.min_margin if np.isfinite(self.min_margin) else None,
                "min_margin_at": list(self.min_margin_at),
                "margins_below_1e-3": self.margins_below_1e_3,
                "failures": [list(map(str, f)) for f in self.failures[:5]]}

    def summary(self) -> str:
        mm = f"{self.min_margin:.3g}" if np.isfinite(self.min_margin) else "none"
        return (f"positions={self.positions} cache_elems={self.cache_elems} "
                f"cache_1ulp={self.cache_ulp_diffs} cache_bias_ulp={self.cache_bias_ulp} "
                f"cache_bias_wide={self.cache_bias_wide} excused={len(self.excused)} "
                f"min_margin={mm} failures={self.failures[:5]}")


# Records of the checks a test run made, by name (the GPU parity tests log
# the full workloads here; conftest prints them at the end of the run and
# writes them to $MARKOV_ACCEPTANCE_OUT when that is set).
RECORDS: dict = {}


def log(name: str, rep: Report) -> Report:
    RECORDS[name] = rep.record()
    return rep


def _key_range(head, embed, base_bits, v, p, T, mode, seed, b, i, tf):
    bias = oracle.bias_one(head, embed, v, p)
    keys = []
    for nb in bf16_nudges(bias):
        l = oracle.lib().orc_logit(int(base_bits[v]), int(nb), *tf)
        if not (T > 0):
            keys.append(float(oracle.bits_to_f32(np.array([l], np.uint16))[0]))
        else:
            keys.append(oracle.gumbel_key(l, T, seed, b, i, v))
    return min(keys), max(keys)


def check(inputs: dict, head_bits: np.ndarray, embed_bits: np.ndarray, mode: int, mult: float,
          cap, gpu_tokens: np.ndarray, gpu_cache: np.ndarray, tok_sentinel: int,
          cache_sentinel: int, nthreads: int = 0) -> Report:
    base = oracle.bf16_bits(inputs["base"])
    anchor = inputs["anchor"].numpy()
    temp = inputs["temperature"].numpy()
    seeds = inputs["seeds"].numpy()
    idx = inputs["row_state_idx"].numpy()
    R, N, V = base.shape
    o_tok, o_cache = oracle.chain(base, head_bits, embed_bits, anchor, temp, seeds, idx, mode,
                                  mult, cap, nthreads=nthreads)
    has_t, m, has_cap, c, inv = oracle.transform_params(mult, cap)
    tf = (has_t, m, has_cap, c, inv)
    rep = Report()
    for b in range(R):
        if idx[b] < 0:
            if not (np.all(gpu_tokens[b] == tok_sentinel) and np.all(gpu_cache[b] == cache_sentinel)):
                rep.failures.append(("padding row written", b))
            continue
        ref_tok = o_tok[b].copy()
        ref_cache = o_cache[b].copy()
        T = float(temp[b])
        seed = int(seeds[b])
        for i in range(N):
            rep.positions += 1
            g = gpu_cache[b, i]
            r_ = ref_cache[i]
            gn, rn = is_nan_bf16(g), is_nan_bf16(r_)
            if np.any(gn != rn):
                rep.failures.append(("cache NaN mismatch", b, i))
            both = ~gn & ~rn
            d = np.zeros(V, dtype=np.int64)
            d[both] = np.abs(ordered_bf16(g[both]) - ordered_bf16(r_[both]))
            rep.cache_elems += int(both.sum())
            p_i = int(anchor[b]) if i == 0 else int(gpu_tokens[b, i - 1])
            for v in np.flatnonzero(d > 1):
                bias = oracle.bias_one(head_bits, embed_bits, int(v), p_i)
                allowed = {oracle.lib().orc_logit(int(base[b, i, v]), int(nb), *tf)
                           for nb in bf16_nudges(bias)}
                if int(g[v]) in allowed:
                    rep.cache_bias_ulp += 1
                else:
                    rep.failures.append(("cache beyond a 1-ulp bias change", b, i, int(v),
                                         int(d[v])))
            ndiff = int((d >= 1).sum())
            rep.cache_ulp_diffs += int((d == 1).sum())
            gt = int(gpu_tokens[b, i])
            _, k1, k2 = oracle.select(r_, T, mode, seed, b, i)
            rep.note_margin(b, i, k1, k2)
            sel, _, _ = oracle.select(g, T, mode, seed, b, i)
            if sel != gt:
                rep.failures.append(("selection on GPU cache differs", b, i, sel, gt))
                continue
            if gt == int(ref_tok[i]):
                continue
            if ndiff == 0:
                rep.failures.append(("token differs with identical cache", b, i, gt,
                                     int(ref_tok[i])))
                continue
            ot = int(ref_tok[i])
            p = int(anchor[b]) if i == 0 else int(gpu_tokens[b, i - 1])
            excuse = None
            margin = float(k1) - float(k2)
            if mode == GUMBEL or not (T > 0):
                lo_w, _ = _key_range(head_bits, embed_bits, base[b, i], ot, p, T, mode, seed, b, i, tf)
                _, hi_g = _key_range(head_bits, embed_bits, base[b, i], gt, p, T, mode, seed, b, i, tf)
                if hi_g >= lo_w:
                    excuse = ("contender", b, i, gt, ot, margin, float(hi_g - lo_w))
            else:
                excuse = ("inverse-cdf on a cache 1 ulp apart", b, i, gt, ot, margin)
            if excuse is None:
                rep.failures.append(("token not excusable", b, i, gt, ot))
                continue
            rep.excused.append(excuse)
            if i + 1 < N:
                idx2 = np.full(R, -1, dtype=np.int64)
                idx2[b] = idx[b]
                ss = np.full(R, i + 1, dtype=np.int32)
                sp = np.zeros(R, dtype=np.int64)
                sp[b] = gt
                t2, c2 = oracle.chain(base, head_bits, embed_bits, anchor, temp, seeds, idx2, mode,
                                      mult, cap, start_step=ss, start_prev=sp, nthreads=nthreads)
                ref_tok[i + 1:] = t2[b, i + 1:]
                ref_cache[i + 1:] = c2[b, i + 1:]
    return rep


# ---------------------------------------------- fp32 base / cache variants

def _base_f32(base, b, i, v) -> float:
    """Base logit (b, i, v) as an fp32 value (BF16 bits or fp32 input)."""
    x = base[b, i, v]
    if base.dtype == np.uint16:
        return float(oracle.bits_to_f32(np.array([x], np.uint16))[0])
    return float(x)


def _typed_logit(base, b, i, v, bias_bits, cache_f32, mult, cap) -> float:
    return float(np.float32(oracle.logit_typed(_base_f32(base, b, i, v), int(bias_bits), cache_f32,
                                               mult, cap)))


def _bias_candidates(head_bits, embed_bits, v: int, p: int) -> set:
    """BF16 biases a correct fp32 reduction of head[v] . embed[p] can round
    to, in any summation order: the oracle's bias one ulp either way, and
    every BF16 value between the roundings of dot - err and dot + err, with
    dot the fp64 dot product and err the fp32 summation error bound
    2 r u sum|h e| (u = 2^-24; twice the textbook gamma_{r-1} for slack in
    the tensor cores' accumulation) plus the fp64 sum's own error.  Any fp32
    sum s within err of the exact product rounds into that range (rounding
    is monotone).  Without cancellation the range is within the oracle's
    bias one ulp either way; under cancellation it spans more than one BF16
    ulp of the small sum, which an fp32 cache keeps (a BF16 cache's rounding
    of base + bias hides it)."""
    cands = set(bf16_nudges(oracle.bias_one(head_bits, embed_bits, v, p)))
    h = oracle.bits_to_f32(np.ascontiguousarray(head_bits[v])).astype(np.float64)
    e = oracle.bits_to_f32(np.ascontiguousarray(embed_bits[p])).astype(np.float64)
    dot = float(np.dot(h, e))
    mag = float(np.sum(np.abs(h * e)))
    err = 2.0 * h.size * 2.0 ** -24 * mag + h.size * 2.0 ** -52 * mag
    lo = oracle.bf16_rne(np.array([dot - err], dtype=np.float32))[0]
    hi = oracle.bf16_rne(np.array([dot + err], dtype=np.float32))[0]
    a, b = int(ordered_bf16(np.array([lo], np.uint16))[0]), int(ordered_bf16(np.array([hi], np.uint16))[0])
    for o in range(min(a, b), max(a, b) + 1):
        cands.add((o if o >= 0 else (0x8000 | (-o))) & 0xFFFF)
    return cands


def check_typed(inputs: dict, head_bits: np.ndarray, embed_bits: np.ndarray, mode: int,
                mult: float, cap, gpu_tokens: np.ndarray, gpu_cache: np.ndarray, cache_f32: bool,
                tok_sentinel: int, cache_sentinel_bits: int, nthreads: int = 0) -> Report:
    """The acceptance rule of `check` for a BF16 or fp32 base and a BF16 or
    fp32 cache.  gpu_cache holds BF16 bits (uint16) or fp32 values (float32).
    An fp32 cache element must equal the oracle's exactly (NaN where the
    oracle has NaN) unless another BF16 bias of the same dot product that a
    correct fp32 reduction can give (_bias_candidates) explains it; a BF16
    cache element as in `check`, with the same bias set.  Tokens as in
    `check`, on fp32 keys."""
    base_t = inputs["base"]
    base = (base_t.numpy() if base_t.dtype == torch.float32 else oracle.bf16_bits(base_t))
    anchor = inputs["anchor"].numpy()
    temp = inputs["temperature"].numpy()
    seeds = inputs["seeds"].numpy()
    idx = inputs["row_state_idx"].numpy()
    R, N, V = base.shape
    o_tok, o_cache = oracle.chain_typed(base, head_bits, embed_bits, anchor, temp, seeds, idx,
                                        mode, mult, cap, cache_f32=cache_f32, nthreads=nthreads)
    rep = Report()
    for b in range(R):
        if idx[b] < 0:
            raw = gpu_cache[b].view(np.uint32 if cache_f32 else np.uint16)
            if not (np.all(gpu_tokens[b] == tok_sentinel) and np.all(raw == cache_sentinel_bits)):
                rep.failures.append(("padding row written", b))
            continue
        ref_tok = o_tok[b].copy()
        ref_cache = o_cache[b].copy()
        T = float(temp[b])
        seed = int(seeds[b])
        for i in range(N):
            rep.positions += 1
            g, r_ = gpu_cache[b, i], ref_cache[i]
            if cache_f32:
                gf, rf = g.astype(np.float32), r_.astype(np.float32)
                gn, rn = np.isnan(gf), np.isnan(rf)
            else:
                gf, rf = oracle.bits_to_f32(g), oracle.bits_to_f32(r_)
                gn, rn = is_nan_bf16(g), is_nan_bf16(r_)
            if np.any(gn != rn):
                rep.failures.append(("cache NaN mismatch", b, i))
            both = ~gn & ~rn
            rep.cache_elems += int(both.sum())
            if cache_f32:
                diff = both & (gf != rf)
                far = diff
            else:
                d = np.zeros(V, dtype=np.int64)
                d[both] = np.abs(ordered_bf16(g[both]) - ordered_bf16(r_[both]))
                diff = d >= 1
                far = d > 1
                rep.cache_ulp_diffs += int((d == 1).sum())
            p_i = int(anchor[b]) if i == 0 else int(gpu_tokens[b, i - 1])
            for v in np.flatnonzero(far):
                near = {_typed_logit(base, b, i, int(v), nb, cache_f32, mult, cap)
                        for nb in bf16_nudges(oracle.bias_one(head_bits, embed_bits, int(v), p_i))}
                if float(gf[v]) in near:
                    rep.cache_bias_ulp += 1
                    continue
                allowed = {_typed_logit(base, b, i, int(v), nb, cache_f32, mult, cap)
                           for nb in _bias_candidates(head_bits, embed_bits, int(v), p_i)}
                if float(gf[v]) in allowed:
                    rep.cache_bias_wide += 1
                else:
                    rep.failures.append(("cache beyond a 1-ulp bias change", b, i, int(v)))
            gt = int(gpu_tokens[b, i])
            _, k1, k2 = oracle.select_f(rf, T, mode, seed, b, i)
            rep.note_margin(b, i, k1, k2)
            sel, _, _ = oracle.select_f(gf, T, mode, seed, b, i)
            if sel != gt:
                rep.failures.append(("selection on GPU cache differs", b, i, sel, gt))
                continue
            if gt == int(ref_tok[i]):
                continue
            if not np.any(diff):
                rep.failures.append(("token differs with identical cache", b, i, gt,
                                     int(ref_tok[i])))
                continue
            ot = int(ref_tok[i])
            excuse = None
            margin = float(k1) - float(k2)
            if mode == GUMBEL or not (T > 0):
                def key_range(v):
                    ks = []
                    for nb in _bias_candidates(head_bits, embed_bits, v, p_i):
                        l = _typed_logit(base, b, i, v, nb, cache_f32, mult, cap)
                        if not (T > 0):
                            ks.append(l)
                        else:
                            x = np.float32(np.float32(l) / np.float32(T))
                            ks.append(float(np.float32(x + np.float32(oracle.gumbel(seed, b, i, v, 1)[0]))))
                    return min(ks), max(ks)
                lo_w, _ = key_range(ot)
                _, hi_g = key_range(gt)
                if hi_g >= lo_w:
                    excuse = ("contender", b, i, gt, ot, margin, float(hi_g - lo_w))
            else:
                excuse = ("inverse-cdf on a cache 1 ulp apart", b, i, gt, ot, margin)
            if excuse is None:
                rep.failures.append(("token not excusable", b, i, gt, ot))
                continue
            rep.excused.append(excuse)
            if i + 1 < N:
                idx2 = np.full(R, -1, dtype=np.int64)
                idx2[b] = idx[b]
                ss = np.full(R, i + 1, dtype=np.int32)
                sp = np.zeros(R, dtype=np.int64)
                sp[b] = gt
                t2, c2 = oracle.chain_typed(base, head_bits, embed_bits, anchor, temp, seeds, idx2,
                                            mode, mult, cap, cache_f32=cache_f32, start_step=ss,
                                            start_prev=sp, nthreads=nthreads)
                ref_tok[i + 1:] = t2[b, i + 1:]
                ref_cache[i + 1:] = c2[b, i + 1:]
    return rep
