"""Seeded synthetic inputs for DSpark sequential Markov sampling.

This module only draws inputs: it holds none of the method's arithmetic, and
it is the one module that both the CUDA path's tests and the CPU oracle's
tests use.  Everything is drawn on the CPU with ``torch.Generator`` so that
the same seed gives the same tensors on every machine.

The shapes follow the pages: the DeepSeek-V4.1 Markov head is [129280, 256]
BF16, 66 MB ("vllm.models.deepseek_v41.nvidia.specialized_decode.sampling.
sharded_markov", module docstring and DSparkShardedMarkovSampler), a chain
call takes at most 8 request rows (same docstring), larger batches take the
per-step loop ("vllm.models.deepseek_v41.nvidia.ops.fused_markov").  The
value distributions (normal weights and logits, injected spikes, exact ties,
NaNs, padding rows) are synthetic stand-ins: no trained head or real logits
are available.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import torch

GUMBEL = 0
INVCDF = 1


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, distributions and sampling settings."""
    name: str
    vocab: int
    rank: int
    rows: int
    steps: int
    mode: int
    weight_std: float
    base_std: float
    temperatures: tuple = (1.0,)        # per-row T drawn uniformly from these
    padding_rows: tuple = ()            # rows with row_state_idx = -1
    spikes: int = 0                     # ids per (row, step) raised by +12 in fp32
    tie_row: int = -1                   # row whose 3 ids per step get base = 64.0
    nan_row: int = -1                   # row whose 4 ids per step get base = NaN
    mult: float = 1.0
    cap: float | None = None
    fixed_seed: int | None = None       # every row's sampling seed, if fixed
    gen_seed: int = 0                   # torch.Generator seed

    @property
    def live_rows(self) -> int:
        return self.rows - len(self.padding_rows)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the benchmark and the parity tests.
TINY = Workload("tiny chain V=4096 r=64 rows=1 N=4 gumbel", 4096, 64, 1, 4, GUMBEL,
                0.02, 2.0, temperatures=(1.0,), fixed_seed=1, gen_seed=1001)
DEEPSEEK = Workload("deepseek-v4.1 chain V=129280 r=256 rows=8 N=8 gumbel", 129280, 256, 8,
                    8, GUMBEL, 0.02, 3.0, temperatures=(0.0, 0.6, 1.0), padding_rows=(2, 5),
                    spikes=8, gen_seed=1002)
LATENCY = Workload("latency chain V=129280 r=256 rows=1 N=8 gumbel", 129280, 256, 1, 8,
                   GUMBEL, 0.02, 3.0, temperatures=(1.0,), spikes=8, gen_seed=1003)
SOFTCAP = Workload("soft-capped chain V=262144 r=128 rows=4 N=6 inverse-cdf", 262144, 128,
                   4, 6, INVCDF, 0.03, 4.0, temperatures=(0.7, 1.0), tie_row=1, nan_row=2,
                   mult=0.5, cap=30.0, gen_seed=1004)
BATCH = Workload("large batch V=129280 r=256 rows=64 N=8 inverse-cdf", 129280, 256, 64, 8,
                 INVCDF, 0.02, 3.0, temperatures=(0.0, 0.5, 0.8, 1.0, 1.2),
                 padding_rows=tuple(range(7, 64, 8)), gen_seed=1005)

BY_NAME = {"tiny": TINY, "deepseek": DEEPSEEK, "latency": LATENCY, "softcap": SOFTCAP,
           "batch": BATCH}


def with_rows(w: Workload, rows: int) -> Workload:
    """The workload with another row count; its padding rows below it stay."""
    return w.with_(rows=rows, padding_rows=tuple(b for b in w.padding_rows if b < rows),
                   name=f"{w.name} at rows={rows}")


def _randn_bf16(shape, std, g):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def _distinct_ids(n, V, g):
    return torch.randperm(V, generator=g)[:n]


def make_weights(w: Workload):
    """(head [V, r], embed [V, r]) BF16, normal with the workload's std."""
    g = torch.Generator("cpu").manual_seed(w.gen_seed)
    head = _randn_bf16((w.vocab, w.rank), w.weight_std, g)
    embed = _randn_bf16((w.vocab, w.rank), w.weight_std, g)
    return head, embed


def make_call(w: Workload, call: int = 0, base_f32: bool = False):
    """The per-call inputs of call number ``call``: base logits [rows, N, V]
    BF16 (fp32 with ``base_f32``), anchor tokens int32, temperature fp32, seeds int64 and
    row_state_idx int64 (-1 on padding rows), all on the CPU.

    Call 0 of every workload draws the base logits; later calls of the same
    workload keep them and draw fresh seeds and anchors (the latency case's
    1000 calls)."""
    g = torch.Generator("cpu").manual_seed(w.gen_seed + 7919)
    R, N, V = w.rows, w.steps, w.vocab
    base32 = torch.randn((R, N, V), generator=g, dtype=torch.float32) * w.base_std
    for b in range(R):
        for i in range(N):
            if w.spikes:
                ids = _distinct_ids(w.spikes, V, g)
                base32[b, i, ids] += 12.0
            if b == w.tie_row:
                base32[b, i, _distinct_ids(3, V, g)] = 64.0
            if b == w.nan_row:
                base32[b, i, _distinct_ids(4, V, g)] = float("nan")
    # an fp32 base keeps the drawn values (not rounded to BF16)
    base = base32.contiguous() if base_f32 else base32.to(torch.bfloat16)
    gc = torch.Generator("cpu").manual_seed(w.gen_seed * 1_000_003 + call)
    anchor = torch.randint(0, V, (R,), generator=gc, dtype=torch.int64).to(torch.int32)
    temps = torch.tensor(w.temperatures, dtype=torch.float32)
    tidx = torch.randint(0, len(w.temperatures), (R,), generator=gc)
    temperature = temps[tidx].contiguous()
    if w.fixed_seed is not None:
        seeds = torch.full((R,), int(w.fixed_seed) + call, dtype=torch.int64)
    else:
        seeds = torch.randint(-(2**63), 2**63 - 1, (R,), generator=gc, dtype=torch.int64)
    idx = torch.arange(R, dtype=torch.int64)
    for b in w.padding_rows:
        idx[b] = -1
    return dict(base=base, anchor=anchor, temperature=temperature, seeds=seeds,
                row_state_idx=idx)


def small(V: int, r: int, rows: int, steps: int, mode: int = GUMBEL, *, seed: int = 0,
          weight_std: float = 0.05, base_std: float = 2.0, temperatures=(0.0, 0.7, 1.0),
          padding_rows=(), mult: float = 1.0, cap: float | None = None, spikes: int = 0,
          tie_row: int = -1, nan_row: int = -1) -> Workload:
    """A small parity workload of any shape (ragged vocab tails included)."""
    return Workload(f"small V={V} r={r} rows={rows} N={steps}", V, r, rows, steps, mode,
                    weight_std, base_std, temperatures=tuple(temperatures),
                    padding_rows=tuple(padding_rows), spikes=spikes, tie_row=tie_row,
                    nan_row=nan_row, mult=mult, cap=cap, gen_seed=50_000 + seed)


# Algorithmic bytes of one call: the head once, the live rows' base-logit
# reads and their cache writes (BF16 unless the element sizes say otherwise).
# Noise bytes are not algorithmic.
def algorithmic_bytes(w: Workload, base_bytes: int = 2, cache_bytes: int = 2) -> int:
    """base_bytes / cache_bytes: element sizes of the base logits and the
    cache (2 for BF16, 4 for fp32)."""
    head = w.vocab * w.rank * 2
    return head + w.live_rows * w.steps * w.vocab * (base_bytes + cache_bytes)
