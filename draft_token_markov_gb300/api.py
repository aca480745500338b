"""Thin Python binding of the C ABI in ``include/markov.h``.

Argument marshalling only: every step of the sampling path runs in the CUDA
library.  Tensors are PyTorch CUDA tensors (PyTorch provides device memory
and streams); their data pointers, strides and the current stream are passed
through ctypes.  The library is loaded on first use; if it is missing or
cannot be loaded this module raises, it never falls back to another
implementation."""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

GUMBEL = 0
INVCDF = 1
PATH_AUTO, PATH_CHAIN, PATH_BATCH, PATH_CHAIN_SIMPLE = 0, 1, 2, 3
Q_CHAIN_CTAS, Q_RESIDENT_HEAD_BYTES, Q_LAST_LAUNCHES, Q_LAST_PATH, Q_SM_COUNT = range(5)

STATUS = {0: "MARKOV_OK", 1: "MARKOV_EINVAL", 2: "MARKOV_EUNSUPPORTED", 3: "MARKOV_ECUDA",
          4: "MARKOV_ETIMEOUT", 5: "MARKOV_ENOTRESIDENT", 6: "MARKOV_EDEVICE"}

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "markov.h")

_lib = None


class MarkovError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({lib().markov_status_string(code).decode()})")


class _Desc(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("num_steps", ctypes.c_int32), ("max_rows", ctypes.c_int32),
                ("device", ctypes.c_int32), ("timeout_ms", ctypes.c_int32)]


def header_symbols() -> list[str]:
    """Names of the functions include/markov.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(markov_[a-z_0-9]+)\s*\(", text)))


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (building it if it is absent or stale)."""
    global _lib
    if _lib is None:
        p = path or _build.build()
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library missing: {p}")
        L = ctypes.CDLL(p)
        _declare(L)
        _lib = L
    return _lib


def _declare(L):
    c = ctypes
    P = c.c_void_p
    i32, i64, f32 = c.c_int32, c.c_int64, c.c_float
    sig = {
        "markov_plan_create": (i32, [c.POINTER(_Desc), c.POINTER(P)]),
        "markov_plan_destroy": (None, [P]),
        "markov_chain_max_rows": (i32, [P]),
        "markov_plan_set_path": (i32, [P, i32]),
        "markov_noise_fork": (i32, [P, P, P, P, i32, P]),
        "markov_noise_join": (i32, [P, P]),
        "markov_chain_sample": (i32, [P, P, i64, i64, P, P, P, P, P, P, i32, i32, f32, f32,
                                      P, i64, P, i64, i64, P]),
        "markov_chain_sample_typed": (i32, [P, P, i32, i64, i64, P, P, P, P, P, P, i32, i32, f32,
                                            f32, P, i64, P, i32, i64, i64, P]),
        "markov_plan_status": (i32, [P]),
        "markov_shard_plan_create": (i32, [c.POINTER(_Desc), i32, c.POINTER(P)]),
        "markov_shard_plan_destroy": (None, [P]),
        "markov_shard_plan_ctas": (i32, [P]),
        "markov_shard_plan_status": (i32, [P]),
        "markov_chain_sample_sharded": (i32, [P, P, i64, i64, P, P, P, P, P, P, i32, f32, f32,
                                              P, i64, P, i64, i64, P]),
        "markov_status_string": (c.c_char_p, [i32]),
        "markov_gumbel_noise": (i32, [P, P, P, i32, i32, i32, P, i64, P]),
        "markov_device_math": (i32, [i32, P, P, i64, P]),
        "markov_plan_query": (i64, [P, i32]),
        "markov_plan_inject_status": (i32, [P, i32, c.c_uint32]),
        "markov_selftest_wait": (i32, [i32, i32, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def _check(code: int, what: str):
    if code != 0:
        raise MarkovError(code, what)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _dev_or_pinned(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    """A CUDA tensor, or a pinned CPU tensor the kernels read (or write) over
    the host link (the inputs and tokens of the sample calls)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise TypeError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        return t.data_ptr()
    return _dev(t, dtype, name)


MARKOV_BF16 = 0
MARKOV_F32 = 1


class Plan:
    """A sampling plan: static shapes plus all scratch, allocated once."""

    def __init__(self, vocab: int, rank: int, num_steps: int, max_rows: int,
                 device: int | None = None, timeout_ms: int = 0):
        if device is None:
            device = torch.cuda.current_device()
        d = _Desc(vocab, rank, num_steps, max_rows, device, timeout_ms)
        h = ctypes.c_void_p()
        _check(lib().markov_plan_create(ctypes.byref(d), ctypes.byref(h)), "markov_plan_create")
        self._h = h
        self.vocab, self.rank, self.num_steps, self.max_rows = vocab, rank, num_steps, max_rows
        self.device = device

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            lib().markov_plan_destroy(self._h)
            self._h = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def query(self, key: int) -> int:
        return int(lib().markov_plan_query(self._h, key))

    def set_path(self, path: int):
        _check(lib().markov_plan_set_path(self._h, path), "markov_plan_set_path")

    @property
    def chain_max_rows(self) -> int:
        return int(lib().markov_chain_max_rows(self._h))


class ShardPlan:
    """A vocabulary-sharded plan: `world` ranks, each with scratch of its own
    (the sharded chain's ranks, emulated on one GPU)."""

    def __init__(self, vocab: int, rank: int, num_steps: int, max_rows: int, world: int,
                 device: int | None = None, timeout_ms: int = 0):
        if device is None:
            device = torch.cuda.current_device()
        d = _Desc(vocab, rank, num_steps, max_rows, device, timeout_ms)
        h = ctypes.c_void_p()
        _check(lib().markov_shard_plan_create(ctypes.byref(d), int(world), ctypes.byref(h)),
               "markov_shard_plan_create")
        self._h = h
        self.vocab, self.rank, self.num_steps, self.max_rows = vocab, rank, num_steps, max_rows
        self.world, self.device = world, device

    @property
    def handle(self):
        return self._h

    @property
    def ctas(self) -> int:
        return int(lib().markov_shard_plan_ctas(self._h))

    def close(self):
        if getattr(self, "_h", None):
            lib().markov_shard_plan_destroy(self._h)
            self._h = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


def shard_range(rank: int, world: int, vocab: int) -> tuple[int, int]:
    """(first id, width) of `rank`'s vocabulary shard: rows [k V / world,
    (k + 1) V / world) of the head (sharded_markov page, module docstring)."""
    if world < 1 or not 0 <= rank < world or vocab % world:
        raise ValueError("vocab must split evenly over the ranks")
    w = vocab // world
    return rank * w, w


def agree_on_shards(group, vocab: int, offset: int, width: int) -> bool:
    """Whether, on every rank of the torch.distributed `group`, (offset,
    width) is that rank's vocabulary shard (shard_range); a collective that
    every rank must enter (sharded_markov page, accepts_shard: a rank that
    skipped it would leave its peers waiting)."""
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    mine = torch.tensor([offset, width], dtype=torch.int64)
    got = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(got, mine, group=group)
    if vocab % world:
        return False
    return all(tuple(int(x) for x in got[k]) == shard_range(k, world, vocab) for k in range(world))


def markov_chain_sample_sharded(plan: ShardPlan, base_logits, head_shards, embed, anchor_tokens,
                                temperature, seeds, row_state_idx, output_multiplier: float = 1.0,
                                soft_cap: float | None = None, draft_tokens=None,
                                logit_caches=None, stream=None):
    """Sample on every rank of `plan`; returns (draft_tokens, logit_caches),
    one [rows, N] and one [rows, N, V] tensor per rank (allocated when not
    given).  head_shards[k] is rank k's [V / world, r] BF16 head rows."""
    rows, N, V = base_logits.shape
    W = plan.world
    dev = base_logits.device
    if len(head_shards) != W:
        raise ValueError(f"{W} head shards expected")
    if draft_tokens is None:
        draft_tokens = [torch.empty((rows, N), dtype=torch.int64, device=dev) for _ in range(W)]
    if logit_caches is None:
        logit_caches = [torch.empty((rows, N, V), dtype=torch.bfloat16, device=dev)
                        for _ in range(W)]
    if base_logits.stride(2) != 1:
        raise ValueError("the last dimension of base_logits must be contiguous")
    for k in range(W):
        if not head_shards[k].is_contiguous():
            raise ValueError("head shards must be contiguous")
        if draft_tokens[k].stride(1) != 1 or logit_caches[k].stride(2) != 1:
            raise ValueError("the last dimension of the outputs must be contiguous")
        if (draft_tokens[k].stride(0) != draft_tokens[0].stride(0) or
                logit_caches[k].stride()[:2] != logit_caches[0].stride()[:2]):
            raise ValueError("every rank's outputs must have the same strides")
    P = ctypes.c_void_p
    heads = (P * W)(*[_dev(h, torch.bfloat16, "head_shards") for h in head_shards])
    toks = (P * W)(*[_dev(t, torch.int64, "draft_tokens") for t in draft_tokens])
    caches = (P * W)(*[_dev(c, torch.bfloat16, "logit_caches") for c in logit_caches])
    cap = -1.0 if soft_cap is None else float(soft_cap)
    code = lib().markov_chain_sample_sharded(
        plan.handle, _dev(base_logits, torch.bfloat16, "base_logits"), base_logits.stride(0),
        base_logits.stride(1), heads, _dev(embed, torch.bfloat16, "embed"),
        _dev(anchor_tokens, torch.int32, "anchor_tokens"),
        _dev(temperature, torch.float32, "temperature"), _dev(seeds, torch.int64, "seeds"),
        _dev(row_state_idx, torch.int64, "row_state_idx"), rows, float(output_multiplier), cap,
        toks, draft_tokens[0].stride(0), caches, logit_caches[0].stride(0),
        logit_caches[0].stride(1), _stream(stream))
    _check(code, "markov_chain_sample_sharded")
    return draft_tokens, logit_caches


def markov_shard_plan_status(plan: ShardPlan) -> int:
    """The sticky device status of the sharded plan's calls (0 = ok); clears it."""
    return int(lib().markov_shard_plan_status(plan.handle))


def markov_noise_fork(plan: Plan, seeds, temperature, row_state_idx, stream=None):
    rows = seeds.shape[0]
    _check(lib().markov_noise_fork(plan.handle, _dev(seeds, torch.int64, "seeds"),
                                   _dev(temperature, torch.float32, "temperature"),
                                   _dev(row_state_idx, torch.int64, "row_state_idx"), rows,
                                   _stream(stream)), "markov_noise_fork")


def markov_noise_join(plan: Plan, stream=None):
    _check(lib().markov_noise_join(plan.handle, _stream(stream)), "markov_noise_join")


def markov_chain_sample(plan: Plan, base_logits, head, embed, anchor_tokens, temperature, seeds,
                        row_state_idx, mode: int, output_multiplier: float = 1.0,
                        soft_cap: float | None = None, draft_tokens=None, logit_cache=None,
                        stream=None):
    """Sample the draft tokens; returns (draft_tokens, logit_cache).  Output
    tensors are allocated when not given (padding rows are then left
    uninitialised, as the library never writes them).  base_logits and
    logit_cache may each be bfloat16 or float32 (markov_chain_sample_typed;
    the cache defaults to bfloat16).  The inputs and draft_tokens may be
    pinned CPU tensors, which the kernels read and write directly."""
    rows, N, V = base_logits.shape
    dev = head.device
    if draft_tokens is None:
        draft_tokens = torch.empty((rows, N), dtype=torch.int64, device=dev)
    if logit_cache is None:
        logit_cache = torch.empty((rows, N, V), dtype=torch.bfloat16, device=dev)
    dtypes = {torch.bfloat16: MARKOV_BF16, torch.float32: MARKOV_F32}
    if base_logits.dtype not in dtypes or logit_cache.dtype not in dtypes:
        raise TypeError("base_logits and logit_cache must be bfloat16 or float32")
    if base_logits.stride(2) != 1 or logit_cache.stride(2) != 1 or draft_tokens.stride(1) != 1:
        raise ValueError("the last dimension of base_logits, logit_cache and draft_tokens must "
                         "be contiguous")
    for t, n in ((head, "head"), (embed, "embed")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    cap = -1.0 if soft_cap is None else float(soft_cap)
    code = lib().markov_chain_sample_typed(
        plan.handle, _dev_or_pinned(base_logits, base_logits.dtype, "base_logits"),
        dtypes[base_logits.dtype], base_logits.stride(0), base_logits.stride(1),
        _dev(head, torch.bfloat16, "head"),
        _dev(embed, torch.bfloat16, "embed"),
        _dev_or_pinned(anchor_tokens, torch.int32, "anchor_tokens"),
        _dev_or_pinned(temperature, torch.float32, "temperature"),
        _dev_or_pinned(seeds, torch.int64, "seeds"),
        _dev_or_pinned(row_state_idx, torch.int64, "row_state_idx"), rows, int(mode),
        float(output_multiplier), cap, _dev_or_pinned(draft_tokens, torch.int64, "draft_tokens"),
        draft_tokens.stride(0), _dev(logit_cache, logit_cache.dtype, "logit_cache"),
        dtypes[logit_cache.dtype], logit_cache.stride(0), logit_cache.stride(1), _stream(stream))
    _check(code, "markov_chain_sample")
    return draft_tokens, logit_cache


def markov_plan_status(plan: Plan) -> int:
    """The sticky device status (0 = ok); clears it."""
    return int(lib().markov_plan_status(plan.handle))


def markov_gumbel_noise(seeds, temperature, row_state_idx, num_steps: int, vocab: int, out=None,
                        stream=None):
    rows = seeds.shape[0]
    if out is None:
        out = torch.full((rows * num_steps, vocab), float("nan"), dtype=torch.float32,
                         device=seeds.device)
    _check(lib().markov_gumbel_noise(_dev(seeds, torch.int64, "seeds"),
                                     _dev(temperature, torch.float32, "temperature"),
                                     _dev(row_state_idx, torch.int64, "row_state_idx"), rows,
                                     num_steps, vocab, _dev(out, torch.float32, "out"),
                                     out.stride(0), _stream(stream)), "markov_gumbel_noise")
    return out


def markov_device_math(fn: int, x, out=None, stream=None):
    if out is None:
        out = torch.empty_like(x)
    _check(lib().markov_device_math(int(fn), _dev(x, torch.float32, "x"),
                                    _dev(out, torch.float32, "out"), x.numel(), _stream(stream)),
           "markov_device_math")
    return out


def markov_plan_inject_status(plan: Plan, code: int, where: int = 0):
    """Record a device status as a failing kernel would (test hook)."""
    _check(lib().markov_plan_inject_status(plan.handle, int(code), int(where)),
           "markov_plan_inject_status")


def markov_selftest_wait(which: int, timeout_us: int, stream=None) -> int:
    """Run one bounded wait that nothing can complete; returns the status it
    recorded (4 = MARKOV_ETIMEOUT when it gave up as designed)."""
    code = lib().markov_selftest_wait(int(which), int(timeout_us), _stream(stream))
    if code not in (0, 4):
        raise MarkovError(code, "markov_selftest_wait")
    return int(code)
