"""Plain CPU oracle for DSpark sequential Markov sampling of draft tokens.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  The product library
(``draft_token_markov_gb300``) never imports, links or runs it, and the two
share no code: the only shared module is the seeded input generator
``draft_token_markov_gb300.workloads``, which holds none of the method's
arithmetic.

The arithmetic lives in ``markov_oracle.c`` (plain C, fp32, explicit
round-to-nearest-even BF16, ``-ffp-contract=off``), compiled here with gcc
and called through ctypes.  Every function cites the documentation page and
section it follows.  Parity status of each part is recorded in the package's
design notes: the bias, cache rounding, transform, noise and selection rules
are pinned by the CPU tests; agreement with the pages' own (unpublished)
kernels is unpinned, since no code or output of theirs exists.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "markov_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

GUMBEL = 0
INVCDF = 1

_lib = None
_lock = threading.Lock()


def _lib_path() -> str:
    return os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (gcc, -O2, no contraction).

    OpenMP is used when the compiler has it; it only splits the independent
    per-vocab-id loop, so results do not depend on the thread count."""
    path = _lib_path()
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    os.makedirs(_BUILD, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    base = ["gcc", "-std=gnu11", "-O2", "-fno-fast-math", "-ffp-contract=off",
            "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:-3] + ["-fopenmp"] + base[-3:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, path)
    return path


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


def _declare(L: ctypes.CDLL) -> None:
    c = ctypes
    P = c.c_void_p
    sig = {
        "orc_bf16_rne": (c.c_uint16, [c.c_float]),
        "orc_bf16_to_f32": (c.c_float, [c.c_uint16]),
        "orc_log": (c.c_float, [c.c_float]),
        "orc_exp": (c.c_float, [c.c_float]),
        "orc_tanh": (c.c_float, [c.c_float]),
        "orc_splitmix64": (c.c_uint64, [c.c_uint64]),
        "orc_row_step_hash": (c.c_uint64, [c.c_uint64, c.c_uint32, c.c_uint32]),
        "orc_uniform": (c.c_float, [c.c_uint64]),
        "orc_gumbel": (c.c_float, [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32]),
        "orc_cdf_hash": (c.c_uint64, [c.c_uint64, c.c_uint32, c.c_uint32]),
        "orc_bias": (c.c_uint16, [P, P, c.c_int]),
        "orc_logit": (c.c_uint16, [c.c_uint16, c.c_uint16, c.c_int, c.c_float, c.c_int,
                                   c.c_float, c.c_float]),
        "orc_gumbel_key": (c.c_float, [c.c_uint16, c.c_float, c.c_uint64, c.c_uint32,
                                       c.c_uint32, c.c_uint32]),
        "orc_select": (c.c_int64, [P, c.c_int, c.c_float, c.c_int, c.c_uint64, c.c_uint32,
                                   c.c_uint32, P, P]),
        "orc_chain": (c.c_int, [c.c_int, c.c_int, c.c_int, c.c_int, P, c.c_int64, c.c_int64,
                                P, P, P, P, P, P, c.c_int, c.c_int, c.c_float, c.c_int,
                                c.c_float, P, c.c_int64, P, c.c_int64, c.c_int64, P, P,
                                c.c_int]),
        "orc_logit_typed": (c.c_float, [c.c_float, c.c_uint16, c.c_int, c.c_int, c.c_float,
                                        c.c_int, c.c_float, c.c_float]),
        "orc_select_f": (c.c_int64, [P, c.c_int, c.c_float, c.c_int, c.c_uint64, c.c_uint32,
                                     c.c_uint32, P, P]),
        "orc_chain_typed": (c.c_int, [c.c_int, c.c_int, c.c_int, c.c_int, P, c.c_int,
                                      c.c_int64, c.c_int64, P, P, P, P, P, P, c.c_int, c.c_int,
                                      c.c_float, c.c_int, c.c_float, P, c.c_int64, P, c.c_int,
                                      c.c_int64, c.c_int64, P, P, c.c_int]),
        "orc_bf16_rne_n": (None, [P, P, c.c_int64]),
        "orc_log_n": (None, [P, P, c.c_int64]),
        "orc_exp_n": (None, [P, P, c.c_int64]),
        "orc_tanh_n": (None, [P, P, c.c_int64]),
        "orc_splitmix64_n": (None, [P, P, c.c_int64]),
        "orc_gumbel_n": (None, [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32, P,
                                c.c_int64]),
        "orc_bias_all": (None, [P, P, c.c_int, c.c_int, c.c_int64, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


# ----------------------------------------------------------------- helpers

def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"] or a.ndim == 0
    return a.ctypes.data


def _u64(x: int) -> int:
    return int(x) & 0xFFFFFFFFFFFFFFFF


def bf16_bits(x) -> np.ndarray:
    """BF16 tensor/array -> uint16 numpy bits (torch bfloat16 or uint16 input)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            assert x.dtype == torch.bfloat16
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    assert x.dtype == np.uint16
    return np.ascontiguousarray(x)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_rne(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_bf16_rne_n(_ptr(x), _ptr(y), x.size)
    return y


def _vec(fn_name: str, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    getattr(lib(), fn_name)(_ptr(x), _ptr(y), x.size)
    return y


def log(x):
    return _vec("orc_log_n", x)


def exp(x):
    return _vec("orc_exp_n", x)


def tanh(x):
    return _vec("orc_tanh_n", x)


def splitmix64(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint64)
    y = np.empty_like(x)
    lib().orc_splitmix64_n(_ptr(x), _ptr(y), x.size)
    return y


def row_step_hash(seed: int, row: int, step: int) -> int:
    return lib().orc_row_step_hash(_u64(seed), row, step)


def cdf_hash(seed: int, row: int, step: int) -> int:
    return lib().orc_cdf_hash(_u64(seed), row, step)


def uniform(h: int) -> float:
    return lib().orc_uniform(_u64(h))


def gumbel(seed: int, row: int, step: int, v0: int, n: int) -> np.ndarray:
    y = np.empty(n, dtype=np.float32)
    lib().orc_gumbel_n(_u64(seed), row, step, v0, _ptr(y), n)
    return y


def bias_all(head_bits: np.ndarray, embed_bits: np.ndarray, p: int) -> np.ndarray:
    V, r = head_bits.shape
    out = np.empty(V, dtype=np.uint16)
    lib().orc_bias_all(_ptr(head_bits), _ptr(embed_bits), V, r, int(p), _ptr(out))
    return out


def bias_one(head_bits: np.ndarray, embed_bits: np.ndarray, v: int, p: int) -> int:
    h = np.ascontiguousarray(head_bits[v])
    e = np.ascontiguousarray(embed_bits[p])
    return lib().orc_bias(_ptr(h), _ptr(e), h.size)


def logit(base_bits: int, bias_bits: int, mult: float = 1.0, cap: float | None = None) -> int:
    has_t, m, has_cap, c, inv = transform_params(mult, cap)
    return lib().orc_logit(int(base_bits), int(bias_bits), has_t, m, has_cap, c, inv)


def transform_params(mult: float, cap: float | None):
    """(has_transform, mult_f32, has_cap, cap_f32, inv_cap_f32): the multiplier
    and cap rounded to fp32 and inv_cap = fp32(1) / fp32(cap)."""
    m = float(np.float32(mult))
    has_cap = cap is not None and cap > 0
    c = float(np.float32(cap)) if has_cap else 1.0
    inv = float(np.float32(1.0) / np.float32(c)) if has_cap else 1.0
    has_t = int(m != 1.0 or has_cap)
    return has_t, m, int(has_cap), c, inv


def gumbel_key(l_bits: int, T: float, seed: int, row: int, step: int, v: int) -> float:
    return lib().orc_gumbel_key(int(l_bits), float(T), _u64(seed), row, step, v)


def select(l_bits: np.ndarray, T: float, mode: int, seed: int, row: int, step: int):
    """(token, winning key, runner-up key) of one position's cached logits."""
    l_bits = np.ascontiguousarray(l_bits, dtype=np.uint16)
    k1 = ctypes.c_float()
    k2 = ctypes.c_float()
    tok = lib().orc_select(_ptr(l_bits), l_bits.size, float(np.float32(T)), int(mode),
                           _u64(seed), row, step, ctypes.addressof(k1), ctypes.addressof(k2))
    return int(tok), k1.value, k2.value


def chain(base_bits: np.ndarray, head_bits: np.ndarray, embed_bits: np.ndarray,
          anchor: np.ndarray, temperature: np.ndarray, seeds: np.ndarray,
          row_state_idx: np.ndarray, mode: int, mult: float = 1.0,
          cap: float | None = None, tokens: np.ndarray | None = None,
          cache: np.ndarray | None = None, start_step: np.ndarray | None = None,
          start_prev: np.ndarray | None = None, nthreads: int = 0):
    """Run the oracle chain.  base_bits [rows, N, V] uint16; head/embed [V, r]
    uint16.  Returns (tokens [rows, N] int64, cache [rows, N, V] uint16);
    padding rows keep the values of the passed-in ``tokens`` / ``cache``
    (sentinels), which default to -1 and 0xFFFF."""
    rows, N, V = base_bits.shape
    Vh, r = head_bits.shape
    assert Vh >= V and embed_bits.shape[1] == r
    base_bits = np.ascontiguousarray(base_bits, dtype=np.uint16)
    head_bits = np.ascontiguousarray(head_bits, dtype=np.uint16)
    embed_bits = np.ascontiguousarray(embed_bits, dtype=np.uint16)
    anchor = np.ascontiguousarray(anchor, dtype=np.int32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    seeds = np.ascontiguousarray(seeds, dtype=np.int64)
    row_state_idx = np.ascontiguousarray(row_state_idx, dtype=np.int64)
    if tokens is None:
        tokens = np.full((rows, N), -1, dtype=np.int64)
    if cache is None:
        cache = np.full((rows, N, V), 0xFFFF, dtype=np.uint16)
    assert tokens.dtype == np.int64 and tokens.flags["C_CONTIGUOUS"]
    assert cache.dtype == np.uint16 and cache.flags["C_CONTIGUOUS"]
    ss = sp = None
    if start_step is not None:
        ss = np.ascontiguousarray(start_step, dtype=np.int32)
        sp = np.ascontiguousarray(start_prev, dtype=np.int64)
    has_t, m, has_cap, c, _ = transform_params(mult, cap)
    rc = lib().orc_chain(V, r, N, rows, _ptr(base_bits), N * V, V, _ptr(head_bits),
                         _ptr(embed_bits), _ptr(anchor), _ptr(temperature), _ptr(seeds),
                         _ptr(row_state_idx), int(mode), has_t, m, has_cap, c,
                         _ptr(tokens), N, _ptr(cache), N * V, V,
                         _ptr(ss) if ss is not None else None,
                         _ptr(sp) if sp is not None else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle chain: anchor or previous token out of range")
    return tokens, cache


# ------------------------------------------------ fp32 base / cache variants

def logit_typed(base: float, bias_bits: int, cache_f32: bool, mult: float = 1.0,
                cap: float | None = None) -> float:
    """The cached logit as an fp32 value for a BF16 (cache_f32 False) or fp32
    cache; base is the base logit's fp32 value."""
    has_t, m, has_cap, c, inv = transform_params(mult, cap)
    return lib().orc_logit_typed(float(np.float32(base)), int(bias_bits), int(bool(cache_f32)),
                                 has_t, m, has_cap, c, inv)


def select_f(l: np.ndarray, T: float, mode: int, seed: int, row: int, step: int):
    """select() on fp32 logit values."""
    l = np.ascontiguousarray(l, dtype=np.float32)
    k1 = ctypes.c_float()
    k2 = ctypes.c_float()
    tok = lib().orc_select_f(_ptr(l), l.size, float(np.float32(T)), int(mode), _u64(seed), row,
                             step, ctypes.addressof(k1), ctypes.addressof(k2))
    return int(tok), k1.value, k2.value


def chain_typed(base: np.ndarray, head_bits: np.ndarray, embed_bits: np.ndarray,
                anchor: np.ndarray, temperature: np.ndarray, seeds: np.ndarray,
                row_state_idx: np.ndarray, mode: int, mult: float = 1.0,
                cap: float | None = None, cache_f32: bool = False,
                tokens: np.ndarray | None = None, cache: np.ndarray | None = None,
                start_step: np.ndarray | None = None, start_prev: np.ndarray | None = None,
                nthreads: int = 0):
    """chain() with the base logits as BF16 bits (uint16) or fp32 values
    (float32) and a BF16 (uint16 bits) or fp32 cache.  Returns (tokens,
    cache); padding rows keep the passed-in values (defaults -1 and
    0xFFFF / NaN)."""
    rows, N, V = base.shape
    Vh, r = head_bits.shape
    assert Vh >= V and embed_bits.shape[1] == r
    base_f32 = base.dtype == np.float32
    base = np.ascontiguousarray(base, dtype=np.float32 if base_f32 else np.uint16)
    head_bits = np.ascontiguousarray(head_bits, dtype=np.uint16)
    embed_bits = np.ascontiguousarray(embed_bits, dtype=np.uint16)
    anchor = np.ascontiguousarray(anchor, dtype=np.int32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    seeds = np.ascontiguousarray(seeds, dtype=np.int64)
    row_state_idx = np.ascontiguousarray(row_state_idx, dtype=np.int64)
    if tokens is None:
        tokens = np.full((rows, N), -1, dtype=np.int64)
    if cache is None:
        cache = (np.full((rows, N, V), np.nan, dtype=np.float32) if cache_f32
                 else np.full((rows, N, V), 0xFFFF, dtype=np.uint16))
    assert tokens.dtype == np.int64 and tokens.flags["C_CONTIGUOUS"]
    assert cache.dtype == (np.float32 if cache_f32 else np.uint16) and cache.flags["C_CONTIGUOUS"]
    ss = sp = None
    if start_step is not None:
        ss = np.ascontiguousarray(start_step, dtype=np.int32)
        sp = np.ascontiguousarray(start_prev, dtype=np.int64)
    has_t, m, has_cap, c, _ = transform_params(mult, cap)
    rc = lib().orc_chain_typed(V, r, N, rows, _ptr(base), int(base_f32), N * V, V,
                               _ptr(head_bits), _ptr(embed_bits), _ptr(anchor),
                               _ptr(temperature), _ptr(seeds), _ptr(row_state_idx), int(mode),
                               has_t, m, has_cap, c, _ptr(tokens), N, _ptr(cache),
                               int(bool(cache_f32)), N * V, V,
                               _ptr(ss) if ss is not None else None,
                               _ptr(sp) if sp is not None else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle chain: anchor or previous token out of range")
    return tokens, cache
