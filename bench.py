"""Benchmark of DSpark sequential Markov draft sampling on one GB300.

A step is one whole Markov call of the DeepSeek-V4.1-shaped workload
(V=129280, r=256, 8 request rows of which 2 are padding, N=8 draft
positions, Gumbel mode) over inputs already resident in HBM: one launch of
the persistent chain kernel, which also draws the call's Gumbel noise.  L2 is flushed (a 256 MB write) before
every timed step and the flush is not timed.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --gpus N > 1 (one process per GPU under torch.distributed.run) every
rank runs an independent replica of the workload: the path has no exchange
step, so there is no collective; value is the tokens of all ranks over the
slowest rank's time.

--impl reference times the CPU oracle (the plain C definition of the method)
on this machine's host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft tokens/s and µs per N-step Markov call; % of GB300 HBM roofline"
UNIT = "draft tokens/s"
# --workload names (workloads.BY_NAME): the default is the DeepSeek-V4.1
# chain the headline is quoted on; the others measure the remaining paths
DEFAULT_WORKLOAD = "deepseek"
WORKLOAD_NAMES = ("batch", "deepseek", "latency", "softcap", "tiny")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "chain_deepseek_traffic.json")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_source_hash() -> str:
    """Hash of the sources the chain kernel is built from: its translation
    unit and every header (the other kernels' .cu files do not enter it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "draft_token_markov_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name == "chain_tc.cu" or name.endswith((".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic():
    """DRAM bytes per chain launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("source_hash") == _kernel_source_hash():
            return int(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a while to start: wait for its first sample
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.window = [time.time(), None]
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.window[0] = time.time()

    def mark_end(self):
        self.window[1] = time.time()

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = self.window[0], self.window[1] or time.time()
        for t, line in self.lines:
            if not (lo <= t <= hi + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float) -> float:
    """The maximum of a per-rank value over the default process group (the
    rank's own value without one): the whole-job time of a step is the
    slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


_ORACLE_INPUTS = {}


def _oracle_inputs(name: str):
    """The oracle's arguments for the workload's first live row (drawn once
    per process; the timed samples reuse them)."""
    if name not in _ORACLE_INPUTS:
        import numpy as np
        import oracle
        from draft_token_markov_gb300 import workloads as W
        w = W.BY_NAME[name]
        head, embed = W.make_weights(w)
        inp = W.make_call(w)
        hb, eb = oracle.bf16_bits(head), oracle.bf16_bits(embed)
        live = [b for b in range(w.rows) if int(inp["row_state_idx"][b]) >= 0]
        b0 = live[0]
        idx = np.full(w.rows, -1, dtype=np.int64)
        idx[b0] = b0
        base = oracle.bf16_bits(inp["base"])
        _ORACLE_INPUTS[name] = (w, (base, hb, eb, inp["anchor"].numpy(),
                                   inp["temperature"].numpy(), inp["seeds"].numpy(), idx,
                                   w.mode, w.mult, w.cap))
    return _ORACLE_INPUTS[name]


def cpu_oracle_sample(seconds_hint: float = 20.0, name: str = DEFAULT_WORKLOAD,
                      threads: int = 0):
    """Time the oracle on a bounded sample of the workload: one call over the
    workload's first live row (all N positions), repeated while the total
    stays near seconds_hint, on `threads` host threads (0: all cores).
    Returns (tokens/s, sample description, threads used)."""
    import oracle
    w, args = _oracle_inputs(name)
    cores = threads or os.cpu_count() or 1
    t0 = time.perf_counter()
    calls = 0
    while True:
        oracle.chain(*args, nthreads=cores)
        calls += 1
        el = time.perf_counter() - t0
        if el * (calls + 1) / calls > seconds_hint or calls >= 50:
            break
    tokens = calls * w.steps
    return tokens / el, (f"{calls} oracle call(s) of the {w.name} workload restricted to one "
                         f"live row ({w.steps} draft tokens each), OpenMP over vocab ids on "
                         f"{cores} thread(s)"), cores


def reference_step_seconds(steps: int, warmup: int) -> float:
    """Oracle seconds per reference-arm step: a bounded sample, sized so the
    whole run stays near two minutes whatever K and W are (each step still
    makes at least one oracle call)."""
    return max(0.05, min(8.0, 120.0 / max(1, steps + warmup)))


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    vals = []
    desc = cores = None
    name = args.workload
    per_step = reference_step_seconds(args.steps, args.warmup)
    for _ in range(args.warmup):
        cpu_oracle_sample(per_step, name)
    for _ in range(args.steps):
        v, desc, cores = cpu_oracle_sample(per_step, name)
        vals.append(v)
    value = statistics.mean(vals)
    from draft_token_markov_gb300 import workloads as W
    w = W.BY_NAME[name]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * w.steps / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, shaped like the pages' DeepSeek-V4.1 Markov head)",
        "config": {"workload": w.name, "sample": "one live row per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from draft_token_markov_gb300 import api
    from draft_token_markov_gb300 import workloads as W

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload
    w = W.BY_NAME[name]
    if args.rows:
        w = W.with_rows(w, args.rows)
    base_f32, cache_f32 = args.base_dtype == "f32", args.cache_dtype == "f32"
    head, embed = W.make_weights(w)
    inp = W.make_call(w, base_f32=base_f32)
    head, embed = head.to(dev), embed.to(dev)
    d = {k: v.to(dev) for k, v in inp.items()}
    R, N, V = w.rows, w.steps, w.vocab
    S = args.shards
    if S:
        # the vocabulary-sharded chain, its S ranks emulated on this GPU: each
        # rank's head rows in an allocation of their own, per-rank outputs
        if w.mode != W.GUMBEL or base_f32 or cache_f32:
            raise SystemExit("--shards takes a Gumbel workload with BF16 base and cache")
        plan = api.ShardPlan(w.vocab, w.rank, w.steps, w.rows, S, device=local)
        heads = [head[k * V // S:(k + 1) * V // S].clone() for k in range(S)]
        toks_l = [torch.full((R, N), -1, dtype=torch.int64, device=dev) for _ in range(S)]
        caches_l = [torch.empty((R, N, V), dtype=torch.bfloat16, device=dev) for _ in range(S)]
        toks = toks_l[0]
        status = api.markov_shard_plan_status
    else:
        plan = api.Plan(w.vocab, w.rank, w.steps, w.rows, device=local)
        plan.set_path({"auto": 0, "chain": 1, "batch": 2, "simple": 3}[args.path])
        toks = torch.full((R, N), -1, dtype=torch.int64, device=dev)
        cache = torch.empty((R, N, V), dtype=torch.float32 if cache_f32 else torch.bfloat16,
                            device=dev)
        status = api.markov_plan_status
    live = int((inp["row_state_idx"] >= 0).sum())
    tokens_per_step = live * N
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    clean = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    def flush_l2(k):
        # write more than L2, then read a different buffer of the same size so
        # the lines left in L2 are clean (not timed)
        flush.fill_(k & 0xFF)
        clean.sum()

    stream = torch.cuda.current_stream(dev)
    L = api.lib()
    # --calls C: C distinct calls (fresh seeds and anchors, drawn up front and
    # staged on the device; the base logits are the workload's), one per step
    calls = None
    if args.calls:
        per = [W.make_call(w, k, base_f32=base_f32) for k in range(args.calls)]
        calls = {key: torch.stack([p[key] for p in per]).to(dev) for key in ("anchor", "seeds")}
    call_no = [0]

    def step(evs=None):
        # one call: the persistent chain kernel draws the noise itself while
        # the head streams in, so a step is a single launch
        anchor, seeds = d["anchor"], d["seeds"]
        if calls is not None:
            k = call_no[0] % args.calls
            call_no[0] += 1
            anchor, seeds = calls["anchor"][k], calls["seeds"][k]
        if evs:
            evs[0].record(stream)
        if S:
            api.markov_chain_sample_sharded(plan, d["base"], heads, embed, anchor,
                                            d["temperature"], seeds, d["row_state_idx"], w.mult,
                                            w.cap, toks_l, caches_l, stream)
        else:
            api.markov_chain_sample(plan, d["base"], head, embed, anchor, d["temperature"],
                                    seeds, d["row_state_idx"], w.mode, w.mult, w.cap, toks,
                                    cache, stream)
        if evs:
            evs[1].record(stream)

    for _ in range(max(args.warmup, 3)):
        flush_l2(1)
        step()
    torch.cuda.synchronize()
    st = status(plan)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    if S:
        launches_per_step = S + 1          # each rank's noise, then the chain
        path = f"vocab-sharded chain ({S} ranks emulated on one GPU)"
    else:
        launches_per_step = plan.query(api.Q_LAST_LAUNCHES)
        path = {1: "tcgen05 chain", 2: "batch", 3: "simple chain"}.get(plan.query(api.Q_LAST_PATH), "?")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # the same loop untimed for a few hundred ms first, so that the
        # sampler (20 ms period) sees the load; its window covers this lead-in
        # and the timed steps
        clocks.mark_start()
        t_lead = time.time()
        while time.time() - t_lead < args.clock_lead_s:
            for k in range(20):
                flush_l2(k)
                step()
            torch.cuda.synchronize()
        call_no[0] = 0
        for k in range(args.steps):
            flush_l2(k)
            step(ev[k])
        torch.cuda.synchronize()
        clocks.mark_end()
    if world > 1:
        dist.barrier()
    st = status(plan)
    if st != 0:
        raise RuntimeError(f"device status {st} in the timed region")
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    chain_ms = step_ms
    # warm: the same calls back to back, no flush between them (reported
    # beside the cold headline)
    warm_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(min(args.steps, 50))]
    for e in warm_ev:
        step(e)
    torch.cuda.synchronize()
    warm_ms = [e[0].elapsed_time(e[1]) for e in warm_ev]
    total_ms = max_over_ranks(sum(step_ms))

    # end to end: the step's inputs in pinned host memory and its tokens back
    # in host memory, per step.  The chain paths take the host arguments
    # directly (the kernels read the inputs and write the tokens over the
    # host link); the per-position path, whose kernels re-read the base
    # logits at every position, copies them in first and the tokens out.
    h_in = {k: v.pin_memory() for k, v in inp.items()}
    h_tok = torch.empty((R, N), dtype=torch.int64).pin_memory()
    e2e_host = not S and path != "batch"
    e2e_ms = []
    for k in range(max(3, min(args.steps, 50)) + 3):
        flush_l2(k)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if e2e_host:
            api.markov_chain_sample(plan, h_in["base"], head, embed, h_in["anchor"],
                                    h_in["temperature"], h_in["seeds"], h_in["row_state_idx"],
                                    w.mode, w.mult, w.cap, h_tok, cache, stream)
        else:
            for key in d:
                d[key].copy_(h_in[key], non_blocking=True)
            step()
            h_tok.copy_(toks, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if k >= 3:
            e2e_ms.append(e0.elapsed_time(e1))
    if e2e_host and status(plan) != 0:
        raise RuntimeError("device status after the end-to-end steps")
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = h_tok.numel() * h_tok.element_size()

    peak, peak_kind = _peaks()
    alg_bytes = W.algorithmic_bytes(w, 4 if base_f32 else 2, 4 if cache_f32 else 2)
    typed = base_f32 or cache_f32
    chain_avg_s = statistics.mean(chain_ms) / 1000.0
    achieved = alg_bytes / chain_avg_s / 1e9
    traffic = None if (typed or S) else _traffic()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, cores = cpu_oracle_sample(args.cpu_seconds, name)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
        v1, desc1, _ = cpu_oracle_sample(max(2.0, args.cpu_seconds / 3.0), name, threads=1)
        cpu["single_thread"] = {"value": v1, "unit": UNIT, "sample": desc1}
    ms_per_step = total_ms / args.steps
    value = tokens_per_step * world * args.steps / (total_ms / 1000.0)
    e2e_step = statistics.mean(e2e_ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if not typed else f"{args.base_dtype} base, {args.cache_dtype} cache",
        "data": "synthetic (seeded, shaped like the pages' DeepSeek-V4.1 Markov head; "
                "random weights)",
        "config": {"workload": w.name, "rows": R, "live_rows": live, "vocab": V, "rank": w.rank,
                   "steps_per_call": N,
                   "mode": "gumbel" if w.mode == W.GUMBEL else "inverse cdf", "l2": "flushed before every step (256 MB write, then a 256 MB read of another buffer)",
                   "parallelism": f"replicas x{world}", "path": path,
                   "distinct_calls": args.calls or 1,
                   "resident_head_bytes": 0 if S else plan.query(api.Q_RESIDENT_HEAD_BYTES)},
        "us_per_call": {"median": statistics.median(step_ms) * 1000.0,
                        "p99": sorted(step_ms)[min(len(step_ms) - 1,
                                                   int(0.99 * len(step_ms)))] * 1000.0,
                        "chain_kernel_median": statistics.median(chain_ms) * 1000.0,
                        "warm_median": statistics.median(warm_ms) * 1000.0},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "frac_of_nominal_8000_gbs": achieved / 8000.0,
                     "kernel": "sharded_chain_kernel" if S else
                               {"tcgen05 chain": "chain_tc_kernel", "simple chain": "chain_kernel",
                                "batch": "batch kernels"}.get(path, path),
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "peak_kind": peak_kind},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens_per_step / (e2e_step / 1000.0), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_step,
                "inputs": ("pinned host memory, read by the kernels over the host link; tokens "
                           "written to pinned host memory" if e2e_host else
                           "copied from pinned host memory; tokens copied back")},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line))
    plan.close()
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--clock-lead-s", type=float, default=0.3,
                    help="seconds of untimed steps inside the clock-sampling window before the "
                         "timed steps")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--base-dtype", default="bf16", choices=["bf16", "f32"],
                    help="element type of the base logits")
    ap.add_argument("--cache-dtype", default="bf16", choices=["bf16", "f32"],
                    help="element type of the logits cache")
    ap.add_argument("--path", default="auto", choices=["auto", "chain", "batch", "simple"],
                    help="force a path (default: the library's automatic choice)")
    ap.add_argument("--calls", type=int, default=0,
                    help="time this many distinct calls (fresh seeds and anchors per call, staged "
                         "on the device up front), one per timed step; sets --steps")
    ap.add_argument("--shards", type=int, default=0, choices=[0, 1, 2, 4, 8],
                    help="run the vocabulary-sharded chain with this many ranks emulated on "
                         "the one GPU (Gumbel workloads)")
    ap.add_argument("--rows", type=int, default=0,
                    help="run the workload with this many rows instead of its own")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=WORKLOAD_NAMES,
                    help="deepseek (default, the headline): V=129280 r=256 8 rows N=8; "
                         "latency: 1 row; softcap: V=262144 r=128 inverse CDF; batch: 64 rows "
                         "(the per-position path); tiny: V=4096 r=64")
    args = ap.parse_args()
    if args.calls:
        args.steps = args.calls
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
