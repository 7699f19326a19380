#!/usr/bin/env python
"""Benchmark of split-KV decode attention on one GB300 (or N replicas).

Workload timed by default: the unified-cache multi-sequence decode -- a
shared fp16 cell-major cache of 262144 rows x 8 KV heads x 128 (1 GiB of K+V),
8 sequences with one query token and 32 q heads each, every sequence reading
its own 32768 rows through a sorted row list (the cache's rows are split among
the sequences).  One step = one skv_attn_partial call: split planning, the
gathered-row split-KV decode kernel and the log-sum-exp combine.

Printed: one JSON line (rank 0) with the throughput in GB/s of algorithmic
K/V bytes, the decode kernel's roofline fraction against the measured HBM
copy bandwidth, an end-to-end number through the C ABI with the inputs copied
from pinned host memory every step, the fp64 CPU oracle timed on a bounded
sample on the host cores, and the SM clocks sampled during the timed region.
``--impl reference`` times the CPU oracle as the reference arm instead.

Extra measurements (window + host tail stream with q8_0/q4_0 rows, pinned
host->device copy bandwidth, the tensor-core prefill chunk, block-sparse decode
through the block cache, KV appends, tiny decode latency) go under "extra".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn KV GB/s & % of HBM roofline; tail H2D GB/s; tokens·heads/s"
WORKLOAD = "unified_cache_multiseq_decode"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extras", action="store_true")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline sample")
    p.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                   help="run one kernel case twice (no timing, no JSON line): the command profiles/ captures")
    return p.parse_args()


PROFILE_CASES = ("decode_unified", "decode_q8q4_window", "prefill_window", "prefill_q8q4_window",
                 "prefill_row_list", "append_q8_0", "block_sparse_warm")


def run_profile_case(name: str) -> int:
    """One workload's call, twice (the second is the one a profiler captures),
    with the inputs the bench times: the unified-cache decode, the q8_0/q4_0
    long-context window (131072 rows), the prefill chunk's window (512 tokens
    over 32768 fp16 keys), the same prefill over q8_0-K / q4_0-V rows, the
    8-sequence row-list prefill over the unified cache, a 32768-row q8_0
    append, and a warm block-sparse call through the block cache (three
    warm-up calls first, so the profiled calls see the steady state)."""
    import torch
    import split_kv_flash_attn_gb300 as skv
    from split_kv_flash_attn_gb300 import build as skv_build
    from split_kv_flash_attn_gb300 import workloads as wl
    if not os.path.exists(skv_build.LIB):
        skv_build.build()
    h = skv.Handle(0)
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()   # noqa: E731
    if name == "decode_unified":
        w = wl.unified_decode()
        q, k, v, rows = cu(w.q), cu(w.k), cu(w.v), cu(w.kv_rows)
        call = lambda: skv.attn_partial(h, q, k, v, Hk=w.Hk, kv_rows=rows)   # noqa: E731
    elif name == "decode_q8q4_window":
        w = wl.long_context_decode()
        q, k, v = cu(w.q), cu(w.k), cu(w.v)
        call = lambda: skv.attn_partial(h, q, k, v, Hk=w.Hk, k_type=w.k_type, v_type=w.v_type)   # noqa: E731
    elif name == "prefill_window":
        w = wl.prefill_chunk()
        q, k, v, qp = cu(w.q), cu(w.k), cu(w.v), cu(w.q_pos)
        call = lambda: skv.attn_partial(h, q, k, v, Hk=w.Hk, q_pos=qp)   # noqa: E731
    elif name == "prefill_q8q4_window":
        w = wl.prefill_quant_window()
        q, k, v, qp = cu(w.q), cu(w.k), cu(w.v), cu(w.q_pos)
        call = lambda: skv.attn_partial(h, q, k, v, Hk=w.Hk, k_type=w.k_type, v_type=w.v_type, q_pos=qp)   # noqa: E731
    elif name == "prefill_row_list":
        w = wl.prefill_row_lists()
        q, k, v, rows, qp = cu(w.q), cu(w.k), cu(w.v), cu(w.kv_rows), cu(w.q_pos)
        call = lambda: skv.attn_partial(h, q, k, v, Hk=w.Hk, kv_rows=rows, q_pos=qp)   # noqa: E731
    elif name == "block_sparse_warm":
        w = wl.block_sparse_decode()
        sel = w.extra["sel"]
        hk, hv = torch.from_numpy(w.k).pin_memory(), torch.from_numpy(w.v).pin_memory()
        c = skv.BlockCache(h, hk, hv, n_blocks=w.extra["n_blocks"], block_rows=64, Hk=w.Hk, D=w.D,
                           n_slots=w.extra["cache_pages"], max_lookups=sel.size)
        q, sel_d = cu(w.q), cu(sel)
        for _ in range(3):
            c.attn(q, sel_d)
        call = lambda: c.attn(q, sel_d)   # noqa: E731
    else:
        rng = wl.generator(6, salt=7)
        Hk, D, n = 8, 128, 32768
        x = cu(wl.new_kv_values(rng, n, Hk, D)[0])
        pos = torch.arange(n, dtype=torch.int32, device="cuda")
        dst = torch.empty((n, Hk * wl.segment_bytes(wl.Q8_0, D)), dtype=torch.uint8, device="cuda")
        call = lambda: skv.kv_append(h, x, pos, dst, None, type_=wl.Q8_0, n_rows0=n, n_rows1=0)   # noqa: E731
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    h.status()
    print(f"profile case {name}: ok")
    return 0


def cpu_model() -> str:
    """The host CPU's model line from /proc/cpuinfo (Arm parts give their
    implementer and part numbers instead of a name)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "Hardware"):
        for line in info:
            if line.split(":")[0].strip() == key and ":" in line:
                return line.split(":", 1)[1].strip()
    impl = [ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU implementer")]
    part = [ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU part")]
    if impl and part:
        return f"arm implementer {impl[0]} part {part[0]}"
    return "unknown"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (getattr(self, "out", "") or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def profile_traffic(kernel_src: str, profile_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now (its sha256 prefix is recorded beside it)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        txt = open(path).read()
        with open(kernel_src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        rec = {}
        for line in txt.splitlines():
            if ":" in line and line.strip().startswith(("- ", "* ")):
                k, v = line.strip()[2:].split(":", 1)
                rec[k.strip()] = v.strip().strip("`")
        if rec.get("kernel_source_sha256") == sha and "dram_bytes_per_launch_full_size" in rec:
            return float(rec["dram_bytes_per_launch_full_size"])
    except Exception:
        pass
    return None


def reduce_max(x: float, world: int, device: str) -> float:
    """Maximum of a per-rank number over all ranks (the slowest replica sets
    the job's step time)."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: int, world: int, step_ms: float) -> float:
    """Whole-job GB/s: every replica moves bytes_per_rank per step, and the
    step takes the slowest replica's time (weak scaling)."""
    return bytes_per_rank * world / (step_ms * 1e-3) / 1e9


# ---------------------------------------------------------------- shared by both arms

def workload_config(n_gpus: int) -> dict:
    """The config dict both arms print (same workload, same keys)."""
    return {"workload": WORKLOAD, "S": 8, "nq": 1, "H": 32, "Hk": 8, "D": 128, "n_cache": 262144,
            "rows_per_seq": 32768, "kv_dtype": "f16",
            "l2": "inputs larger than L2: 1 GiB of K/V gathered per step vs 126 MB L2",
            "parallelism": f"replicas x{n_gpus}"}


def time_oracle(w, n_warm: int, n_timed: int):
    """The fp64 CPU oracle on the unified-cache workload, one sequence per
    call (sequence i % 8 for call i), timed call by call on all host cores.
    Returns (seconds of each timed call, K+V bytes one call gathers, threads)."""
    import oracle
    oracle.build()
    bytes_per_seq = int((w.kv_rows[0] >= 0).sum()) * w.Hk * w.D * 2 * 2
    times = []
    for i in range(n_warm + n_timed):
        s = i % w.S
        t0 = time.perf_counter()
        oracle.attention(w.q[s:s + 1], D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v,
                         n_rows0=w.k.shape[0], k_row_bytes0=w.k.shape[1], v_row_bytes0=w.v.shape[1],
                         n_keys=w.n_keys, kv_rows=w.kv_rows[s:s + 1])
        if i >= n_warm:
            times.append(time.perf_counter() - t0)
    return times, bytes_per_seq, oracle.max_threads()


def oracle_baseline(times, bytes_per_seq, threads) -> dict:
    med = statistics.median(times)
    return {"value": bytes_per_seq / med / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(times)} timed calls (after warm-up), each one of the 8 sequences in turn: 32 q heads x "
                      f"32768 gathered rows x 8 KV heads ({bytes_per_seq} B of K+V); value from the median call",
            "median_s": med, "min_s": min(times), "max_s": max(times), "cpu_model": cpu_model()}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from split_kv_flash_attn_gb300 import workloads as wl
    w = wl.unified_decode()
    times, bytes_per_seq, threads = time_oracle(w, args.warmup, args.steps)
    cpu = oracle_baseline(times, bytes_per_seq, threads)
    value = cpu["value"]
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": cpu["median_s"] * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.gpus),
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def main():
    args = parse()
    if args.profile_case:
        return run_profile_case(args.profile_case)
    if args.impl == "reference":
        return run_reference(args)
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from split_kv_flash_attn_gb300 import build as skv_build
    if not os.path.exists(skv_build.LIB):
        skv_build.build()
    import split_kv_flash_attn_gb300 as skv
    from split_kv_flash_attn_gb300 import workloads as wl

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, world, "cuda")

    hbm_peak, _, peak_kind = peaks()
    w = wl.unified_decode()
    h = skv.Handle(local)
    q = torch.from_numpy(w.q).cuda()
    K = torch.from_numpy(w.k).cuda()
    V = torch.from_numpy(w.v).cuda()
    rows = torch.from_numpy(w.kv_rows).cuda()
    o = torch.empty((w.S, 1, w.H, w.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.S, 1, w.H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    n_valid = int((w.kv_rows >= 0).sum())
    algo_bytes = n_valid * w.Hk * w.D * 2 * 2              # K + V head segments actually gathered
    tokens_heads = w.S * w.H

    def step():
        skv.attn_partial(h, q, K, V, Hk=w.Hk, kv_rows=rows, o=o, lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K_ = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_)]
    for a, b in kev:                        # materialise the events before handing them to the library
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        for i in range(K_):
            ev[i][0].record(stream)
            h.set_profile_events(kev[i][0], kev[i][1])
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
    h.set_profile_events(None, None)
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K_
    kern_ms = sum(a.elapsed_time(b) for a, b in kev) / K_
    step_ms = max_over_ranks(step_ms)
    value = job_throughput(algo_bytes, world, step_ms)
    achieved = algo_bytes / (kern_ms * 1e-3) / 1e9
    launches_per_step = 1          # the split merge runs inside the decode kernel

    # ---- end to end through the C ABI with host buffers ---------------------
    e2e = None
    try:
        hq, hK, hV, hrows = (torch.from_numpy(x).pin_memory() for x in (w.q, w.k, w.v, w.kv_rows))
        ho = torch.empty(o.shape, dtype=torch.float32).pin_memory()
        hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        dq, dK, dV, drows = (torch.empty_like(x, device="cuda") for x in (hq, hK, hV, hrows))

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dK.copy_(hK, non_blocking=True)
            dV.copy_(hV, non_blocking=True)
            drows.copy_(hrows, non_blocking=True)
            skv.attn_partial(h, dq, dK, dV, Hk=w.Hk, kv_rows=drows, o=o, lse=lse, stream=stream)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, min(K_ // 2, 40))
        barrier()
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hK, hV, hrows))
        d2h = ho.numel() * 4 + hl.numel() * 4
        e2e = {"value": job_throughput(algo_bytes, world, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        del hK, hV, dK, dV
    except Exception as exc:  # noqa: BLE001 -- report, do not lose the main line
        e2e = {"value": None, "unit": "GB/s", "error": repr(exc)[:200]}

    # ---- CPU oracle baseline on a bounded sample (rank 0) --------------------
    cpu = None
    if rank == 0 and not args.no_cpu:
        try:
            cpu = oracle_baseline(*time_oracle(w, 1, 6))
        except Exception as exc:  # noqa: BLE001
            cpu = {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle", "sample": repr(exc)[:200]}

    extra = {}
    if not args.no_extras and rank == 0:
        extra = run_extras(torch, skv, wl, h, hbm_peak)

    traffic = profile_traffic(os.path.join(ROOT, "split_kv_flash_attn_gb300", "csrc", "decode_kernel.cuh"),
                              "splitkv_decode_unified_cache.md")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K_, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": workload_config(world),
        "tokens_heads_per_s": tokens_heads * world / (step_ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "kernel": "splitkv_decode_kernel<128,f16,f16>", "kernel_ms": kern_ms,
                     "peak_kind": f"{peak_kind} (hbm_gbs, STREAM-style copy)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K_,
        "clocks": clk.summary(),
        "extra": extra,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_extras(torch, skv, wl, h, hbm_peak):
    """Window + host-tail decode with q8_0 K / q4_0 V (1,048,576 rows), the
    pinned host->device copy bandwidth at the tail's tile size, and the tiny
    decode's latency."""
    out = {}
    stream = torch.cuda.current_stream()
    try:
        w = wl.long_context_decode()
        q = torch.from_numpy(w.q).cuda()
        kw_, vw_ = torch.from_numpy(w.k).cuda(), torch.from_numpy(w.v).cuda()
        kt, vt = torch.from_numpy(w.k_tail).pin_memory(), torch.from_numpy(w.v_tail).pin_memory()
        o = torch.empty((1, 1, w.H, w.D), dtype=torch.float32, device="cuda")
        lse = torch.empty((1, 1, w.H), dtype=torch.float32, device="cuda")
        # window alone: the decode kernel over 131072 quantised rows in HBM
        b, a = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b.record(stream)
        a.record(stream)
        for _ in range(3):
            skv.attn_partial(h, q, kw_, vw_, Hk=w.Hk, k_type=w.k_type, v_type=w.v_type, o=o, lse=lse)
        torch.cuda.synchronize()
        h.set_profile_events(b, a)
        ks = []
        for _ in range(10):
            skv.attn_partial(h, q, kw_, vw_, Hk=w.Hk, k_type=w.k_type, v_type=w.v_type, o=o, lse=lse)
            torch.cuda.synchronize()
            ks.append(b.elapsed_time(a))
        h.set_profile_events(None, None)
        win_bytes = w.k.nbytes + w.v.nbytes
        win_ms = statistics.median(ks)
        # the whole window call: the decode kernel plus the combine of its splits
        call_ms = _time_calls(torch, lambda: skv.attn_partial(h, q, kw_, vw_, Hk=w.Hk, k_type=w.k_type,
                                                              v_type=w.v_type, o=o, lse=lse), 20)
        out["long_context_window"] = {"rows": w.k.shape[0], "bytes": win_bytes, "kernel_ms": win_ms,
                                      "GBps": win_bytes / win_ms / 1e6, "frac_hbm": win_bytes / win_ms / 1e6 / hbm_peak,
                                      "call_ms": call_ms, "call_GBps": win_bytes / call_ms / 1e6}
        # whole call: window + 28 streamed tail tiles + combine
        for _ in range(2):
            skv.attn_window_tail(h, q, kw_, vw_, kt, vt, Hk=w.Hk, tile_rows=w.tile_rows, k_type=w.k_type,
                                 v_type=w.v_type, o=o, lse=lse)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = 5
        for _ in range(n):
            skv.attn_window_tail(h, q, kw_, vw_, kt, vt, Hk=w.Hk, tile_rows=w.tile_rows, k_type=w.k_type,
                                 v_type=w.v_type, o=o, lse=lse)
        e1.record(stream)
        torch.cuda.synchronize()
        call_ms = e0.elapsed_time(e1) / n
        tail_bytes = w.k_tail.nbytes + w.v_tail.nbytes
        # pinned H2D microbenchmark with the same transfer sizes (one K and one V tile copy)
        tk = w.tile_rows * w.k.shape[1]
        tv = w.tile_rows * w.v.shape[1]
        dst = torch.empty(tk + tv, dtype=torch.uint8, device="cuda")
        src = torch.from_numpy(np.ascontiguousarray(w.k_tail[:w.tile_rows]).reshape(-1)).pin_memory()
        srcv = torch.from_numpy(np.ascontiguousarray(w.v_tail[:w.tile_rows]).reshape(-1)).pin_memory()
        for _ in range(3):
            dst[:tk].copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0.record(stream)
        reps = 20
        for _ in range(reps):
            dst[:tk].copy_(src, non_blocking=True)
            dst[tk:].copy_(srcv, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = reps * (tk + tv) / (e0.elapsed_time(e1) * 1e-3) / 1e9
        tail_gbs = tail_bytes / (call_ms * 1e-3) / 1e9
        # the call can take no less than the longer of the window kernel and
        # the tail's copy at the pinned H2D rate
        bound_ms = max(win_ms, tail_bytes / (h2d_gbs * 1e9) * 1e3)
        out["long_context_window_tail"] = {
            "n_kv": w.extra["n_kv"], "wc": w.extra["wc"], "tile_rows": w.tile_rows, "tail_bytes": tail_bytes,
            "call_ms": call_ms, "tail_stream_GBps": tail_gbs, "pinned_h2d_GBps": h2d_gbs,
            "frac_of_pinned_h2d": tail_gbs / h2d_gbs, "bound_ms": bound_ms, "frac_of_bound": bound_ms / call_ms,
            "tokens_heads_per_s": w.H / (call_ms * 1e-3)}
        del kw_, vw_, kt, vt, dst, src, srcv
    except Exception as exc:  # noqa: BLE001
        out["long_context_error"] = repr(exc)[:300]
    try:
        out["prefill_chunk"] = bench_prefill(torch, skv, wl, h)
    except Exception as exc:  # noqa: BLE001
        out["prefill_error"] = repr(exc)[:300]
    try:
        bs = bench_block_sparse(torch, skv, wl, h, hbm_peak)
        h2d = out.get("long_context_window_tail", {}).get("pinned_h2d_GBps")
        if h2d:
            # hits read from HBM, misses cross the host link: serial and
            # overlapped lower bounds on a warm call
            miss_b = bs["warm_miss_pages_per_call"] * bs["page_bytes"]
            hit_b = bs["call_bytes"] - miss_b
            t_hit, t_miss = hit_b / (hbm_peak * 1e9) * 1e3, miss_b / (h2d * 1e9) * 1e3
            bs.update({"bound_ms_serial": t_hit + t_miss, "bound_ms_overlapped": max(t_hit, t_miss),
                       "frac_of_serial_bound": (t_hit + t_miss) / bs["warm_ms"],
                       "frac_of_overlapped_bound": max(t_hit, t_miss) / bs["warm_ms"]})
        out["block_sparse"] = bs
    except Exception as exc:  # noqa: BLE001
        out["block_sparse_error"] = repr(exc)[:300]
    try:
        out["prefill_variants"] = bench_prefill_variants(torch, skv, wl, h)
    except Exception as exc:  # noqa: BLE001
        out["prefill_variants_error"] = repr(exc)[:300]
    try:
        out["kv_append"] = bench_append(torch, skv, wl, h, hbm_peak)
    except Exception as exc:  # noqa: BLE001
        out["kv_append_error"] = repr(exc)[:300]
    try:
        w = wl.tiny_decode()
        q = torch.from_numpy(w.q).cuda()
        kw_, vw_ = torch.from_numpy(w.k).cuda(), torch.from_numpy(w.v).cuda()
        kt, vt = torch.from_numpy(w.k_tail).pin_memory(), torch.from_numpy(w.v_tail).pin_memory()
        o_t = torch.empty((1, 1, w.H, w.D), dtype=torch.float32, device="cuda")
        l_t = torch.empty((1, 1, w.H), dtype=torch.float32, device="cuda")
        for _ in range(5):
            skv.attn_window_tail(h, q, kw_, vw_, kt, vt, Hk=w.Hk, tile_rows=w.tile_rows, o=o_t, lse=l_t)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = 50
        for _ in range(n):   # a decode loop: outputs reused, every call through the Python binding
            skv.attn_window_tail(h, q, kw_, vw_, kt, vt, Hk=w.Hk, tile_rows=w.tile_rows, o=o_t, lse=l_t)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / n * 1e3
        # the same call captured once in a CUDA graph and replayed: what the
        # device needs per call once the host's per-call API work is gone
        cs = torch.cuda.Stream()
        o_g = torch.empty((1, 1, w.H, w.D), dtype=torch.float32, device="cuda")
        l_g = torch.empty((1, 1, w.H), dtype=torch.float32, device="cuda")
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            skv.attn_window_tail(h, q, kw_, vw_, kt, vt, Hk=w.Hk, tile_rows=w.tile_rows, o=o_g, lse=l_g, stream=cs)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs, capture_error_mode="thread_local"):
            skv.attn_window_tail(h, q, kw_, vw_, kt, vt, Hk=w.Hk, tile_rows=w.tile_rows, o=o_g, lse=l_g, stream=cs)
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        g_us = e0.elapsed_time(e1) / n * 1e3
        out["tiny_decode_window_tail"] = {"us_per_call": us, "tokens_heads_per_s": w.H / (us * 1e-6),
                                          "graph_replay_us_per_call": g_us}
    except Exception as exc:  # noqa: BLE001
        out["tiny_error"] = repr(exc)[:300]
    return out


def _time_calls(torch, fn, n, warm=2):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(n):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def _graph_us(torch, fn, per_graph=50, replays=20):
    """Device time of one call of fn (a launch-bound call), from a CUDA graph
    holding per_graph calls replayed `replays` times."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            fn()
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(replays):
        g.replay()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (per_graph * replays)


def bench_prefill(torch, skv, wl, h):
    """Prefill chunk: 512 causal tokens x 32 heads over 65536 keys (32768 in
    HBM + a 32768-row pinned tail in 8192-row tiles).  The tensor-core kernel
    alone is timed on the window (every key visible to every token)."""
    _, bf16_peak, kind = peaks()
    w = wl.prefill_chunk()
    q = torch.from_numpy(w.q).cuda()
    kw_, vw_ = torch.from_numpy(w.k).cuda(), torch.from_numpy(w.v).cuda()
    kt, vt = torch.from_numpy(w.k_tail).pin_memory(), torch.from_numpy(w.v_tail).pin_memory()
    qp = torch.from_numpy(w.q_pos).cuda()
    o = torch.empty((1, w.nq, w.H, w.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, w.nq, w.H), dtype=torch.float32, device="cuda")
    rows_q = w.nq * w.H
    n_win = w.k.shape[0]
    win_flop = 4.0 * w.D * rows_q * n_win
    b, a = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    b.record(s)
    a.record(s)
    for _ in range(2):
        skv.attn_partial(h, q, kw_, vw_, Hk=w.Hk, q_pos=qp, o=o, lse=lse)
    torch.cuda.synchronize()
    h.set_profile_events(b, a)
    ks = []
    for _ in range(5):
        skv.attn_partial(h, q, kw_, vw_, Hk=w.Hk, q_pos=qp, o=o, lse=lse)
        torch.cuda.synchronize()
        ks.append(b.elapsed_time(a))
    h.set_profile_events(None, None)
    k_ms = statistics.median(ks)
    # causal pairs of the whole chunk: token i at 65024+i sees keys 0..65024+i
    pos = w.q_pos.reshape(-1).astype(np.int64)
    total_flop = 4.0 * w.D * w.H * float((pos + 1).sum())
    call_ms = _time_calls(torch, lambda: skv.attn_window_tail(h, q, kw_, vw_, kt, vt, Hk=w.Hk,
                                                               tile_rows=w.tile_rows, q_pos=qp, o=o, lse=lse), 5)
    tail_bytes = w.k_tail.nbytes + w.v_tail.nbytes
    h.status()
    return {"kernel_ms_window": k_ms, "kernel_TFLOPs_window": win_flop / k_ms / 1e9,
            "frac_of_bf16_peak": win_flop / k_ms / 1e9 / bf16_peak, "peak_TFLOPs": bf16_peak,
            "peak_kind": f"{kind} bf16 dense (fp16 runs at the same tensor rate)",
            "call_ms_window_tail": call_ms, "call_TFLOPs": total_flop / call_ms / 1e9, "flop": total_flop,
            "tail_bytes": tail_bytes, "tail_GBps_if_copy_bound": tail_bytes / call_ms / 1e6}


def bench_prefill_variants(torch, skv, wl, h):
    """Tensor-core prefill with software producers: (a) 512 causal tokens x 32
    heads over a 32768-row q8_0-K / q4_0-V window (keys split exactly into two
    fp16 operands, so QK^T takes twice the MMAs); (b) 8 sequences x 64 tokens
    x 32 heads, each over its own 32768 rows of the 1 GiB unified fp16 cache
    through a row list.  FLOP counted as 4*D per (query row, visible key)."""
    _, bf16_peak, _ = peaks()
    out = {}
    s = torch.cuda.current_stream()
    b, a = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def kernel_ms(fn, n=5):
        fn()
        torch.cuda.synchronize()
        b.record(s)
        a.record(s)
        h.set_profile_events(b, a)
        ks = []
        for _ in range(n):
            fn()
            torch.cuda.synchronize()
            ks.append(b.elapsed_time(a))
        h.set_profile_events(None, None)
        return statistics.median(ks)

    wq = wl.prefill_quant_window()
    nq, H, Hk, D, n = wq.nq, wq.H, wq.Hk, wq.D, wq.n_keys
    q = torch.from_numpy(wq.q).cuda()
    K = torch.from_numpy(wq.k).cuda()
    V = torch.from_numpy(wq.v).cuda()
    qp = torch.from_numpy(wq.q_pos).cuda()
    o = torch.empty((1, nq, H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, nq, H), dtype=torch.float32, device="cuda")
    ms = kernel_ms(lambda: skv.attn_partial(h, q, K, V, Hk=Hk, k_type=wq.k_type, v_type=wq.v_type, q_pos=qp, o=o,
                                            lse=lse))
    pairs = float(np.arange(n - nq, n, dtype=np.int64).sum() + nq)
    flop = 4.0 * D * H * pairs
    out["quant_window_q8k_q4v"] = {"rows": n, "nq": nq, "kernel_ms": ms, "TFLOPs": flop / ms / 1e9,
                                   "frac_of_bf16_peak": flop / ms / 1e9 / bf16_peak,
                                   "bytes": K.numel() + V.numel()}
    del K, V
    w = wl.prefill_row_lists()
    S, nq2 = w.S, w.nq
    q2 = torch.from_numpy(w.q).cuda()
    kc, vc = torch.from_numpy(w.k).cuda(), torch.from_numpy(w.v).cuda()
    rows = torch.from_numpy(w.kv_rows).cuda()
    n_list = w.kv_rows.shape[1]
    qp2 = torch.from_numpy(w.q_pos).cuda()
    o2 = torch.empty((S, nq2, w.H, w.D), dtype=torch.float32, device="cuda")
    l2 = torch.empty((S, nq2, w.H), dtype=torch.float32, device="cuda")
    ms = kernel_ms(lambda: skv.attn_partial(h, q2, kc, vc, Hk=w.Hk, kv_rows=rows, q_pos=qp2, o=o2, lse=l2))
    pairs = S * float(np.arange(n_list - nq2, n_list, dtype=np.int64).sum() + nq2)
    flop = 4.0 * w.D * w.H * pairs
    out["row_list_unified_cache"] = {"S": S, "nq": nq2, "rows_per_seq": n_list, "kernel_ms": ms,
                                     "TFLOPs": flop / ms / 1e9, "frac_of_bf16_peak": flop / ms / 1e9 / bf16_peak,
                                     "gathered_GBps": S * n_list * w.Hk * w.D * 4 / ms / 1e6}
    h.status()
    return out


def bench_append(torch, skv, wl, h, hbm_peak):
    """KV append: a 32768-row chunk of fp32 K (8 KV heads x 128) written into
    a device window as fp16 / q8_0 / q4_0 (128 MiB read, more than L2), the
    same chunk as fp16 into a pinned host tail, one decode step's row, and the
    block cache's write-through append (host copy + resident pages)."""
    Hk, D, n = 8, 128, 32768
    rng = wl.generator(6, salt=7)
    k, _ = wl.new_kv_values(rng, n, Hk, D)
    x = torch.from_numpy(k).cuda()
    pos = torch.arange(n, dtype=torch.int32, device="cuda")
    out = {"rows": n, "Hk": Hk, "D": D}
    for name, t in (("f16", wl.F16), ("q8_0", wl.Q8_0), ("q4_0", wl.Q4_0)):
        rb = Hk * wl.segment_bytes(t, D)
        win = torch.empty((n, rb), dtype=torch.uint8, device="cuda")
        ms = _time_calls(torch, lambda: skv.kv_append(h, x, pos, win, None, type_=t, n_rows0=n, n_rows1=0), 10)
        moved = x.numel() * 4 + n * rb
        out[f"window_{name}"] = {"ms": ms, "bytes": moved, "GBps": moved / ms / 1e6,
                                 "frac_hbm": moved / ms / 1e6 / hbm_peak}
        del win
    rb = Hk * 2 * D
    tail = torch.empty((n, rb), dtype=torch.uint8).pin_memory()
    ms = _time_calls(torch, lambda: skv.kv_append(h, x, pos, None, tail, n_rows0=0, n_rows1=n), 5)
    out["tail_f16"] = {"ms": ms, "host_bytes_written": n * rb, "host_write_GBps": n * rb / ms / 1e6}
    win = torch.empty((n, rb), dtype=torch.uint8, device="cuda")
    one, x1 = pos[:1] + (n - 1), x[:1]
    out["decode_step_row_us"] = _graph_us(torch, lambda: skv.kv_append(h, x1, one, win, None, n_rows0=n, n_rows1=0))
    # block cache: 512 blocks of 64 rows, 256 resident pages; appends of one
    # decode row and of a 4096-row chunk
    nb, br = 512, 64
    hk = torch.zeros((nb, Hk, br, D), dtype=torch.float16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    c = skv.BlockCache(h, hk, hv, n_blocks=nb, block_rows=br, Hk=Hk, D=D, n_slots=256, max_lookups=Hk * 32)
    sel = torch.from_numpy(np.stack([np.arange(32, dtype=np.int32) * 16] * Hk)[None]).cuda()
    c.resolve(sel)
    chunk = 4096
    xc = x[:chunk]
    pc = torch.arange(chunk, dtype=torch.int32, device="cuda") * 8      # spread over all blocks
    ms = _time_calls(torch, lambda: c.append(xc, xc, pc), 5)
    out["bcache_chunk"] = {"rows": chunk, "ms": ms, "host_bytes_written": 2 * chunk * rb,
                           "host_write_GBps": 2 * chunk * rb / ms / 1e6}
    p1 = pc[:1]
    out["bcache_decode_row_us"] = _graph_us(torch, lambda: c.append(x1, x1, p1))
    c.close()
    # ring layout: a 128-block ring (8192 cells) over the same host copy; one
    # decode step = append one row + attention of 32 q heads over the last
    # 4096 cells through the ring
    r = skv.BlockCache(h, hk, hv, n_blocks=nb, block_rows=br, Hk=Hk, D=D, ring_blocks=128, max_seqs=1)
    n_keys = nb * br - 64
    r.ring_restore(n_keys)
    q = torch.from_numpy(wl.normal_f16(rng, (1, 1, 4 * Hk, D))).cuda()
    o = torch.empty((1, 1, 4 * Hk, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, 1, 4 * Hk), dtype=torch.float32, device="cuda")
    pn = torch.full((1,), n_keys, dtype=torch.int32, device="cuda")

    def ring_step():
        r.append(x1, x1, pn)
        r.ring_attn(q, n_keys + 1, 4096, o=o, lse=lse)
    us = _graph_us(torch, ring_step, per_graph=20, replays=20)
    out["ring_decode_step"] = {"window": 4096, "ring_cells": 128 * br, "us_per_step": us,
                               "tokens_heads_per_s": 4 * Hk / (us * 1e-6),
                               "kv_bytes_per_step": 4096 * Hk * 2 * D * 2}
    r.close()
    h.status()
    return out


def bench_block_sparse(torch, skv, wl, h, hbm_peak):
    """Block-sparse decode through the block cache: 4 sequences x 4 KV heads x
    512 selected 64-row blocks (268,435,456 B of K+V per call) from a pinned
    paged host cache of 262144 rows, 2048 resident pages.  Cold (after a
    reset), warm (same selection) and drift (10% of blocks redrawn per call)."""
    w = wl.block_sparse_decode()
    sel = w.extra["sel"]
    hk, hv = torch.from_numpy(w.k).pin_memory(), torch.from_numpy(w.v).pin_memory()
    c = skv.BlockCache(h, hk, hv, n_blocks=w.extra["n_blocks"], block_rows=64, Hk=w.Hk, D=w.D,
                       n_slots=w.extra["cache_pages"], max_lookups=w.S * w.Hk * sel.shape[-1])
    q = torch.from_numpy(w.q).cuda()
    o = torch.empty((w.S, 1, w.H, w.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.S, 1, w.H), dtype=torch.float32, device="cuda")
    sel_d = torch.from_numpy(sel).cuda()
    call_bytes = sel.size * 64 * w.D * 2 * 2
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # cold
    c.attn(q, sel_d, o=o, lse=lse)
    torch.cuda.synchronize()
    c.reset()
    e0.record(s)
    c.attn(q, sel_d, o=o, lse=lse)
    e1.record(s)
    torch.cuda.synchronize()
    cold_ms = e0.elapsed_time(e1)
    st0 = c.stats()
    warm_ms = _time_calls(torch, lambda: c.attn(q, sel_d, o=o, lse=lse), 8, warm=1)
    st1 = c.stats()
    rng = np.random.default_rng(5)
    sels = [sel]
    for _ in range(8):
        sels.append(wl.redraw_selection(sels[-1], w.extra["n_blocks"], 0.1, rng))
    sels_d = [torch.from_numpy(x).cuda() for x in sels[1:]]
    torch.cuda.synchronize()
    e0.record(s)
    for sd in sels_d:
        c.attn(q, sd, o=o, lse=lse)
    e1.record(s)
    torch.cuda.synchronize()
    drift_ms = e0.elapsed_time(e1) / len(sels_d)
    st2 = c.stats()
    violations = c.check()
    page_bytes = 64 * w.D * 2 * 2

    def hit_rate(a, b):
        look = b["lookups"] - a["lookups"]
        return (b["hits"] - a["hits"]) / max(1, look)
    warm_calls = st1["calls"] - st0["calls"]
    miss_pages_warm = (st1["misses"] - st0["misses"]) / max(1, warm_calls)
    c.close()
    return {"call_bytes": call_bytes, "page_bytes": page_bytes, "cold_ms": cold_ms, "warm_ms": warm_ms,
            "drift_ms": drift_ms,
            "cold_misses": st0["last_misses"], "warm_hit_rate": hit_rate(st0, st1),
            "warm_miss_pages_per_call": miss_pages_warm,
            "warm_miss_GBps": miss_pages_warm * page_bytes / warm_ms / 1e6,
            "drift_hit_rate": hit_rate(st1, st2), "effective_GBps_warm": call_bytes / warm_ms / 1e6,
            "tokens_heads_per_s_warm": w.S * w.H / (warm_ms * 1e-3), "invariant_violations": violations}


if __name__ == "__main__":
    sys.exit(main())
