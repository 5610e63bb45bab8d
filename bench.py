#!/usr/bin/env python
"""EntmaxKV decode-step benchmark.

One step = score_pages -> select -> decode (the whole decode hot path) for the
batched 128K-context workload: batch 8, 32 query / 8 kv heads, d = 128, 131072
tokens per sequence, pages of 32, bf16 K/V, 8 planted high-score pages per
(sequence, kv head), alpha = 1.5, 4096-token budget.  Inputs are seeded
synthetic data resident in HBM; the 4 GiB K/V pool is far larger than L2 and
L2 is also flushed (a 512 MiB write) between timed steps, outside the timed
events.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle on a
bounded sample of the same step instead.  With torchrun (N > 1) every rank runs
an independent replica (the path needs no collective); the time is the max over
ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse entmax decode µs/step and achieved HBM GB/s (frac of peak) at 128K ctx"
FULL_METRIC = "full-cache entmax decode µs/step and achieved HBM GB/s (frac of peak)"
MODE_METRIC = {
    "full": FULL_METRIC,
    "softmax": "sparse softmax decode (same kept pages) µs/step and achieved HBM GB/s",
    "softmax_full": "full-cache softmax decode µs/step and achieved HBM GB/s (frac of peak)",
}
FALLBACK_HBM_GBS = 6400.0
KERNELS_PER_STEP = 5   # score, select, plan, qk, tpv (threshold + values)


def kernels_per_step(w) -> int:
    """Kernel launches of one step: score, select, plan, qk, tpv -- without the
    plan where the top-k selection builds the page union itself (per-head or
    shared top-k over at most 4096 pages per sequence: one CTA per selection)."""
    planned = w.policy in ("topk", "topk_shared") and w.max_pages <= 4096
    return KERNELS_PER_STEP - (1 if planned else 0)


def parse():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="long128k")
    ap.add_argument("--alpha", type=float, default=None)
    ap.add_argument("--policy", choices=["topk", "gauss", "topk_shared"], default=None,
                    help="override the workload's selection policy")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch")
    ap.add_argument("--context", type=int, default=None, help="override the context length")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--mode", choices=["sparse", "full", "softmax", "softmax_full", "meta"],
                    default="sparse",
                    help="sparse: the EntmaxKV step (headline); full: full-cache entmax decode; "
                         "softmax: softmax over the same kept pages; softmax_full: full-cache "
                         "softmax; meta: the page-metadata build (prefill) alone")
    ap.add_argument("--cpu-1core", action="store_true",
                    help="also time the oracle on one host thread (cpu_baseline_1core)")
    ap.add_argument("--e2e-breakdown", action="store_true",
                    help="where the end-to-end step time goes: host wall clock of a tiny graph, "
                         "the device-only step graph and the host-buffer step, each with its sync")
    return ap.parse_args()


def overrides(args) -> dict:
    kw = {}
    if args.alpha is not None:
        kw["alpha"] = args.alpha
    if args.policy is not None:
        kw["policy"] = args.policy
    if args.batch is not None:
        kw["batch"] = args.batch
    if args.context is not None:
        kw["context"] = args.context
    return kw


# ---------------------------------------------------------------------------
# multi-rank helpers (replicas: every rank runs its own step, no data-path
# collective; only the timing is combined)
# ---------------------------------------------------------------------------
def rank_seed(workload: str, rank: int) -> int:
    """Each replica decodes its own synthetic cache."""
    from sparse_long_context_08_b300.workloads import CONFIGS
    return CONFIGS[workload]["seed"] + 1000 * rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (time of the timed region)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_step(ms_per_step_max: float, world: int) -> float:
    """World ranks each ran the timed steps within the slowest rank's time:
    microseconds per step of work over the whole job."""
    return ms_per_step_max * 1e3 / world


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_cpu_model() -> str:
    """The host CPU's model name (the oracle baseline's hardware)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def workload_config(w):
    return {"workload": f"{w.name}: batch {w.batch}, {w.num_q_heads} q / {w.num_kv_heads} kv heads, "
                        f"d={w.head_dim}, context {w.params['context']}, page {w.page_size}, "
                        f"{w.dtype} K/V, alpha={w.alpha}, policy {w.policy}, "
                        f"budget {w.budget_tokens} tokens",
            "batch": w.batch, "context": w.params["context"], "page_size": w.page_size,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "alpha": w.alpha, "policy": w.policy,
            "budget_tokens": w.budget_tokens, "kv_dtype": w.dtype, "seed": w.seed,
            "l2": "inputs (4 GiB K/V) larger than L2; L2 flushed between timed steps (512 MiB write, then 256 MiB read)"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.proc = None
        self.lines: list[str] = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if bus_id:
            cmd += ["-i", bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def bus_id_of(dev: int) -> str | None:
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


def measured_traffic(kernel: str, units: int):
    """DRAM bytes (read + write) of one launch of `kernel` that processes
    `units` (union pages for qk / pv, metadata pages for score), from the
    committed ncu summary's bytes per unit; None when there is no capture for
    the kernel or its source has changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            k = json.load(f)["kernels"][kernel]
        with open(os.path.join(ROOT, k["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != k["source_sha256"]:
                return None
        return int(round(float(k["bytes_per_unit"]) * units))
    except (OSError, KeyError, ValueError):
        return None


def timed_replays(graph, k: int, flush_l2) -> list[float]:
    """Device time (ms) of k replays of `graph`, each behind an L2 flush.

    Every replay is enqueued right behind the previous flush, with no host
    synchronisation in between, so the GPU is still busy flushing when the
    start event and the graph's kernels are enqueued: the events bracket the
    step's execution on the device, not the host's launch latency (which the
    end-to-end figure carries)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
    flush_l2(0)
    for i in range(k):
        starts[i].record()
        graph.replay()
        ends[i].record()
        flush_l2(i + 7)                    # the next step's flush, enqueued behind this one
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


# ---------------------------------------------------------------------------
# oracle (CPU) timing: the cpu_baseline leg and the reference arm
# ---------------------------------------------------------------------------
def oracle_time_per_step(w, seconds: float, steps: int | None = None):
    """Times the fp64 oracle's score -> select -> sparse attention on a bounded
    sample of query heads; returns (us per full step, sample description, cores,
    per-step list)."""
    import numpy as np
    import oracle
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)       # prefill work, not part of a decode step
    BH = w.batch * w.num_q_heads
    cores = oracle.get_threads()
    t0 = time.perf_counter()
    oracle.sparse_step(kv, w, heads=np.arange(min(BH, cores), dtype=np.int32), meta=meta)
    per_head = max(1e-6, (time.perf_counter() - t0) / min(BH, cores))  # wall time per head, parallel
    if steps is None:
        n_heads = BH
        reps = max(1, int(seconds / max(per_head * BH / max(1, cores), 1e-3)))
        reps = min(reps, 50)
    else:
        budget = seconds / max(1, steps)
        n_heads = int(min(BH, max(cores, budget / per_head * cores)))
        reps = steps
    rng = np.random.default_rng(0)
    times = []
    for _ in range(reps):
        heads = np.sort(rng.choice(BH, size=n_heads, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.sparse_step(kv, w, heads=heads, meta=meta)
        times.append((time.perf_counter() - t0) * 1e6 * BH / n_heads)
    desc = (f"{n_heads} of {BH} query heads per step (score, top-k/tau-hat select, sparse "
            f"attention; fp64), {reps} steps, scaled to a full step; metadata prebuilt")
    return statistics.mean(times), desc, cores, times


def oracle_full_time_per_step(w, seconds: float, steps: int = 1, mode: str = "full"):
    """Times the fp64 oracle's version of a variant (full-cache entmax, sparse
    softmax over the selected pages, full-cache softmax) on a bounded sample
    of query heads; returns (us per full step, sample description, cores)."""
    import numpy as np
    import oracle
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv) if mode == "softmax" else None   # prefill work, not timed
    BH = w.batch * w.num_q_heads
    cores = oracle.get_threads()
    s = float(w.scale)

    def run(heads):
        if mode == "full":
            oracle.decode_full(kv, s, w.alpha, heads=heads)
        elif mode == "softmax_full":
            oracle.decode_softmax(kv, s, full=True, heads=heads)
        else:
            r = oracle.sparse_step(kv, w, heads=heads, meta=meta)
            oracle.decode_softmax(kv, s, r["sel"], r["n_sel"], heads=heads)

    n0 = min(BH, cores)
    t0 = time.perf_counter()
    run(np.arange(n0, dtype=np.int32))
    per_head = max(1e-6, (time.perf_counter() - t0) / n0)        # wall time per head, parallel
    n_heads = int(min(BH, max(n0, seconds / max(1, steps) / per_head)))
    rng = np.random.default_rng(0)
    times = []
    for _ in range(steps):
        heads = np.sort(rng.choice(BH, size=n_heads, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        run(heads)
        times.append((time.perf_counter() - t0) * 1e6 * BH / n_heads)
    what = {"full": "full-cache scores, exact tau, attention",
            "softmax": "bound scores, top-k, softmax attention over the kept pages",
            "softmax_full": "full-cache scores, softmax attention"}[mode]
    desc = (f"{n_heads} of {BH} query heads per step ({what}; fp64), {steps} steps, scaled to a "
            f"full step" + ("; metadata prebuilt" if mode == "softmax" else ""))
    return statistics.mean(times), desc, cores


def selection_ties(w, sel, n_sel, heads, tie_rtol: float = 2e-5) -> dict:
    """The GPU page selection of `heads` against the fp64 oracle's: heads with
    the same page set, heads that differ only by pages whose oracle decision
    score lies within tie_rtol (relative to the score's magnitude) of the
    decision boundary, and heads that differ otherwise (a parity failure)."""
    import numpy as np
    import oracle
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    r = oracle.sparse_step(kv, w, heads=np.asarray(heads, dtype=np.int32), meta=meta)
    s = float(w.scale)
    G = w.group
    same = tied = other = 0
    for bh in heads:
        gs = set(sel[bh, :n_sel[bh]].tolist())
        os_ = set(r["sel"][bh, :r["n_sel"][bh]].tolist())
        if gs == os_:
            same += 1
            continue
        b, h = divmod(bh, w.num_q_heads)
        qa = np.abs(w.q[b, h].astype(np.float64))
        ok = True
        for p in gs ^ os_:
            blk = w.page_table[b, p]
            if w.policy == "gauss":
                c = w.alpha - 1.0
                mag = c * s * (np.abs(meta.mean[blk, h // G]) @ qa
                               + np.sqrt(meta.var[blk, h // G] @ (qa * qa))) + 1e-6
                zs = c * r["zmax"][bh]
                np_ = w.pages_of(b)
                passing = np.sort(zs[:np_][zs[:np_] >= r["tau_hat"][bh] - w.delta])[::-1]
                bnd = (passing[w.cap_pages - 1] if len(passing) > w.cap_pages
                       else r["tau_hat"][bh] - w.delta)
                score = zs[p]
            else:
                amp = np.maximum(np.abs(meta.kmin[blk]), np.abs(meta.kmax[blk]))
                gh = range(G) if w.policy == "topk_shared" else [h % G]
                mag = max(s * (amp[h // G] @ np.abs(w.q[b, (h // G) * G + g].astype(np.float64)))
                          for g in gh)
                score = (r["shared"][bh, p] if w.policy == "topk_shared" else r["bound"][bh, p])
                bnd = r["kth"][bh]
            ok = ok and abs(score - bnd) <= tie_rtol * mag
        if ok:
            tied += 1
        else:
            other += 1
    return {"heads_checked": len(heads), "identical": same, "ties_at_boundary": tied,
            "other_differences": other, "tie_window": f"{tie_rtol:g} of the score magnitude"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    from sparse_long_context_08_b300.workloads import make_workload
    w = make_workload(args.workload, **overrides(args))
    budget = 150.0
    if args.mode != "sparse":
        oracle_full_time_per_step(w, budget * 0.1, steps=max(1, min(args.warmup, 3)),
                                  mode=args.mode)
        us, desc, cores = oracle_full_time_per_step(w, budget, steps=max(1, min(args.steps, 5)),
                                                    mode=args.mode)
        line = {"metric": MODE_METRIC[args.mode], "impl": "reference", "value": us, "unit": "us/step",
                "n_gpus": args.gpus, "steps": max(1, min(args.steps, 5)), "warmup": args.warmup,
                "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": dict(workload_config(w), mode=args.mode),
                "cpu_baseline": {"value": us, "unit": "us/step", "cores": cores,
                                 "kind": "oracle", "sample": desc,
               "cpu_model": host_cpu_model()},
                "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return
    oracle_time_per_step(w, budget * 0.1, steps=max(1, args.warmup))   # warm-up steps
    us, desc, cores, _ = oracle_time_per_step(w, budget, steps=args.steps)
    line = {"metric": METRIC, "impl": "reference", "value": us, "unit": "us/step",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": us, "unit": "us/step", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from sparse_long_context_08_b300 import entmaxkv as E
    from sparse_long_context_08_b300.api import EntmaxKVDecoder, upload_workload
    from sparse_long_context_08_b300.workloads import make_workload

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    E.lib()
    from sparse_long_context_08_b300.workloads import CONFIGS
    kw = overrides(args)
    w = make_workload(args.workload, seed=rank_seed(args.workload, rank), **kw)
    kv, q = upload_workload(w)
    dec = EntmaxKVDecoder(kv, w.num_q_heads, float(w.scale), w.alpha, w.policy,
                          w.budget_tokens, w.delta)
    dec.build_meta()
    torch.cuda.synchronize()
    # L2 flush between timed steps: write a buffer larger than L2, then read
    # another one so that the written lines are evicted (and written back)
    # before the next step rather than during it
    flush = torch.empty(max(1, args.flush_mb) << 20, dtype=torch.uint8, device="cuda")
    flush_read = torch.ones(max(1, args.flush_mb // 2) << 20, dtype=torch.uint8, device="cuda")

    def flush_l2(i):
        flush.fill_(i & 255)
        flush_read.sum(dtype=torch.int32)
    stream = torch.cuda.current_stream()

    # Two CUDA graphs of the step: the plain one (the five kernels back to back)
    # is the one timed for the headline; a copy with event-record nodes at the
    # stage boundaries times score | select | plan | qk | tpv (its total is a
    # little longer).
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(6)]
    for x in evs:
        x.record()             # materialise the events before capture
    torch.cuda.synchronize()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap_stream):
        for _ in range(2):
            dec.step(q)        # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(cap_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap_stream):
        dec.step(q)
    staged = torch.cuda.CUDAGraph()
    with torch.cuda.graph(staged, stream=cap_stream):
        evs[0].record()
        dec.score(q)
        evs[1].record()
        E.entmaxkv_set_stage_events(evs[2:6])
        dec.select_decode(q)            # select | plan (inside select when it builds the union) | qk | tpv
        E.entmaxkv_set_stage_events(None)
    torch.cuda.synchronize()

    for i in range(max(3, args.warmup)):
        graph.replay()
        staged.replay()
        flush_l2(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    K = args.steps
    names = ["score", "select", "plan", "qk", "tpv"]
    stage = {n: [] for n in names}
    sampler = ClockSampler(bus_id_of(local_rank)) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    torch.cuda.synchronize()
    total = timed_replays(graph, K, flush_l2)
    for i in range(min(K, 100)):
        flush_l2(i + 3)                     # keeps the GPU busy while the replay is enqueued
        staged.replay()
        torch.cuda.synchronize()
        t = [evs[j].elapsed_time(evs[j + 1]) for j in range(5)]
        for n_, v in zip(names, t):
            stage[n_].append(v)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms_per_step = max_over_ranks(sum(total), world, "cuda") / K

    # bytes the step reads (metadata + selected pages + small tensors)
    up, vr = E.entmaxkv_decode_counts(dec.workspace, w.batch, w.num_q_heads, w.num_kv_heads,
                                      w.head_dim, w.page_size, w.max_pages, dec.cap)
    esz = 2 if w.dtype == "bf16" else 4
    pages = sum(w.pages_of(b) for b in range(w.batch))
    page_bytes = w.page_size * w.head_dim * esz
    meta_row = 2 * w.head_dim * (esz if w.policy != "gauss" else 4)
    bytes_meta = pages * w.num_kv_heads * meta_row + pages * 4
    bytes_k = int(up.sum()) * page_bytes
    bytes_v = int(vr.sum()) * w.head_dim * esz
    small = 2 * w.batch * w.num_q_heads * w.head_dim * 4
    bytes_step = bytes_meta + bytes_k + bytes_v + small
    mean = {n: statistics.mean(v) for n, v in stage.items()}
    per_kernel_bytes = {"score": bytes_meta, "qk": bytes_k, "tpv": bytes_v}
    dom = max(mean, key=mean.get)
    peak, peak_kind = measured_peak()
    dom_bytes = per_kernel_bytes.get(dom)
    achieved = dom_bytes / (mean[dom] * 1e-3) / 1e9 if dom_bytes else None
    traffic = measured_traffic(dom, {"qk": int(up.sum()), "score": pages}.get(dom, 0)) \
        if dom in ("qk", "score") else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                "peak_kind": f"{peak_kind} copy bandwidth", "traffic": traffic,
                "algorithmic_bytes": dom_bytes}

    # end to end through the public API: pinned host q in, pinned host out back
    e2e = None
    if not args.no_e2e:
        q_host = q.cpu().pin_memory()
        out_host = torch.empty(dec.out.shape, dtype=torch.float32).pin_memory()
        q_dev = torch.empty_like(q)
        for _ in range(3):
            dec.step_host(q_host, out_host, q_dev)
            stream.synchronize()
        torch.cuda.synchronize()
        times = []
        for i in range(K):
            flush_l2(i)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            dec.step_host(q_host, out_host, q_dev)
            stream.synchronize()
            times.append(time.perf_counter() - t0)
        e2e = {"value": whole_job_us_per_step(max_over_ranks(sum(times), world, "cuda") * 1e3 / K,
                                              world), "unit": "us/step",
               "h2d_bytes_per_step": q_host.numel() * 4, "d2h_bytes_per_step": out_host.numel() * 4,
               "timing": "host wall clock per step: step_host (one graph replay: a kernel "
                         "copying q from pinned host memory, the step's kernels, the last "
                         "writing out into pinned host memory) and the sync"}

    cpu = None
    ties = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us, desc, cores, _ = oracle_time_per_step(w, args.cpu_seconds)
        cpu = {"value": us, "unit": "us/step", "cores": cores, "kind": "oracle", "sample": desc,
               "cpu_model": host_cpu_model()}
        import numpy as np
        BH = w.batch * w.num_q_heads
        sample = np.sort(np.random.default_rng(5).choice(BH, size=min(BH, 32), replace=False))
        ties = selection_ties(w, dec.sel.cpu().numpy().reshape(BH, -1),
                              dec.n_sel.cpu().numpy().reshape(BH), sample.tolist())
        if args.cpu_1core:
            import oracle
            nthreads = oracle.get_threads()
            oracle.set_threads(1)
            us1, desc1, _, _ = oracle_time_per_step(w, args.cpu_seconds, steps=2)
            oracle.set_threads(nthreads)
            cpu["one_core"] = {"value": us1, "unit": "us/step", "cores": 1, "sample": desc1}

    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    value_us = whole_job_us_per_step(ms_per_step, world)
    line = {
        "metric": METRIC, "value": value_us, "unit": "us/step", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic", "config": workload_config(w),
        "hbm_gbs": bytes_step / (ms_per_step * 1e-3) / 1e9,
        "hbm_frac_of_measured": bytes_step / (ms_per_step * 1e-3) / 1e9 / peak,
        "hbm_frac_of_8tbs": bytes_step / (ms_per_step * 1e-3) / 1e9 / 8000.0,
        "bytes_per_step": bytes_step,
        "bytes_breakdown": {"metadata_and_page_table": bytes_meta, "k_union_pages": bytes_k,
                            "v_support_rows": bytes_v, "q_and_out": small,
                            "union_pages": int(up.sum()), "v_rows": int(vr.sum())},
        "stage_us": {n: v * 1e3 for n, v in mean.items()},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "selection": ties,
        "gpu_launches": kernels_per_step(w) * K, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_full(args):
    """The variants, timed like the sparse step: full-cache entmax decode (plan
    -> qk -> tpv over the whole cache), softmax over the kept pages (score ->
    select -> plan -> qk -> pv -> merge) and full-cache softmax."""
    import torch
    import torch.distributed as dist

    from sparse_long_context_08_b300 import entmaxkv as E
    from sparse_long_context_08_b300.api import (EntmaxKVFullDecoder, EntmaxKVSoftmaxDecoder,
                                                 upload_workload)
    from sparse_long_context_08_b300.workloads import CONFIGS, make_workload

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    E.lib()
    w = make_workload(args.workload, seed=rank_seed(args.workload, rank), **overrides(args))
    kv, q = upload_workload(w)
    mode = args.mode
    pre = []                                   # stages before the decode call
    if mode == "full":
        dec = EntmaxKVFullDecoder(kv, w.num_q_heads, float(w.scale), w.alpha)
        step = lambda: dec.decode(q)
        dnames, launches = ["plan", "qk", "tpv"], 3
    else:
        dec = EntmaxKVSoftmaxDecoder(kv, w.num_q_heads, float(w.scale), w.policy, w.budget_tokens,
                                     w.delta, w.alpha, full=(mode == "softmax_full"))
        dec.build_meta()
        step = lambda: dec.step(q)
        dnames, launches = ["plan", "qk", "pv"], 4
        if mode == "softmax":
            pre = [("score", lambda: dec.sparse.score(q)), ("select", lambda: dec.sparse.select())]
            launches = 6
    torch.cuda.synchronize()
    flush = torch.empty(max(1, args.flush_mb) << 20, dtype=torch.uint8, device="cuda")
    flush_read = torch.ones(max(1, args.flush_mb // 2) << 20, dtype=torch.uint8, device="cuda")

    def flush_l2(i):
        flush.fill_(i & 255)
        flush_read.sum(dtype=torch.int32)

    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4 + len(pre))]
    for x in evs:
        x.record()
    torch.cuda.synchronize()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap_stream):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(cap_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap_stream):
        step()
    staged = torch.cuda.CUDAGraph()
    with torch.cuda.graph(staged, stream=cap_stream):
        for j, (_, fn) in enumerate(pre):
            evs[j].record()
            fn()
        E.entmaxkv_set_stage_events(evs[len(pre):])
        dec.decode(q)
        E.entmaxkv_set_stage_events(None)
    torch.cuda.synchronize()
    for i in range(max(3, args.warmup)):
        graph.replay()
        staged.replay()
        flush_l2(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    K = args.steps
    names = [n for n, _ in pre] + dnames
    stage = {n: [] for n in names}
    sampler = ClockSampler(bus_id_of(local_rank)) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    torch.cuda.synchronize()
    total = timed_replays(graph, K, flush_l2)
    for i in range(min(K, 50)):
        flush_l2(i + 3)
        staged.replay()
        torch.cuda.synchronize()
        for j, n_ in enumerate(names):
            stage[n_].append(evs[j].elapsed_time(evs[j + 1]))
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms_per_step = max_over_ranks(sum(total), world, "cuda") / K

    up, vr = E.entmaxkv_decode_counts(dec.workspace, w.batch, w.num_q_heads, w.num_kv_heads,
                                      w.head_dim, w.page_size, w.max_pages, dec.cap if mode != "full"
                                      else w.max_pages)
    esz = 2 if w.dtype == "bf16" else 4
    page_bytes = w.page_size * w.head_dim * esz
    bytes_k = int(up.sum()) * page_bytes
    # entmax reads the V rows of its support; softmax the V of every page it attends to
    bytes_v = int(vr.sum()) * w.head_dim * esz if mode == "full" else bytes_k
    small = 2 * w.batch * w.num_q_heads * w.head_dim * 4 + w.batch * w.max_pages * 4
    pages = sum(w.pages_of(b) for b in range(w.batch))
    bytes_meta = pages * w.num_kv_heads * 2 * w.head_dim * esz if mode == "softmax" else 0
    bytes_step = bytes_meta + bytes_k + bytes_v + small
    mean = {n: statistics.mean(v) for n, v in stage.items()}
    dom = max(mean, key=mean.get)
    peak, peak_kind = measured_peak()
    dom_bytes = {"score": bytes_meta or None, "qk": bytes_k,
                 "tpv": bytes_v, "pv": bytes_v}.get(dom)
    achieved = dom_bytes / (mean[dom] * 1e-3) / 1e9 if dom_bytes else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                "peak_kind": f"{peak_kind} copy bandwidth",
                "traffic": measured_traffic(dom, {"qk": int(up.sum()), "pv": int(up.sum()),
                                                  "score": pages}.get(dom, 0))
                if dom in ("qk", "pv", "score") else None,
                "algorithmic_bytes": dom_bytes}

    e2e = None
    if not args.no_e2e:
        q_host = q.cpu().pin_memory()
        out_host = torch.empty(dec.out.shape, dtype=torch.float32).pin_memory()
        q_dev = torch.empty_like(q)
        for _ in range(3):
            dec.step_host(q_host, out_host, q_dev)
            stream.synchronize()
        times = []
        for i in range(min(K, 100)):
            flush_l2(i)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            dec.step_host(q_host, out_host, q_dev)
            stream.synchronize()
            times.append(time.perf_counter() - t0)
        e2e = {"value": whole_job_us_per_step(
                   max_over_ranks(sum(times) / len(times), world, "cuda") * 1e3, world),
               "unit": "us/step",
               "h2d_bytes_per_step": q_host.numel() * 4, "d2h_bytes_per_step": out_host.numel() * 4,
               "timing": "host wall clock per step: step_host (one graph replay of the pinned "
                         "H2D of q, the kernels and the D2H of out) and the sync"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us, desc, cores = oracle_full_time_per_step(w, args.cpu_seconds, mode=mode)
        cpu = {"value": us, "unit": "us/step", "cores": cores, "kind": "oracle", "sample": desc,
               "cpu_model": host_cpu_model()}

    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": MODE_METRIC[mode], "value": whole_job_us_per_step(ms_per_step, world),
        "unit": "us/step",
        "n_gpus": world, "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic", "config": dict(workload_config(w), mode=mode),
        "hbm_gbs": bytes_step / (ms_per_step * 1e-3) / 1e9,
        "hbm_frac_of_measured": bytes_step / (ms_per_step * 1e-3) / 1e9 / peak,
        "bytes_per_step": bytes_step,
        "bytes_breakdown": {"metadata": bytes_meta, "k_pages": bytes_k,
                            ("v_support_rows" if mode == "full" else "v_pages"): bytes_v,
                            "q_out_page_table": small, "pages": int(up.sum()),
                            "v_rows": int(vr.sum()) if mode == "full" else None},
        "stage_us": {n: v * 1e3 for n, v in mean.items()},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches * K, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_meta(args):
    """The page-metadata build of the whole cache (kmin/kmax for the bound
    policies, mean/var for the Gaussian one), timed like the step: a CUDA
    graph of one entmaxkv_build_page_meta call, L2 flushed between calls.
    Bytes: the valid K pages read, the metadata written, the page table."""
    import torch
    import torch.distributed as dist

    from sparse_long_context_08_b300 import entmaxkv as E
    from sparse_long_context_08_b300.api import EntmaxKVDecoder, upload_workload
    from sparse_long_context_08_b300.workloads import make_workload

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    E.lib()
    w = make_workload(args.workload, seed=rank_seed(args.workload, rank), **overrides(args))
    kv, q = upload_workload(w)
    dec = EntmaxKVDecoder(kv, w.num_q_heads, float(w.scale), w.alpha, w.policy,
                          w.budget_tokens, w.delta)
    torch.cuda.synchronize()
    flush = torch.empty(max(1, args.flush_mb) << 20, dtype=torch.uint8, device="cuda")
    flush_read = torch.ones(max(1, args.flush_mb // 2) << 20, dtype=torch.uint8, device="cuda")

    def flush_l2(i):
        flush.fill_(i & 255)
        flush_read.sum(dtype=torch.int32)
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap_stream):
        for _ in range(2):
            dec.build_meta(stream=cap_stream)
    torch.cuda.current_stream().wait_stream(cap_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap_stream):
        dec.build_meta(stream=cap_stream)
    for i in range(max(3, args.warmup)):
        graph.replay()
        flush_l2(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(bus_id_of(local_rank)) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    K = args.steps
    total = timed_replays(graph, K, flush_l2)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(sum(total), world, "cuda") / K
    esz = 2 if w.dtype == "bf16" else 4
    pages = sum(w.pages_of(b) for b in range(w.batch))
    gauss = w.policy == "gauss"
    bytes_k = sum(int(w.seq_lens[b]) for b in range(w.batch)) * w.num_kv_heads * w.head_dim * esz
    bytes_meta = pages * w.num_kv_heads * 2 * w.head_dim * (4 if gauss else esz)
    bytes_all = bytes_k + bytes_meta + pages * 4
    peak, peak_kind = measured_peak()
    gbs = bytes_all / (ms * 1e-3) / 1e9
    if rank == 0:
        line = {"metric": "page-metadata build us and achieved HBM GB/s (frac of peak)",
                "value": whole_job_us_per_step(ms, world), "unit": "us/build", "n_gpus": world,
                "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms,
                "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32" if gauss else w.dtype, "data": "synthetic",
                "config": dict(workload_config(w), mode="meta",
                               statistics="mean/var" if gauss else "kmin/kmax"),
                "hbm_gbs": gbs, "hbm_frac_of_measured": gbs / peak, "hbm_frac_of_8tbs": gbs / 8000.0,
                "bytes_per_step": bytes_all,
                "bytes_breakdown": {"k_read": bytes_k, "metadata_written": bytes_meta,
                                    "page_table": pages * 4},
                "roofline": {"bound": "hbm", "kernel": "build_meta", "achieved": gbs, "peak": peak,
                             "unit": "GB/s", "frac": gbs / peak,
                             "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                             "algorithmic_bytes": bytes_all},
                "cpu_baseline": None, "e2e": None, "gpu_launches": K, "clocks": clocks}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_e2e_breakdown(args):
    """Host wall clock (median of 200, the GPU idle before each call) of the
    pieces of an end-to-end step: a graph of one tiny kernel plus the stream
    sync (the launch and wake-up floor), the device-only step graph plus the
    sync, and the host-buffer step (EntmaxKVDecoder.step_host) plus the sync.
    One JSON line."""
    import torch

    from sparse_long_context_08_b300.api import EntmaxKVDecoder, upload_workload
    from sparse_long_context_08_b300.workloads import make_workload

    w = make_workload(args.workload, **overrides(args))
    kv, q = upload_workload(w)
    dec = EntmaxKVDecoder(kv, w.num_q_heads, float(w.scale), w.alpha, w.policy,
                          w.budget_tokens, w.delta)
    dec.build_meta()
    torch.cuda.synchronize()
    flush = torch.empty(max(1, args.flush_mb) << 20, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    q_host = q.cpu().pin_memory()
    out_host = torch.empty(dec.out.shape, dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(q)
    with torch.cuda.stream(s):
        for _ in range(2):
            dec.step(q)
    s.synchronize()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=s):
        dec.step(q)
    tiny = torch.zeros(1, device="cuda")
    with torch.cuda.stream(s):
        tiny.add_(1)
    g_tiny = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_tiny, stream=s):
        tiny.add_(1)
    for _ in range(3):
        dec.step_host(q_host, out_host, q_dev, s)
        s.synchronize()

    def replay(g):
        def f():
            with torch.cuda.stream(s):
                g.replay()
        return f

    def median_us(fn, n=200):
        ts = []
        for i in range(n):
            flush.fill_(i & 255)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            s.synchronize()
            ts.append((time.perf_counter() - t0) * 1e6)
        return statistics.median(ts)

    rows = {"tiny_graph_and_sync_us": median_us(replay(g_tiny)),
            "device_step_graph_and_sync_us": median_us(replay(g_step)),
            "step_host_and_sync_us": median_us(
                lambda: dec.step_host(q_host, out_host, q_dev, s))}
    print(json.dumps({"e2e_breakdown": rows, "workload": workload_config(w)["workload"],
                      "timing": "host wall clock, median of 200 calls, L2 flushed and the GPU "
                                "idle before each"}), flush=True)


def main():
    args = parse()
    if args.e2e_breakdown:
        run_e2e_breakdown(args)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.mode == "meta":
        run_meta(args)
    elif args.mode != "sparse":
        run_full(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
