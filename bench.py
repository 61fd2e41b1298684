"""Benchmark: fork decode attention on one B300 (or N, one independent problem per GPU).

Metric: unique-KV HBM GB/s (the fraction of HBM peak is in ``roofline``) and branch-queries/s.
One step = one fork_attn_decode (plan-driven kernels + merge) over the whole workload, inputs
resident in HBM, L2 flushed between timed steps (a 256 MiB write, then a 256 MiB read that
writes the first one's dirty lines back to HBM before the step starts).  Default workload: the
128K-token shared prefix with rolling tool drops, 64 branches (Hq 64 / Hkv 8).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]

Under torchrun every rank runs its own problem (seed offset by rank) on its GPU; rank 0 prints
one JSON line.  ``--impl reference`` times the fp64 CPU oracle on bounded samples instead.
"""
import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import shared_prefix_paged_attn_b300 as fa  # noqa: E402
from shared_prefix_paged_attn_b300 import workloads as W  # noqa: E402

METRIC = "fork decode attention: unique-KV HBM GB/s (% of peak), branch-queries/sec"
KV_BYTES_PER_SLOT_HEAD = 2 * 128 * 2  # K + V, bf16
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the burst cuBLAS figure, since each kernel is timed per
    launch within a sub-second loop."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["bf16_tflops"]), "measured (burst)"
    return FALLBACK_BF16_TFLOPS, "fallback"


def code_text(src: str) -> str:
    """C/C++/CUDA source with each comment and each run of whitespace turned into one space
    (string and character literals kept), so that a comment or layout edit leaves the hash of
    the code unchanged."""
    import re
    tok = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|\s+', re.S)
    out = tok.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else "\0", src)
    return re.sub("\0+", " ", out).strip()


def kernel_source_hash(read=None):
    """Short hash of the decode's code (planner and kernels, comments and whitespace removed;
    the compaction op is compiled apart): DRAM traffic read from an ncu capture only counts
    for the kernels it was taken on."""
    import hashlib
    csrc = os.path.join(ROOT, "shared_prefix_paged_attn_b300", "csrc")
    read = read or (lambda f: open(os.path.join(csrc, f), encoding="utf-8").read())
    h = hashlib.sha256()
    for f in sorted(x for x in os.listdir(csrc) if not x.startswith("compact")):
        h.update(f.encode() + b"\0" + code_text(read(f)).encode())
    return h.hexdigest()[:12]


def ncu_traffic(workload):
    """Per-launch DRAM bytes (read + write) of each kernel from profiles/ncu_traffic.md, rows
    `| kernel | workload | source hash | bytes |`; only rows whose hash matches these sources."""
    out = {}
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return out
    want = kernel_source_hash()
    for line in open(path):
        f = [x.strip() for x in line.strip().strip("|").split("|")]
        if len(f) >= 4 and f[1] == workload and f[2] == want:
            try:
                out[f[0]] = int(f[3])
            except ValueError:
                pass
    return out


class L2Flush:
    """Evicts the inputs from L2 (126 MB) between timed steps: writes a 256 MiB buffer, then
    reads a second one.  After the write alone, L2 is full of dirty lines whose write-back to
    HBM would fall inside the next timed step (about 126 MB of extra DRAM writes); the read
    evicts them first, and leaves L2 holding clean lines that no step reads."""

    def __init__(self, dev, nbytes=256 << 20):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 4, dtype=torch.int32, device=dev)
        self.acc = torch.zeros((), dtype=torch.int64, device=dev)

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, dtype=torch.int64, out=self.acc)


class ClockSampler:
    """Samples the SM clock and the throttle reasons while a timed region runs.

    One sample is taken synchronously on entry and one on exit (right before and right after
    the region: a short region still yields a record), and a thread samples every `period_s`
    in between.  NVML through ``pynvml`` when it loads, else one-shot ``nvidia-smi`` queries."""

    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index, period_s=0.002):
        self.index, self.period = index, period_s
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._thr = None
        self._h = None
        self.source = None

    def _bits(self):
        import pynvml
        return {
            "hw_slowdown": getattr(pynvml, "nvmlClocksEventReasonHwSlowdown", 0x8),
            "hw_thermal_slowdown": getattr(pynvml, "nvmlClocksEventReasonHwThermalSlowdown", 0x40),
            "sw_thermal_slowdown": getattr(pynvml, "nvmlClocksEventReasonSwThermalSlowdown", 0x20),
            "sw_power_cap": getattr(pynvml, "nvmlClocksEventReasonSwPowerCap", 0x4),
            "hw_power_brake_slowdown": getattr(pynvml, "nvmlClocksEventReasonHwPowerBrakeSlowdown", 0x80),
        }

    def _sample_nvml(self):
        import pynvml
        try:
            self.samples.append(float(pynvml.nvmlDeviceGetClockInfo(self._h, pynvml.NVML_CLOCK_SM)))
            fn = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                pynvml.nvmlDeviceGetCurrentClocksThrottleReasons
            r = fn(self._h)
            for n, bit in self._bits().items():
                if r & bit:
                    self.reasons.add(n)
        except Exception as e:  # keep sampling; record that a query failed
            self.reasons.add(f"query_failed:{type(e).__name__}")

    def _sample_smi(self):
        import subprocess
        q = "clocks.sm,clocks.max.sm," + ",".join("clocks_event_reasons." + n for n in self.NAMES)
        try:
            out = subprocess.run(["nvidia-smi", f"--query-gpu={q}", "-i", str(self.index),
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=20).stdout
        except Exception as e:
            self.reasons.add(f"clock_sampling_unavailable:{type(e).__name__}")
            return
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 2 + len(self.NAMES):
                continue
            try:
                self.samples.append(float(f[0]))
                self.max_mhz = float(f[1])
            except ValueError:
                continue
            for n, v in zip(self.NAMES, f[2:]):
                if v.lower() in ("active", "1", "yes"):
                    self.reasons.add(n)

    def __enter__(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            self._h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.max_mhz = float(pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM))
            self.source = "nvml"
        except Exception as e:
            self.nvml_error = f"{type(e).__name__}: {e}"
            self.source = "nvidia-smi"
        sample = self._sample_nvml if self.source == "nvml" else self._sample_smi
        sample()  # right before the region

        def loop():
            while True:  # sample first, then look at the stop flag
                sample()
                if self._stop.wait(self.period if self.source == "nvml" else 0.05):
                    break

        self._thr = threading.Thread(target=loop, daemon=True)
        self._thr.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._thr.join()
        (self._sample_nvml if self.source == "nvml" else self._sample_smi)()  # right after

    def record(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "reasons": sorted(self.reasons), "source": self.source}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def rank_workload(config, rank, device, values=True, split="none", world=1):
    """Rank r's problem.  split "none": the workload's structure with values drawn from
    seed + 1000 r (independent problems, one per GPU: weak scaling).  split "head",
    "request" or "sequence": rank r's share of the one workload (strong scaling); only the
    split by sequence exchanges data (an all-gather of partials in each step)."""
    if split != "none" and world > 1:
        from shared_prefix_paged_attn_b300 import shard
        w = W.make(config, device=device, values=values)
        cid = config
        if split == "head":
            w = shard.split_by_kv_head(w, rank, world)
        elif split == "request":
            w = shard.split_by_request(w, rank, world)[0]
        else:
            w = shard.split_by_sequence(w, rank, world)
        w.meta["config_id"] = cid
        return w
    w = W.make(config, device=device, values=values and rank == 0)
    if rank:
        w.meta["seed"] += 1000 * rank
        if values:
            W.fill_values(w, device=device)
    return w


def sum_over_ranks(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def max_over_ranks(dist, ms, device):
    """The slowest rank's time per step (every rank gets it)."""
    if dist is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(w, budget_s, max_tasks=None):
    """Times the fp64 oracle on whole branches (all heads) until ~budget_s of CPU work."""
    import oracle
    Hq = w.num_q_heads
    done_q, t_total, branches = 0, 0.0, 0
    order = list(range(w.num_branches))
    for b in order:
        rows = np.arange(int(w.branch_q_off[b]) * Hq, int(w.branch_q_off[b + 1]) * Hq)
        t0 = time.perf_counter()
        oracle.fork_attn(w, rows=rows)
        t_total += time.perf_counter() - t0
        done_q += int(w.branch_q_off[b + 1] - w.branch_q_off[b])
        branches += 1
        if t_total >= budget_s or (max_tasks and branches >= max_tasks):
            break
    return done_q, branches, t_total, oracle.threads_default()


def host_copy(w):
    """Host (pinned) copies of the workload's tensors, for the oracle and the e2e leg."""
    return (w.q.cpu().pin_memory(), w.k_pages.cpu().pin_memory(), w.v_pages.cpu().pin_memory())


def workload_config(w, unique_bytes, touched_pages):
    """The `config` dict of a bench line: the same keys and values in both arms.  Besides the
    unique-KV bytes (the metric's numerator), the touched-page bytes (whole pages holding a
    visible slot) and the per-step bytes of Q, out (bf16), LSE and the plan's records are
    reported apart."""
    hd = w.head_dim
    return {"workload": w.name, "config_id": int(w.meta.get("config_id", 0)),
            "Hq": w.num_q_heads, "Hkv": w.num_kv_heads, "branches": w.num_branches,
            "total_q": w.total_q, "unique_kv_bytes": int(unique_bytes),
            "touched_page_bytes": int(touched_pages) * w.num_kv_heads * w.page_size * hd * 2 * 2,
            "qol_bytes": int(w.total_q * w.num_q_heads * (hd * 2 + hd * 2 + 4)),
            "l2": "flushed between steps (256 MiB write, then 256 MiB read)"}


def run_reference(args):
    """The oracle as it stands, on the host cores: one (query token, query head) row per step
    (about 0.1 s on the long-context workload, so that even a 1000-step run ends within a few
    minutes), the GB/s prorated by the row's share of the call."""
    dist, rank, world, local = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle
    dev = "cuda" if torch.cuda.is_available() else "cpu"  # torch's RNG only draws the inputs
    w = W.make(args.config, device=dev)
    w.meta["config_id"] = args.config
    w.q, w.k_pages, w.v_pages = w.q.cpu(), w.k_pages.cpu(), w.v_pages.cpu()
    uslots, upages = oracle.unique_slots(w)
    unique_bytes = uslots * w.num_kv_heads * KV_BYTES_PER_SLOT_HEAD
    Hq, Hkv = w.num_q_heads, w.num_kv_heads
    times = []
    n_rows = w.total_q * Hq
    for s in range(args.warmup + args.steps):
        row = (s * 7919) % n_rows  # spread over branches and heads
        t0 = time.perf_counter()
        oracle.fork_attn(w, rows=np.array([row], dtype=np.int64))
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = unique_bytes / n_rows / sec / 1e9  # prorated share of one call
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, unique_bytes, upages),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.threads_default(),
                             "kind": "oracle",
                             "sample": "per step one (query token, query head) row of the workload, "
                                       "fp64 copied-context attention; GB/s prorated by 1/(total_q*Hq)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


KERNEL_NAMES = ["row8_kernel", "row_kernel", "tcgen05_kernel", "merge_kernel"]


def kernels_present(st):
    return [st["num_items_row8"] > 0, st["num_items_rows"] > st["num_items_row8"],
            st["num_items_tensor"] > 0, st["merge_rows"] > 0]


def kernel_rooflines(st, w, avg, traffic):
    """Per-kernel roofline entries from the one-by-one timings `avg` (ms, KERNEL_NAMES order)."""
    hbm_peak, peak_kind = peaks()
    tflops_peak, tpeak_kind = tensor_peak()
    part_bytes = st["partial_rows"] * (128 * 4 + 4) * 2  # fp32 partial O + lse, written then read
    slots = {"row8_kernel": st["unique_slots_row8"], "row_kernel": st["unique_slots_row32"]}
    kernels = {}
    for j, n in enumerate(KERNEL_NAMES):
        if not kernels_present(st)[j]:
            continue
        if n == "tcgen05_kernel":
            alg, unit, peak, pk, bound = st["flops_tensor"], "TFLOP/s", tflops_peak, tpeak_kind, "tensor"
            scale = 1e12
        else:
            alg = (slots[n] * w.num_kv_heads * KV_BYTES_PER_SLOT_HEAD if n in slots
                   else part_bytes // 2 + st["merge_rows"] * (128 * 2 + 4))
            unit, peak, pk, bound, scale = "GB/s", hbm_peak, peak_kind, "hbm", 1e9
        ach = alg / (avg[j] * 1e-3) / scale
        kernels[n] = {"bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                      "frac": ach / peak, "ms": avg[j], "peak_kind": pk, "algorithmic": alg,
                      "traffic": traffic.get(n)}
    return kernels


def measure_config(cfg, args, dev, flush, dist, rank, world, steps, keep=False):
    """Plans one workload, runs `steps` timed decodes (L2 flushed before each, CUDA events on
    the launching stream, clocks sampled) and then the same number of one-by-one decodes for
    the per-kernel times.  Returns a dict; with keep=True it also holds the workload and the
    ForkAttention object (for the end-to-end and CPU legs)."""
    split = getattr(args, "split", "none")
    w = rank_workload(cfg, rank, str(dev), split=split, world=world)
    w.meta["config_id"] = cfg
    seq = split == "sequence"
    t0 = time.perf_counter()
    # a split by sequence decodes fp32 partials of every row, gathered and merged each step
    run = fa.ForkAttention(w, out_dtype=fa.FA_F32 if seq else fa.FA_BF16, device=dev)
    plan_s = time.perf_counter() - t0
    st = run.plan.stats()
    unique_bytes = st["unique_visible_slots"] * w.num_kv_heads * KV_BYTES_PER_SLOT_HEAD
    stream = torch.cuda.current_stream(dev)
    q, k, v = w.q, w.k_pages, w.v_pages
    if seq:
        g_out = torch.empty((world,) + tuple(run.out.shape), dtype=torch.float32, device=dev)
        g_lse = torch.empty((world,) + tuple(run.lse.shape), dtype=torch.float32, device=dev)
        final_out = torch.empty(tuple(run.out.shape), dtype=torch.bfloat16, device=dev)
        final_lse = torch.empty(tuple(run.lse.shape), dtype=torch.float32, device=dev)

    def step(events=None):
        if events is None:
            fa.fork_attn_decode(q, k, v, run.plan, run.out, run.lse, stream)
            if seq:  # the split's one exchange: every rank's partials, then the merge
                if dist:
                    dist.all_gather_into_tensor(g_out, run.out)
                    dist.all_gather_into_tensor(g_lse, run.lse)
                else:
                    g_out[0].copy_(run.out)
                    g_lse[0].copy_(run.lse)
                fa.fork_attn_merge_parts(g_out, g_lse, final_out, final_lse, stream)
        else:
            fa.fork_attn_decode_timed(q, k, v, run.plan, run.out, run.lse, events, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    assert fa.fork_attn_check(run.plan, stream) == 0, "device error word set during warm-up"

    # The timed region: `steps` decodes exactly as a caller runs them.
    ev_start = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev_stop = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for i in range(steps):
            flush.zero_()
            ev_start[i].record(stream)
            step()
            ev_stop[i].record(stream)
        torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev_start, ev_stop)]
    assert fa.fork_attn_check(run.plan, stream) == 0, "device error word set in the timed region"
    ms = sum(step_ms) / steps
    ms_max = max_over_ranks(dist, ms, dev)

    # Per-kernel durations: inside the decode the kernels overlap on one stream (the row
    # kernels are programmatic dependent launches beside the tcgen05 kernel), where a CUDA
    # event between two of them would serialise them.  So each kernel is timed alone, with
    # CUDA events on the launching stream, in further steps of the same decode with its
    # kernels one after another (fork_attn_decode_timed), L2 flushed before every step.
    Kk = min(steps, 100)
    aev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(KERNEL_NAMES))] for _ in range(Kk)]
    for i in range(Kk):
        flush.zero_()
        step(aev[i])
    torch.cuda.synchronize(dev)
    assert fa.fork_attn_check(run.plan, stream) == 0, "device error word set in the one-by-one pass"
    avg = [sum(aev[i][2 * j].elapsed_time(aev[i][2 * j + 1]) for i in range(Kk)) / Kk
           for j in range(len(KERNEL_NAMES))]
    kernels = kernel_rooflines(st, w, avg, ncu_traffic(w.name))
    hbm_peak, _ = peaks()
    # whole-job unique KV bytes: every rank's own problem (weak), or the one problem the ranks
    # share (strong: its own count, as a split by sequence may read a mounted page twice)
    if split == "none":
        job_bytes, job_q = unique_bytes * world, w.total_q * world
    else:
        wf = W.make(cfg, values=False)
        job_bytes = fa.plan_for(wf).stats()["unique_visible_slots"] * wf.num_kv_heads * KV_BYTES_PER_SLOT_HEAD
        job_q = wf.total_q
    value = job_bytes / (ms_max * 1e-3) / 1e9
    res = {"cfg": cfg, "w": w if keep else None, "run": run if keep else None, "stats": st,
           "unique_bytes": unique_bytes, "plan_s": plan_s, "ms": ms_max, "step_ms": step_ms,
           "wall": wall, "value": value, "bq_s": job_q / (ms_max * 1e-3),
           "frac": value / world / hbm_peak, "kernels": kernels,
           "kernel_ms": {n: a for n, a, p in zip(KERNEL_NAMES, avg, kernels_present(st)) if p},
           "clocks": clk.record(), "config": workload_config(w, unique_bytes, st["touched_pages"]),
           "plan_bytes": run.plan.sizes()[0], "scratch_bytes": run.plan.sizes()[1], "Kk": Kk,
           "launches_per_step": sum(kernels_present(st))}
    if not keep:
        del run, w, q, k, v
        torch.cuda.empty_cache()
    return res


def measure_scoring(args, dev, flush, steps):
    """Key scoring by 32 representative queries of each of the first 8 branches of the
    long-context rolling-drop workload, then a keep of a quarter of each branch's visible
    entries: pass 1 (the lse of every representative row), pass 2 (the tcgen05
    scoring kernel + head reduce) and the top-k, each timed with CUDA events on the stream."""
    w = W.make(4, device=str(dev))
    ws = W.with_representatives(w, list(range(8)), reps=32, device=str(dev))
    del w
    sc = fa.KeyScorer(ws, device=dev)
    st = sc.plan.stats()
    n_vis = []
    for b in range(ws.num_branches):
        words = ws.vis_bits[ws.vis_word_off[b]:ws.vis_word_off[b + 1]]
        bits = np.unpackbits(words.view(np.uint8), bitorder="little")[:ws.branch_len(b)]
        n_vis.append(int(bits.sum()))
    keep_k = torch.as_tensor(np.array([n // 4 for n in n_vis], np.int32), device=dev)
    stream = torch.cuda.current_stream(dev)
    q, k, v = ws.q, ws.k_pages, ws.v_pages
    for _ in range(args.warmup):
        flush.zero_()
        sc.score(q, k, v, stream)
        sc.topk(keep_k, stream)
    torch.cuda.synchronize(dev)
    assert fa.fork_attn_check(sc.plan, stream) == 0
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            fa.fork_attn_score_lse(q, k, sc.plan, sc.lse, stream)
            ev[i][1].record(stream)
            fa.fork_attn_score(q, k, sc.plan, sc.lse, sc.scores, stream)
            ev[i][2].record(stream)
            sc.topk(keep_k, stream)
            ev[i][3].record(stream)
        torch.cuda.synchronize(dev)
    assert fa.fork_attn_check(sc.plan, stream) == 0
    t = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in ev])  # ms
    ms = t.mean(axis=0)
    step = float(t.sum(axis=1).mean())
    keys = sum(n_vis)
    flops2 = keys * ws.meta["reps"] * ws.num_q_heads * 2 * 128  # QK^T of pass 2 (visible keys)
    tpk, tpk_kind = tensor_peak()
    return {"workload": ws.name, "branches": ws.num_branches, "reps": ws.meta["reps"],
            "Hq": ws.num_q_heads, "Hkv": ws.num_kv_heads, "visible_keys": keys,
            "metric": "keys scored and kept per second (both passes + top-k)",
            "value": keys / (step * 1e-3), "unit": "keys/s", "ms_per_step": step,
            "ms_lse_pass": float(ms[0]), "ms_score_pass": float(ms[1]), "ms_topk": float(ms[2]),
            "score_pass": {"bound": "tensor", "achieved": flops2 / (ms[1] * 1e-3) / 1e12,
                           "unit": "TFLOP/s", "peak": tpk, "peak_kind": tpk_kind,
                           "frac": flops2 / (ms[1] * 1e-3) / 1e12 / tpk, "algorithmic": flops2,
                           "exp_per_s": keys * ws.meta["reps"] * ws.num_q_heads / (ms[1] * 1e-3)},
            "lse_pass_tflops": flops2 / (ms[0] * 1e-3) / 1e12,  # its QK^T, the same contraction as pass 2
            "keep": "a quarter of each branch's visible entries", "steps": steps,
            "clocks": clk.record(),
            # lse pass: the tcgen05 kernel (+ merge); score pass: score + head reduce; top-k
            "gpu_launches": steps * (1 + int(st["merge_rows"] > 0) + 2 + 1)}


def run_ours(args):
    dist, rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    flush = L2Flush(dev)
    K = args.steps
    head = measure_config(args.config, args, dev, flush, dist, rank, world, K, keep=True)
    w, run, st, unique_bytes = head["w"], head["run"], head["stats"], head["unique_bytes"]
    stream = torch.cuda.current_stream(dev)
    q, k, v = w.q, w.k_pages, w.v_pages
    kernels = head["kernels"]
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    roof = dict(kernels[dom])
    roof["kernel"] = dom

    e2e = None
    if not args.no_e2e and rank == 0:
        hq, hk, hv = host_copy(w)
        out_h = torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory()
        lse_h = torch.empty(run.lse.shape, dtype=run.lse.dtype).pin_memory()
        n_e2e = max(3, min(10, K))
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n_e2e):
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            fa.fork_attn_decode(q, k, v, run.plan, run.out, run.lse, stream)
            out_h.copy_(run.out, non_blocking=True)
            lse_h.copy_(run.lse, non_blocking=True)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = t0.elapsed_time(t1) / n_e2e
        e2e = {"value": unique_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2),
               "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size() + lse_h.numel() * 4)}

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        import oracle
        hw = W.Workload(**{f: getattr(w, f) for f in ("name", "num_q_heads", "num_kv_heads", "page_ids", "segs",
                                                       "branch_seg_off", "branch_segs", "branch_q_off",
                                                       "vis_bits", "vis_word_off", "num_pages_pool")},
                        meta=dict(w.meta))
        hw.q, hw.k_pages, hw.v_pages = w.q.cpu(), w.k_pages.cpu(), w.v_pages.cpu()
        nq, nb, secs, cores = oracle_sample(hw, budget_s=args.cpu_budget)
        share = nq / w.total_q
        cpu = {"value": unique_bytes * share / secs / 1e9, "unit": "GB/s", "cores": cores,
               "kind": "oracle", "branch_queries_per_s": nq / secs,
               "sample": f"{nb} of {w.num_branches} branches (all heads), fp64 copied-context "
                         f"attention, {secs:.1f} s; GB/s prorated by the share of query tokens"}
        # the tiny fork workload on one host core, whole (all 4 branches, all heads)
        w1 = W.make(1)
        t0 = time.perf_counter()
        oracle.fork_attn(w1, threads=1)
        s1 = time.perf_counter() - t0
        u1 = oracle.unique_slots(w1)[0] * w1.num_kv_heads * KV_BYTES_PER_SLOT_HEAD
        cpu["single_core"] = {"workload": w1.name, "seconds": s1, "cores": 1,
                              "branch_queries_per_s": w1.total_q / s1,
                              "value": u1 / s1 / 1e9, "unit": "GB/s"}

    # the other workloads, each its own timed region with its own clock record
    per_config = {}
    if not args.no_per_config:
        del q, k, v
        for cfg in sorted(W.CONFIGS):
            try:
                r = head if cfg == args.config else measure_config(cfg, args, dev, flush, dist, rank,
                                                                   world, K)
            except ValueError as e:  # a split this workload does not have (one request)
                per_config[str(cfg)] = {"skipped": str(e)}
                continue
            per_config[str(cfg)] = {
                "workload": r["config"]["workload"], "value": r["value"], "unit": "GB/s",
                "frac_of_hbm_peak": r["frac"], "branch_queries_per_s": r["bq_s"],
                "ms_per_step": r["ms"], "step_ms_median": statistics.median(r["step_ms"]),
                "kernel_ms": r["kernel_ms"], "unique_kv_bytes": r["unique_bytes"],
                "tensor_ctas": r["stats"]["tensor_ctas"], "clocks": r["clocks"],
                "steps": K}

    # the packed DAG prefill (every token a query): tensor-bound, so its figure is the
    # causally visible flops per second against the dense bf16 peak
    prefill = None
    r = None
    if not args.no_prefill:
        try:
            r = measure_config(W.PREFILL, args, dev, flush, dist, rank, world, max(3, min(K, 20)))
        except ValueError as e:  # a split this workload does not have (one request)
            prefill = {"skipped": str(e)}
    if r is not None:
        rs = r["stats"]
        flops = rs["flops_rows"] + rs["flops_tensor"]
        tpk, tpk_kind = tensor_peak()
        job_flops = flops * world if args.split == "none" else sum_over_ranks(dist, flops, dev)
        tfl = job_flops / (r["ms"] * 1e-3) / 1e12
        prefill = {"workload": r["config"]["workload"], "metric": "causal attention TFLOP/s",
                   "value": tfl, "unit": "TFLOP/s", "frac_of_bf16_peak": tfl / world / tpk,
                   "peak": tpk, "peak_kind": tpk_kind, "flops_per_step": flops,
                   "flops_counted": "4 x 128 per (query row, KV head, visible key at or before "
                                    "the query's position): causal pairs only",
                   "ms_per_step": r["ms"], "step_ms_median": statistics.median(r["step_ms"]),
                   "total_q": r["config"]["total_q"], "kernel_ms": r["kernel_ms"],
                   "kernels": r["kernels"], "items_skipped": rs["items_skipped"],
                   "tensor_ctas": rs["tensor_ctas"], "clocks": r["clocks"],
                   "steps": max(3, min(K, 20)), "gpu_launches": max(3, min(K, 20)) * r["launches_per_step"]}

    scoring = None
    if not args.no_scoring and rank == 0 and world == 1:
        scoring = measure_scoring(args, dev, flush, max(3, min(K, 20)))

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": head["ms"], "higher_is_better": True,
            "scaling": "weak" if args.split == "none" else "strong", "split": args.split,
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": head["config"],
            "plan_s": head["plan_s"],
            "plan_bytes": head["plan_bytes"], "scratch_bytes": head["scratch_bytes"],
            "branch_queries_per_s": head["bq_s"],
            "frac_of_hbm_peak": head["frac"],
            "roofline": roof,
            "kernels": kernels,
            "kernel_ms": head["kernel_ms"],
            "per_kernel_timing": f"each kernel alone: CUDA events on the launching stream over "
                                 f"{head['Kk']} steps of the decode with its kernels one after "
                                 f"another; in the timed region they overlap",
            "step_ms_min": min(head["step_ms"]), "step_ms_median": statistics.median(head["step_ms"]),
            "wall_s_timed_region": head["wall"],
            "tensor_ctas": st["tensor_ctas"],
            "gpu_launches": K * head["launches_per_step"],
            "flops_per_step": st["flops_rows"] + st["flops_tensor"],
            "clocks": head["clocks"],
            "e2e": e2e,
            "cpu_baseline": cpu,
            "per_config": per_config,
            "packed_dag_prefill": prefill,
            "key_scoring": scoring,
            "gpu": torch.cuda.get_device_name(dev),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_compact(args):
    """Physical compaction (with and without repositioning, each branch on its own or the
    common prefix once) of the first 8 branches of the workload into fresh pages of a grown
    pool; one JSON line per mode.  Bytes per launch: the moved entries' K and V read and
    written (moved x Hkv x 512 B x 2)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.make(args.config, device=str(dev))
    branches = list(range(min(8, w.num_branches)))
    # destination pages for every listed entry (an upper bound on the kept ones)
    listed = [int(sum(int(w.segs[s][2]) for s in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]))
              for b in branches]
    need = sum((n + 15) // 16 for n in listed)
    pool = w.num_pages_pool
    shape = (pool + need,) + tuple(w.k_pages.shape[1:])
    k = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    v = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    k[:pool], v[:pool] = w.k_pages, w.v_pages
    w.k_pages = w.v_pages = None
    w.num_pages_pool = shape[0]
    fresh = np.arange(pool, pool + need, dtype=np.int32)
    flush = L2Flush(dev)
    hbm_peak, peak_kind = peaks()
    for rep, share in ((False, False), (True, False), (False, True), (True, True)):
        t0 = time.perf_counter()
        plan = fa.fork_attn_compact_create(w, branches, fresh, reposition=rep, share_prefix=share)
        plan_s = time.perf_counter() - t0
        kept, wb = plan.sizes()
        rs, _ = plan.shared()
        entries = rs + int((kept - rs).sum())  # entries moved: the shared run once
        moved = entries * w.num_kv_heads * KV_BYTES_PER_SLOT_HEAD * 2
        work = torch.empty(wb // 4 + 64, dtype=torch.int32, device=dev)
        fa.fork_attn_compact_upload(plan, work)
        for _ in range(args.warmup):
            flush.zero_()
            fa.fork_attn_compact_run(plan, k, v)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            flush.zero_()
            a.record()
            fa.fork_attn_compact_run(plan, k, v)
            b.record()
        torch.cuda.synchronize(dev)
        ms = sorted(a.elapsed_time(b) for a, b in ev)
        med = ms[len(ms) // 2]
        gbs = moved / (med * 1e-3) / 1e9
        print(json.dumps({"metric": "compaction: kept K/V bytes read + written per second", "op": "compact",
                          "reposition": rep, "share_prefix": share, "value": gbs, "unit": "GB/s",
                          "ms_per_launch": med,
                          "ms_min": ms[0], "steps": args.steps, "warmup": args.warmup,
                          "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                          "config": {"workload": w.name, "branches": len(branches), "kept_tokens": int(kept.sum()),
                                     "moved_entries": entries, "shared_kept": rs,
                                     "Hkv": w.num_kv_heads, "bytes_per_launch": moved,
                                     "l2": "flushed between launches (256 MiB write, then 256 MiB read)", "plan_s": plan_s},
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                                       "frac": gbs / hbm_peak, "peak_kind": peak_kind}}), flush=True)
        plan.destroy()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --config (the line's per_config then stays empty)")
    ap.add_argument("--split", choices=["none", "head", "request", "sequence"], default="none",
                    help="with N > 1: every rank its own problem (none, weak scaling) or a share "
                         "of one problem by KV head, by request or by sequence (strong scaling; "
                         "the sequence split all-gathers partials and merges them every step)")
    ap.add_argument("--no-scoring", action="store_true",
                    help="leave out the key-scoring entry of the line")
    ap.add_argument("--no-prefill", action="store_true",
                    help="leave out the packed DAG prefill entry of the line")
    ap.add_argument("--compact", action="store_true",
                    help="time the compaction op (8 branches of --config) instead of the decode")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.compact:
        run_compact(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
