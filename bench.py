"""Benchmark of the fused AdamW step with compressed moment state.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload gpt_1p3b] [--modes q8,bf16m,fp32] [--no-cpu-baseline] [--no-extra]

A mode is fp32, bf16m, q8 or q8v, optionally with overrides: "q8/bs256" (block size 256),
"q8/p99" (percentile 99), "q8v/bs4096/p99.9", and "/approx" for the opt-in approximate
square root and quotient in the update (any mode). Overrides away from block 2048 or to a
percentile rank above 4 run the library's general kernel.

One step = one call of the library over the workload's whole tensor list (load, dequantize,
AdamW, requantize, store: a single kernel launch per <=440 tensors). The headline workload
is the GPT-style 1.3B list (292 tensors, 1,315,819,520 params, bf16 grads widened in the
kernel) with 8-bit block-wise moments (block 2048, round to nearest); the JSON line also
reports the same list with bf16, fp32 and fp32-m/8-bit-v moments and the opt-in approximate
update (`modes`), and, under `workloads`, ViT-Base (86.5M params, every moment mode), the
2^30-param tensor with stochastic rounding and 99.9th-percentile scales, the general kernel
on 16.7M params, and the 1M tensor as a latency. Inputs are synthetic and seeded
(workloads.py) and resident in HBM before the timed region; up to 8 distinct grad sets are
cycled. Between timed steps the L2 is flushed, outside the per-step CUDA events: a 384 MB
buffer is written and then read back, so the L2 holds none of the step's inputs and none of
the flush's writes are still waiting to go to HBM when the step starts.

value      = params updated per second over all ranks (Gparams/s), device-timed
e2e        = the same through the public API with host buffers: each step copies its grads
             from pinned host memory and the updated params back, inside the timed span
roofline   = algorithmic HBM bytes per launch / mean launch time vs MEASURED_PEAKS.json
cpu_baseline = the CPU oracle (single thread) on a bounded sample of the workload; its
             all_cores entry: the same oracle on every host core, one sample per thread

Under torchrun (N > 1) every rank runs its own shard of the same size on its own GPU
(weak scaling, no collective in the step); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "Gparams/s per AdamW step and achieved HBM GB/s (% of GB300 peak), per moment mode"
L2_FLUSH_BYTES = 384 << 20
STATE_BYTES = {"fp32": (4, 4), "bf16m": (2, 2), "q8": (1, 1), "q8v": (4, 1)}   # per m, v element


def parse_mode(spec: str):
    """"q8/bs256/p99/sr" -> ("q8", {"block_size": 256, "percentile": 99.0,
    "stochastic_rounding": True}); "approx" asks for the approximate update."""
    base, *opts = spec.split("/")
    if base not in STATE_BYTES:
        raise SystemExit(f"unknown moment mode {base!r}")
    over = {}
    for o in opts:
        if o == "approx":
            over["approx_update"] = True
        elif o.startswith("bs") and base in ("q8", "q8v"):
            over["block_size"] = int(o[2:])
        elif o.startswith("p") and base in ("q8", "q8v"):
            over["percentile"] = float(o[1:])
        elif o == "sr" and base in ("q8", "q8v"):
            over["stochastic_rounding"] = True
        else:
            raise SystemExit(f"bad mode option {o!r} in {spec!r}")
    return base, over


def algorithmic_bytes(mode: str, sizes, grad_dtype: str, zero_grads: bool = False, block_size: int = 2048) -> int:
    """Bytes the step must move once each: p read+write, g read (and written with zeros
    when zero_grads), m and v read+write, and for 8-bit moments the fp32 scales of every
    block read+write."""
    g = 4 if grad_dtype == "f32" else 2
    mb, vb = STATE_BYTES[mode]
    per = 8 + g * (2 if zero_grads else 1) + 2 * mb + 2 * vb
    total = per * sum(sizes)
    scales = {"q8": 2, "q8v": 1}.get(mode, 0)  # fp32 scale arrays, read + written per block
    total += 8 * scales * sum((n + block_size - 1) // block_size for n in sizes)
    return total


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and with whitespace runs collapsed: what the
    compiler sees of it (string and character literals are left alone)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # a literal: copy it to its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(sources: dict | None = None) -> str:
    """Hash of the kernel sources (csrc/) as the compiler sees them: an edit to a comment
    keeps it, so the stored ncu traffic stays attached to the code it measured.
    sources: {file name: text} to hash instead of the files on disk."""
    if sources is None:
        sources = {}
        for f in sorted(glob.glob(os.path.join(ROOT, "precision_state_adam_gb300", "csrc", "*"))):
            if f.endswith((".cu", ".cuh", ".h")):
                with open(f, encoding="utf-8", errors="replace") as fh:
                    sources[os.path.basename(f)] = fh.read()
    h = hashlib.sha256()
    for name in sorted(sources):
        h.update(name.encode() + b"\0" + _code_only(sources[name]).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def ncu_traffic(workload: str, mode: str):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel sources have
    not changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(f"{workload}/{mode}")
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks during the timed region
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        # nvidia-smi's output goes to a pseudo-terminal: into a pipe it is block-buffered and
        # its samples would only arrive when it exits
        import pty
        try:
            master, slave = pty.openpty()
        except OSError:
            master = slave = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=slave if slave is not None else subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, stdin=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            for fd in (master, slave):
                if fd is not None:
                    os.close(fd)
            return
        if slave is not None:
            os.close(slave)
            self.stream = os.fdopen(master, "r", errors="replace")
        else:
            self.stream = io.TextIOWrapper(self.proc.stdout, errors="replace")
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # nvidia-smi takes a moment to start: wait for its first sample (at most 5 s) so the
        # samples span the timed regions that follow
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.02)

    def _read(self):
        try:
            for line in self.stream:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    self.rows.append(parts)
        except OSError:  # the terminal's other end closed (EIO)
            pass

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        try:
            self.stream.close()
        except OSError:
            pass
        rows = [r for r in self.rows if self.uuid is None or self.uuid in r[0]] or self.rows
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ multi-rank aggregation
def max_over_ranks(seconds: float, dist, device) -> float:
    """The slowest rank's time: every rank passes its own, all get the max."""
    if dist is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gparams_per_s(params_per_rank: int, steps: int, seconds: float, world: int) -> float:
    """Whole-job throughput: every rank updates its own shard of `params_per_rank`
    params per step (weak scaling), timed by the slowest rank."""
    return world * params_per_rank * steps / seconds / 1e9


# ------------------------------------------------------------------ our implementation
GRAD_SET_BUDGET = 16 << 30  # bytes of resident grad sets per workload (at least two sets)


def n_grad_sets(w: workloads.Workload, steps: int, warmup: int) -> int:
    """Seeded grad sets kept resident and cycled: 8, fewer when they would exceed the budget
    (the 1.3B list and the 2^30 tensor); every set is far larger than the L2 either way."""
    per_set = sum(w.sizes) * (4 if w.grad_dtype == "f32" else 2)
    return max(2, min(8, steps + warmup, GRAD_SET_BUDGET // max(per_set, 1)))


def flush_l2(flush, t: int) -> None:
    """Evict the L2 (129 MB) between timed steps: write the 384 MB buffer, then read it. The
    read misses evict the written lines (their write-back happens here, not inside the next
    step) and leave only clean lines of the buffer behind."""
    flush.fill_(float(t))
    flush.sum()


def bench_workload(args, w: workloads.Workload, modes, rank: int, world: int, dist, dev, steps: int,
                   warmup: int, with_e2e: bool):
    """Device-timed steps of every mode of `modes` on workload `w`: per-step CUDA events on the
    launching stream, L2 flushed between steps outside the events. Returns {mode: result}."""
    import torch
    import precision_state_adam_gb300 as psa

    sizes = w.sizes
    numel = sum(sizes)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    n_sets = n_grad_sets(w, steps, warmup)
    grads = []
    for s in range(n_sets):
        grads.append(workloads.grads_torch(sizes, s + 1, w.grad_std, dev, seed=workloads.DEFAULT_SEED + 1000 * rank,
                                           kind=w.grad_kind, dtype=w.grad_dtype))
    # with in-step grad zeroing, every step gets its grad set back (outside the step events)
    pristine = [[g.clone() for g in gs] for gs in grads] if args.zero_grads else None
    results = {}
    for spec in modes:
        mode, over = parse_mode(spec)
        bs = over.get("block_size", 2048)
        params = workloads.init_params_torch(w.specs, dev, seed=workloads.DEFAULT_SEED + rank, flat=True)
        state = psa.zeros_state(params, mode, bs)
        kw = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay)
        if mode in ("q8", "q8v"):
            kw.update(stochastic_rounding=w.stochastic_rounding, seed=w.seed, percentile=w.percentile)
        kw.update(over)
        if args.zero_grads:
            kw.update(zero_grads=True)
        launches_per_step = launches_per_call(sizes)
        # one marshalled plan per grad set: a step is then a single C call
        plans = [psa.StepPlan(mode, params, grads[s], state, **kw) for s in range(n_sets)]
        t = 0
        for _ in range(warmup):
            t += 1
            if pristine is not None:
                for d, src in zip(grads[(t - 1) % n_sets], pristine[(t - 1) % n_sets]):
                    d.copy_(src)
            plans[(t - 1) % n_sets].step(t)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        evs = []
        for _ in range(steps):
            t += 1
            if pristine is not None:
                for d, src in zip(grads[(t - 1) % n_sets], pristine[(t - 1) % n_sets]):
                    d.copy_(src)
            flush_l2(flush, t)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plans[(t - 1) % n_sets].step(t)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        step_ms = [a.elapsed_time(b) for a, b in evs]
        total_s = max_over_ranks(sum(step_ms) / 1e3, dist, dev)
        nbytes = algorithmic_bytes(mode, sizes, w.grad_dtype, args.zero_grads, bs)
        mean_s = sum(step_ms) / len(step_ms) / 1e3
        results[spec] = {
            "gparams_per_s": job_gparams_per_s(numel, steps, total_s, world),
            "ms_per_step": total_s * 1e3 / steps,
            "median_ms": statistics.median(step_ms),
            "bytes_per_step": nbytes,
            "achieved_gbs": nbytes / mean_s / 1e9,
            "launches": launches_per_step * steps,
        }
        # ---- end to end through the public API with host buffers (the headline mode only)
        if with_e2e and spec == modes[0]:
            results[spec]["e2e"] = run_e2e(args, psa, torch, dev, stream, w, spec, params, state, kw, t, flush, dist,
                                           world, steps)
            results[spec]["launches"] += from_host_launches(sizes, args.e2e_chunks, bs) * steps
        del plans, params, state
        torch.cuda.empty_cache()
    del grads, pristine, flush
    torch.cuda.empty_cache()
    return results


def mode_line(w: workloads.Workload, spec: str, x: dict, peak: float, zero_grads: bool) -> dict:
    """One mode's figures as the JSON line reports them."""
    out = {"gparams_per_s": round(x["gparams_per_s"], 3), "achieved_gbs": round(x["achieved_gbs"], 1),
           "frac_of_measured_peak": round(x["achieved_gbs"] / peak, 4),
           "bytes_per_param": round(x["bytes_per_step"] / sum(w.sizes), 4),
           "median_ms": round(x["median_ms"], 5)}
    if not zero_grads:  # the captures are of the plain step; grad zeroing runs another kernel flavour
        out["traffic"] = ncu_traffic(w.name, spec)
    return out


def extra_workloads(args, head_workload: str):
    """The other workloads the JSON line carries beside the headline, with their modes:
    ViT-Base (the 86.5M list, every moment mode), the 2^30 tensor with stochastic rounding and
    99.9th-percentile scales, the general kernel on 16.7M params (block 256; percentile 99 =
    rank 21), and the 1M tensor as a latency figure (it fits in the L2)."""
    plan = [("vit_base", ["q8", "bf16m", "fp32", "q8v"]),
            ("flat_1g_heavy", ["q8", "q8v", "q8/approx"]),
            ("flat_16m", ["q8", "q8/bs256", "q8/p99", "q8/p99.9"]),
            ("flat_1m", ["bf16m"])]
    return [(n, m) for n, m in plan if n != head_workload]


def run_ours(args, rank: int, world: int, dist):
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    results = bench_workload(args, w, args.modes, rank, world, dist, dev, args.steps, args.warmup,
                             with_e2e=args.e2e)
    extras = {}
    if args.extra:
        for name, modes in extra_workloads(args, w.name):
            extras[name] = bench_workload(args, workloads.WORKLOADS[name], modes, rank, world, dist, dev, args.steps,
                                          args.warmup, with_e2e=False)
    clk = clocks.stop()
    return results, extras, clk


def launches_per_call(sizes) -> int:
    """Kernel launches of one step call over a list: one per at most 8 tensors for lists of
    up to 8, else one per at most 440 (empty tensors take no slot)."""
    live = [n for n in sizes if n > 0]
    if not live:
        return 0
    return -(-len(live) // (8 if len(live) <= 8 else 440))


MAX_CUT = 4 * (2**31 - 1)  # last element offset at which psadam_step_from_host may cut a tensor


def from_host_launches(sizes, n_chunks: int, block_size: int) -> int:
    """Launches of one psadam_step_from_host call: the library's chunking (whole tensors in
    order; a tensor that does not fit the current chunk cut at a multiple of `unit` elements,
    4 blocks rounded up to a multiple of 16), then launches_per_call for each chunk."""
    live = [n for n in sizes if n > 0]
    if not live:
        return 0
    if n_chunks <= 1:
        return launches_per_call(live)
    unit = 4 * block_size
    while unit % 16:
        unit *= 2
    target = max(unit, -(-(sum(live) // n_chunks) // unit) * unit)
    chunks, cur, size = [], [], 0
    for n in live:
        lo = 0
        while lo < n:
            hi = n if n - lo <= target - size else lo + (target - size) // unit * unit
            if hi < n and hi > MAX_CUT:  # the library cuts no tensor past 4 * INT_MAX elements
                hi = n
            if hi <= lo:
                chunks.append(cur)
                cur, size = [], 0
                continue
            cur.append(hi - lo)
            size += hi - lo
            lo = hi
            if size >= target or lo < n:
                chunks.append(cur)
                cur, size = [], 0
    if cur:
        chunks.append(cur)
    return sum(launches_per_call(c) for c in chunks if c)


def run_e2e(args, psa, torch, dev, stream, w, spec, params, state, kw, t, flush, dist, world, steps):
    """The step through the public API with host buffers: every step copies its grads from
    pinned host memory and the updated params back, inside the timed span. One call per step,
    StepPlan.step_from_host: the library cuts the list into block-aligned chunks whose
    uploads, steps and downloads overlap on three streams (bit for bit the one-call step).
    The host grads follow the workload's own distribution."""
    sizes = w.sizes
    mode, over = parse_mode(spec)
    gdt = torch.float32 if w.grad_dtype == "f32" else torch.bfloat16
    # flat buffers, as a flat-parameter optimizer keeps them: the library then moves each chunk
    # with one copy per direction
    host_g = []
    for s in range(2):
        gs = workloads.grads_torch(sizes, s + 1, w.grad_std, dev, kind=w.grad_kind, dtype=w.grad_dtype)
        _, views = workloads.flat_views(sizes, gdt, pin=True)
        for v, g in zip(views, gs):
            v.copy_(g)
        host_g.append(views)
        del gs
    _, host_p = workloads.flat_views(sizes, torch.float32, pin=True)
    _, dev_g = workloads.flat_views(sizes, gdt, dev)
    h2d = sum(g.numel() * g.element_size() for g in host_g[0])
    d2h = sum(p.numel() * 4 for p in params)
    plan = psa.StepPlan(mode, params, dev_g, state, **kw)
    piped = args.e2e_chunks > 1
    s_in, s_out = (torch.cuda.Stream(dev), torch.cuda.Stream(dev)) if piped else (None, None)

    def one_step(k, tt):
        plan.step_from_host(tt, host_g[k], host_p, n_chunks=args.e2e_chunks, stream=stream, stream_in=s_in,
                            stream_out=s_out)

    link = host_link_rates(torch, dev, host_g[0], dev_g, params, host_p)

    for i in range(3):  # warm the copy engines
        t += 1
        one_step(i % 2, t)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    # the steps are queued back to back with no host wait between them, as a training loop
    # issues them: a host thread that stalls for a moment does not leave the link idle
    evs = []
    for i in range(steps):
        t += 1
        flush_l2(flush, t)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one_step(i % 2, t)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    ms = [a.elapsed_time(b) for a, b in evs]
    total_s = max_over_ranks(sum(ms) / 1e3, dist, dev)
    # the link again after the steps (another tenant's host traffic can change it): the cap
    # takes the faster of the two measurements of each direction
    after = host_link_rates(torch, dev, host_g[0], dev_g, params, host_p)
    best = {k: max(link[k], after[k]) for k in link}
    # the copies alone bound the step: at best the uploads and downloads of a step overlap
    # completely, each at its measured rate and both together at the both-ways rate
    floor_s = max(h2d / (best["h2d_gbs"] * 1e9), d2h / (best["d2h_gbs"] * 1e9),
                  (h2d + d2h) / (best["both_gbs"] * 1e9))
    value = job_gparams_per_s(sum(sizes), steps, total_s, world)
    cap = job_gparams_per_s(sum(sizes), 1, floor_s, world)
    return {"value": round(value, 3), "unit": "Gparams/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_plus_d2h_gbs": round((h2d + d2h) * steps / total_s / 1e9, 1),
            "step_ms": {"min": round(min(ms), 3), "median": round(statistics.median(ms), 3),
                        "max": round(max(ms), 3), "all": [round(x, 2) for x in ms]},
            "host_link": {**link, "after_steps": after, "cap_gparams_per_s": round(cap, 3),
                          "frac_of_cap": round(value / cap, 4),
                          "how": "pinned cudaMemcpyAsync over the same flat buffers, one copy per "
                                 "direction: grads up, params down, and both at once on two streams"},
            "pipeline": f"psadam_step_from_host, {args.e2e_chunks} chunks on 3 streams" if piped else
                        "psadam_step_from_host, one stream"}


def _span(views):
    """The one contiguous range that back-to-back views cover (first start to last end)."""
    base = views[0]
    n = (views[-1].data_ptr() - base.data_ptr()) // base.element_size() + views[-1].numel()
    return base.as_strided((n,), (1,))


def host_link_rates(torch, dev, host_g, dev_g, params, host_p, reps: int = 3) -> dict:
    """GB/s of pinned host<->device copies over the end-to-end leg's own flat buffers, each
    direction as one copy: uploads alone, downloads alone, and both at once (two streams);
    best of `reps`."""
    host_g, dev_g, params, host_p = [_span(host_g)], [_span(dev_g)], [_span(params)], [_span(host_p)]
    up_b = sum(g.numel() * g.element_size() for g in host_g)
    down_b = sum(p.numel() * 4 for p in params)
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
        return best

    def up():
        with torch.cuda.stream(s_up):
            for d, h in zip(dev_g, host_g):
                d.copy_(h, non_blocking=True)

    def down():
        with torch.cuda.stream(s_down):
            for h, p in zip(host_p, params):
                h.copy_(p, non_blocking=True)

    def both():
        up()
        down()

    t_up, t_down, t_both = timed(up), timed(down), timed(both)
    return {"h2d_gbs": round(up_b / t_up / 1e9, 1), "d2h_gbs": round(down_b / t_down / 1e9, 1),
            "both_gbs": round((up_b + down_b) / t_both / 1e9, 1)}


# ------------------------------------------------------------------ the CPU oracle as a baseline
def oracle_sample_rate(w: workloads.Workload, spec: str, budget_s: float, threads: int = 1):
    """Time the CPU oracle (as it is: plain scalar C) on whole 2048-element blocks of the
    workload's first tensor, step after step, for about `budget_s` seconds. With threads > 1
    each thread steps its own copy of the sample (the oracle's C calls release the GIL) and
    the rate is the params all threads updated per second."""
    import numpy as np
    import oracle

    mode, over = parse_mode(spec)
    bs = over.get("block_size", 2048)
    n = min(w.sizes[0], 256 * 2048)

    def sample():
        rng = np.random.default_rng(0)
        p = (rng.standard_normal(n) * 0.02).astype(np.float32)
        if mode == "fp32":
            st = [np.zeros(n, np.float32), np.zeros(n, np.float32)]
        elif mode == "bf16m":
            st = [np.zeros(n, np.uint16), np.zeros(n, np.uint16)]
        elif mode == "q8v":
            st = [np.zeros(n, np.float32), np.zeros(n, np.uint8), np.zeros(oracle.n_blocks(n, bs), np.float32)]
        else:
            nb = oracle.n_blocks(n, bs)
            st = [np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, np.float32), np.zeros(nb, np.float32)]
        g = (rng.standard_normal(n) * w.grad_std).astype(np.float32)
        if w.grad_dtype == "bf16":
            g = (g.view(np.uint32) >> 16).astype(np.uint16)
        return p, g, st

    hp = oracle.HParams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    q8 = oracle.Q8Opts(over.get("stochastic_rounding", w.stochastic_rounding), w.seed,
                       over.get("percentile", w.percentile), block_size=bs)
    samples = [sample() for _ in range(threads)]
    steps = [0] * threads
    start = threading.Barrier(threads)
    t0 = [0.0]

    def worker(i):
        p, g, st = samples[i]
        start.wait()
        if i == 0:
            t0[0] = time.perf_counter()
        t, begin = 0, time.perf_counter()
        while True:
            t += 1
            oracle.step_list(mode, [p], [g], [st], t, hp, q8)
            if time.perf_counter() - begin >= budget_s:
                break
        steps[i] = t

    if threads == 1:
        worker(0)
    else:
        pool = [threading.Thread(target=worker, args=(i,)) for i in range(threads)]
        for th in pool:
            th.start()
        for th in pool:
            th.join()
    el = time.perf_counter() - t0[0]
    done = n * sum(steps)
    who = "one thread" if threads == 1 else f"{threads} threads, each on its own copy"
    return done / el / 1e9, f"{sum(steps)} steps over the first {n:,} params of the workload ({-(-n // bs)} blocks), " \
                            f"{el:.1f} s, {who}"


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def workload_config(w: workloads.Workload, head: str, zero_grads: bool, steps: int, warmup: int) -> dict:
    """The `config` of a JSON line: the workload and how it is timed (the same dict in both arms)."""
    mode, over = parse_mode(head)
    return {"workload": w.name, "description": w.description, "moment_mode": head,
            "params": sum(w.sizes), "tensors": len(w.sizes), "grad_dtype": w.grad_dtype,
            "bytes_per_step": algorithmic_bytes(mode, w.sizes, w.grad_dtype, zero_grads,
                                                over.get("block_size", 2048)),
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MB written, then read back, outside the "
                  "step events)",
            "zero_grads": bool(zero_grads),
            "grads": f"{n_grad_sets(w, steps, warmup)} seeded sets resident in HBM, cycled"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on this machine's host cores."""
    w = workloads.WORKLOADS[args.workload]
    mode = args.modes[0]
    times = []
    vals = []
    for _ in range(args.warmup):
        oracle_sample_rate(w, mode, 0.5)
    sample = ""
    for _ in range(args.steps):
        v, sample = oracle_sample_rate(w, mode, args.ref_step_seconds)
        vals.append(v)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "Gparams/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sum(w.sizes) / (value * 1e9) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, mode, args.zero_grads, args.steps, args.warmup),
        "cpu_baseline": {"value": round(value, 6), "unit": "Gparams/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: {sample}"},
        "e2e": {"value": round(value, 6), "unit": "Gparams/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def default_modes(w: workloads.Workload):
    """The headline mode first, then the other moment modes of the same list and the opt-in
    approximate update."""
    rest = [m for m in ("q8", "bf16m", "fp32", "q8v") if m != w.mode]
    return [w.mode] + rest + ["q8/approx"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gpt_1p3b", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--modes", default=None, help="comma list; the first is the headline (default: workload's)")
    ap.add_argument("--numel", type=int, default=None,
                    help="resize a one-tensor workload (for profiling small cases)")
    ap.add_argument("--zero-grads", action="store_true",
                    help="zero the grads inside the step (adds a grad write per param)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="time the headline workload only (no `workloads` lines)")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false",
                    help="skip the end-to-end leg (host buffers), e.g. for profiling runs")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="end-to-end leg: chunks whose copies overlap the step (1 = one stream, in series)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-seconds-all", type=float, default=6.0, help="oracle on every host core (0: skip)")
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    args = ap.parse_args()
    w = workloads.WORKLOADS[args.workload]
    if args.numel is not None:
        if len(w.specs) != 1:
            raise SystemExit("--numel applies to one-tensor workloads only")
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}@{args.numel}",
                                specs=(workloads.TensorSpec(w.specs[0].name, (args.numel,)),),
                                description=w.description + f" (resized to {args.numel:,} params)")
        workloads.WORKLOADS[w.name] = w
        args.workload = w.name
    args.modes = default_modes(w) if args.modes is None else args.modes.split(",")
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, rank, world)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    results, extras, clk = run_ours(args, rank, world, dist)
    if rank == 0:
        head = args.modes[0]
        r = results[head]
        peak, peak_kind = measured_peaks()
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            v, sample = oracle_sample_rate(w, head, args.cpu_seconds)
            cpu = {"value": round(v, 6), "unit": "Gparams/s", "cores": 1, "kind": "oracle", "sample": sample}
            nt = host_threads()
            if nt > 1 and args.cpu_seconds_all > 0:  # the oracle on every host core, each thread its own sample
                va, sa = oracle_sample_rate(w, head, args.cpu_seconds_all, threads=nt)
                cpu["all_cores"] = {"value": round(va, 6), "unit": "Gparams/s", "cores": nt, "sample": sa}
        modes = {m: mode_line(w, m, x, peak, args.zero_grads) for m, x in results.items()}
        wl = {}
        for name, res in extras.items():
            we = workloads.WORKLOADS[name]
            wl[name] = {"params": sum(we.sizes), "tensors": len(we.sizes), "grad_dtype": we.grad_dtype,
                        "description": we.description,
                        "modes": {m: mode_line(we, m, x, peak, args.zero_grads) for m, x in res.items()}}
            if name == "flat_1m":  # fits in the L2: a launch-latency figure, not a roofline fraction
                wl[name]["latency_us_per_step"] = {m: round(x["median_ms"] * 1e3, 2) for m, x in res.items()}
                wl[name]["note"] = ("21 MB of traffic per step fits in the 129 MB L2; the step is bound by launch "
                                    "latency and ramp-up, so read it as a latency, not as a roofline fraction")
        line = {
            "metric": METRIC, "value": round(r["gparams_per_s"], 3), "unit": "Gparams/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, head, args.zero_grads, args.steps, args.warmup),
            "roofline": {"bound": "hbm", "achieved": round(r["achieved_gbs"], 1), "peak": peak, "unit": "GB/s",
                         "frac": round(r["achieved_gbs"] / peak, 4), "peak_kind": peak_kind,
                         "traffic": modes[head].get("traffic"), "kernel": f"psadam_step_kernel ({head})",
                         "frac_of_8tbs_nominal": round(r["achieved_gbs"] / 8000.0, 4)},
            "modes": modes,
            "workloads": wl,
            "cpu_baseline": cpu,
            "e2e": r.get("e2e"),
            "gpu_launches": sum(x["launches"] for x in results.values()) +
                            sum(x["launches"] for res in extras.values() for x in res.values()),
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
