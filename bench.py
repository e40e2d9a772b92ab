#!/usr/bin/env python
"""Benchmark: one decode step of weight-absorbed MLA over a paged latent cache.

A step is the whole hot path on one batch: the split-KV planner
(mla_decode_plan), the main attention kernel and the split merge
(mla_decode), on synthetic inputs already resident in HBM.  The default
workload is the 4K-uniform decode batch (B=64, s_q=1, 128 heads, every
seq_len 4096); ``--workload`` picks another for manual runs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
    python bench.py --stage prolog [--workload W]     # the step before attention, alone
    python bench.py --stage epilog [--workload W]     # the step after it (W_UV, o_proj), alone
    python bench.py --stage layer [--workload W]      # prolog, decode and epilog in one step

Prints one JSON line.  ``value`` is KV-cache TB/s (algorithmic bytes: every
cached row once, 1152 B per key) over all ranks; TFLOPS, microseconds per
step and the roofline fraction ride along.  ``--impl reference`` times the
fp64 CPU oracle on a bounded sample of the same workload instead.

Multi-GPU runs are replicas (the path shards by request with no exchange):
launch with torchrun, one rank per GPU, each rank running the full workload.
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

import workloads as W  # noqa: E402

METRIC = "MLA decode KV-cache TB/s, TFLOPS and % of GB300 roofline; µs per decode step"
LAYER_METRIC = "MLA layer step (prolog, decode, epilog) algorithmic HBM GB/s; µs per layer step"
EPILOG_METRIC = "MLA epilog (W_UV per head, o_proj) algorithmic HBM GB/s; µs per step"
PROLOG_METRIC = "MLA prolog (absorbed q, RoPE, RMSNorm, paged append) algorithmic HBM GB/s; µs per launch"
NOMINAL_HBM_TBS = 8.0
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
MAIN_KERNEL_SRC = os.path.join(ROOT, "mla_decode_attention_02_gb300", "csrc")


def _args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="minimum timed steps (the region is stretched to >= 1.5 s of step time "
                         "so that the clock sampler sees it)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--stage", choices=["decode", "prolog", "epilog", "layer"], default="decode",
                    help="decode: the attention step (default); prolog / epilog: the step before / "
                         "after it alone")
    ap.add_argument("--workload", default="uniform", choices=sorted(W.SEEDS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per_workload lines (mixed, mtp, long, long1m, and uniform and mixed with "
                         "power-of-two maxima) of the decode stage")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps eagerly instead of from one captured CUDA graph")
    ap.add_argument("--cache", choices=["bf16", "fp8"], default="bf16",
                    help="decode stage: the latent cache's format (fp8: e4m3 rows of 656 bytes, "
                         "quantised by the library before the timed region; 656 algorithmic bytes per key)")
    return ap.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


_CUDART = None


def reduce_over_ranks(values, op: str, world: int, device=None) -> list:
    """Fold per-rank numbers over all ranks ("max" or "min"); the identity on one rank.

    The timed region counts at its slowest rank (max); the adaptive step count
    is the smallest any rank chose (min), so every rank runs the same steps.
    NCCL ranks pass their CUDA device; gloo ranks (the CPU tests) pass none.
    """
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.MIN)
    return t.tolist()


def whole_job_tbs(world: int, cache_bytes_per_rank: float, step_ms: float) -> float:
    """Whole-job cache TB/s: every rank runs the full workload (weak scaling)."""
    return world * cache_bytes_per_rank / (step_ms * 1e-3) / 1e12


def _cudart():
    import ctypes
    global _CUDART
    if _CUDART is None:
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                _CUDART = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if _CUDART is None:
            import glob
            import torch
            cands = glob.glob(os.path.join(os.path.dirname(torch.__file__), "..", "nvidia", "*",
                                           "lib", "libcudart.so*"))
            _CUDART = ctypes.CDLL(cands[0])
        _CUDART.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                                 ctypes.c_void_p]
        _CUDART.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_uint]
    return _CUDART


def _record(ev, stream, external: bool) -> None:
    """Record a torch event on `stream`; as an external node when capturing a graph."""
    import ctypes
    rc = _cudart().cudaEventRecordWithFlags(ctypes.c_void_p(ev.cuda_event),
                                             ctypes.c_void_p(stream.cuda_stream),
                                             1 if external else 0)
    if rc != 0:
        raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")


def _event_ms(e0, e1) -> float:
    """cudaEventElapsedTime on torch events that the library recorded through the C ABI.

    torch only reports elapsed time for events it recorded itself, so this asks the
    CUDA runtime that torch already loaded.
    """
    import ctypes
    ms = ctypes.c_float(0.0)
    rc = _cudart().cudaEventElapsedTime(ctypes.byref(ms), ctypes.c_void_p(e0.cuda_event),
                                        ctypes.c_void_p(e1.cuda_event))
    if rc != 0:
        raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
    return ms.value


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _kernel_hash() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(MAIN_KERNEL_SRC)):
        if name.startswith("mla_main") or name.endswith((".h", ".cuh")):
            with open(os.path.join(MAIN_KERNEL_SRC, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(workload: str):
    """DRAM bytes per launch of the main kernel from a committed ncu summary, if it is current."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not rec or rec.get("kernel_hash") != _kernel_hash():
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def _cpu_baseline(w, inp, budget_s: float = 15.0, fp8: bool = False):
    """The oracle as it stands, on this host's cores, over a bounded sample of the workload.

    With fp8, the oracle's fp8 decode (attention of the dequantised rows) over the sampled
    requests' pages, quantised by the oracle's own quantiser outside the timed part.
    """
    import torch
    import oracle
    from oracle import fp8 as OF
    threads = oracle.default_threads()

    def run(reqs):
        rows = [(b, t, h) for b in reqs for t in range(w.s_q) for h in range(W.NUM_HEADS)]
        if not fp8:
            t0 = time.perf_counter()
            oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"], inp["block_table"],
                          inp["seq_lens"], s_q=w.s_q, scale=inp["scale"], rows=rows, threads=threads)
            return time.perf_counter() - t0
        # the sampled requests' pages only, renumbered
        pages = sorted({int(p) for b in reqs
                        for p in inp["block_table"][b, :(w.seq_lens[b] + W.PAGE - 1) // W.PAGE].tolist()})
        remap = {p: i for i, p in enumerate(pages)}
        bt = torch.full_like(inp["block_table"], -1)
        for b in reqs:
            n = (w.seq_lens[b] + W.PAGE - 1) // W.PAGE
            bt[b, :n] = torch.tensor([remap[int(p)] for p in inp["block_table"][b, :n].tolist()],
                                     dtype=torch.int32)
        q8 = OF.quantize_cache(inp["kv_cache"][torch.tensor(pages, dtype=torch.long)])
        t0 = time.perf_counter()
        OF.decode(inp["q_latent"], inp["q_rope"], q8, bt, inp["seq_lens"], s_q=w.s_q, scale=inp["scale"],
                  rows=rows, threads=threads)
        return time.perf_counter() - t0

    order = sorted(range(w.batch), key=lambda b: w.seq_lens[b])
    # calibrate on the shortest request, then grow the sample to the time budget
    t1 = run([order[0]])
    per_key = t1 / max(1, w.seq_lens[order[0]])
    reqs, keys = [], 0
    for b in order:
        if (keys + w.seq_lens[b]) * per_key > budget_s and reqs:
            break
        reqs.append(b)
        keys += w.seq_lens[b]
    dt = run(reqs)
    sample_lens = [w.seq_lens[b] for b in reqs]
    nbytes = W.cache_bytes_fp8(sample_lens) if fp8 else W.cache_bytes(sample_lens)
    return {"value": nbytes / dt / 1e12, "unit": "TB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(reqs)} of {w.batch} requests (all {W.NUM_HEADS} heads, "
                      f"{keys} keys{', fp8 cache' if fp8 else ''}), {dt:.1f} s wall, fp64"}


def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle on the host cores, one bounded sample per step."""
    if rank != 0:
        return 0
    import oracle
    w = W.workload(args.workload)
    inp = W.make_inputs(w)
    threads = oracle.default_threads()
    b = min(range(w.batch), key=lambda i: w.seq_lens[i])
    # rows of one request per step; cap heads so a step stays around a second
    heads = W.NUM_HEADS
    rows_all = [(b, t, h) for t in range(w.s_q) for h in range(heads)]
    t0 = time.perf_counter()
    oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"], inp["block_table"],
                  inp["seq_lens"], s_q=w.s_q, scale=inp["scale"], rows=rows_all[:8],
                  threads=threads)
    per_row = (time.perf_counter() - t0) / 8
    nrows = max(threads, min(len(rows_all), int(1.0 / max(per_row, 1e-9))))
    rows = rows_all[:nrows]
    steps = args.steps if args.steps is not None else 20
    times = []
    for i in range(args.warmup + steps):
        t0 = time.perf_counter()
        oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"], inp["block_table"],
                      inp["seq_lens"], s_q=w.s_q, scale=inp["scale"], rows=rows, threads=threads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    frac = nrows / (w.s_q * W.NUM_HEADS)
    nbytes = W.cache_bytes([w.seq_lens[b]]) * frac
    value = nbytes / dt / 1e12
    sample = (f"request {b} (seq_len {w.seq_lens[b]}), {nrows} of {w.s_q * W.NUM_HEADS} "
              f"(token, head) rows per step, fp64 oracle")
    line = {"metric": METRIC, "value": value, "unit": "TB/s", "impl": "reference",
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w),
            "cpu_baseline": {"value": value, "unit": "TB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def _config(w, fp8: bool = False):
    lens = sorted(set(w.seq_lens))
    desc = (f"{w.batch}x{lens[0]}" if len(lens) == 1 else
            f"{len(w.seq_lens)} rows, seq_len {min(lens)}..{max(lens)}")
    return {"workload": w.name, "batch": w.batch, "s_q": w.s_q, "heads": W.NUM_HEADS,
            "d_latent": W.D_LATENT, "d_rope": W.D_ROPE, "page": W.PAGE, "seq_lens": desc,
            "total_keys": sum(w.seq_lens),
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write); "
                  f"cache {(W.cache_bytes_fp8 if fp8 else W.cache_bytes)(w.seq_lens) / 1e6:.0f} MB"}


PER_WORKLOADS = ("mixed", "mtp", "long", "long1m", "uniform+pow2", "mixed+pow2", "uniform+fp8",
                 "mixed+fp8", "long+fp8")
STEP_KERNELS = 3          # launches per step: planner, main kernel, merge


def _measure(w, dev, world, min_steps: int, min_seconds: float, use_graph: bool, warmup: int,
             sampler_gpu=None, cpu=None, pow2_max: bool = False, fp8: bool = False):
    """Time plan + decode of workload `w` on `dev`; returns a dict of times and the inputs.

    Two timed regions run the same steps, each step after a 256 MiB L2 flush:
    (1) events at step boundaries only (the planner, main kernel and merge
    overlap through programmatic dependent launch, which events between the
    kernels would serialise); (2) events around each kernel, for the per-kernel
    times behind the roofline figure.  Steps are captured in a CUDA graph of K
    steps that is replayed until at least `min_steps` steps and `min_seconds`
    of step time have run, so that the clock sampler sees the region.  With `fp8` the
    cache is first quantised by the library's quantiser (outside the timed region) and
    the steps decode over the fp8 cache.
    """
    import torch
    import torch.distributed as dist
    import mla_decode_attention_02_gb300 as mla

    if cpu is None:
        cpu = W.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    if fp8:
        d["kv8"] = mla.quantize_cache_fp8(d.pop("kv_cache"))
    B, S = w.batch, w.s_q
    mp = d["block_table"].shape[1]
    ws = torch.empty(mla.workspace_size(B, S, mp), dtype=torch.uint8, device=dev)
    out = torch.empty((B, S, W.NUM_HEADS, W.D_LATENT), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, S, W.NUM_HEADS), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(events=None):
        p = mla.plan(d["seq_lens"], s_q=S, max_pages_per_seq=mp, workspace=ws)
        if fp8:
            mla.decode_fp8(p, d["q_latent"], d["q_rope"], d["kv8"], d["block_table"],
                           scale=d["scale"], out=out, lse=lse, events=events, pow2_max=pow2_max)
        else:
            mla.decode(p, d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"],
                       scale=d["scale"], out=out, lse=lse, events=events, pow2_max=pow2_max)
        return p

    for _ in range(max(3, warmup)):
        p = step()
    status = mla.check(p)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} during warm-up")

    # calibrate: per-step time with the flush, to size the timed region
    per = 0.0
    for _ in range(2):  # the first pass still pays one-time costs; keep the second
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(5):
            flush.fill_(1)
            step()
        e1.record()
        torch.cuda.synchronize()
        per = e0.elapsed_time(e1) / 5 / 1e3
    want = max(min_steps, int(min_seconds / max(per, 1e-6)) + 1)
    want = int(reduce_over_ranks([want], "min", world, dev)[0])
    K = min(want, 1000 if use_graph else want)
    reps = -(-want // K)

    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev_s = [mk() for _ in range(K)]
    ev_e = [mk() for _ in range(K)]
    ev_k = [[mk(), mk(), mk()] for _ in range(K)]
    # torch creates each CUDA event on its first record; the timed loop re-records them
    # through the CUDA runtime (and the library, through the C ABI)
    for e in ev_s + ev_e + [x for evs in ev_k for x in evs]:
        e.record(stream)
    torch.cuda.synchronize()

    def timed_steps(external: bool, phases: bool):
        cur = torch.cuda.current_stream()
        for k in range(K):
            flush.fill_(k & 0xFF)
            _record(ev_s[k], cur, external)
            step(events=ev_k[k] if phases else None)
            _record(ev_e[k], cur, external)

    graphs = []
    if use_graph:
        for phases in (False, True):
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                timed_steps(external=True, phases=phases)
            graphs.append(g_)
        torch.cuda.synchronize()

    def run_region(phases: bool):
        """reps x K steps; returns the per-step times (ms) and, with phases, per-kernel times."""
        steps_ms, main_ms, comb_ms, plan_ms = [], [], [], []
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for _ in range(reps):
            if graphs:
                graphs[1 if phases else 0].replay()
            else:
                timed_steps(external=False, phases=phases)
            torch.cuda.synchronize()
            steps_ms += [_event_ms(ev_s[k], ev_e[k]) for k in range(K)]
            if phases:
                main_ms += [_event_ms(ev_k[k][0], ev_k[k][1]) for k in range(K)]
                comb_ms += [_event_ms(ev_k[k][1], ev_k[k][2]) for k in range(K)]
                plan_ms += [_event_ms(ev_s[k], ev_k[k][0]) for k in range(K)]
        if world > 1:
            dist.barrier()
        return steps_ms, main_ms, comb_ms, plan_ms

    sampler = ClockSampler(sampler_gpu) if sampler_gpu is not False else None
    if sampler is not None:
        time.sleep(0.5)
    t_start = time.time()
    steps_ms, _, _, _ = run_region(phases=False)
    t_end = time.time()
    clocks = sampler.summary(t_start, t_end) if sampler else None
    ph_steps, main_l, comb_l, plan_l = run_region(phases=True)
    step_ms = statistics.mean(steps_ms)
    vals = [step_ms, statistics.mean(main_l), statistics.mean(comb_l), statistics.mean(plan_l),
            statistics.mean(ph_steps)]
    step_ms, main_ms, comb_ms, plan_ms, phase_step_ms = reduce_over_ranks(vals, "max", world, dev)
    status = mla.check(p)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after the timed region")
    return {"step_ms": step_ms, "main_ms": main_ms, "comb_ms": comb_ms, "plan_ms": plan_ms,
            "phase_step_ms": phase_step_ms, "steps": K * reps, "clocks": clocks,
            "d": d, "cpu": cpu, "ws": ws, "out": out, "lse": lse, "flush": flush, "mp": mp,
            "region_s": t_end - t_start}


def _roofline(w, main_ms, peaks, peak_src, traffic, fp8: bool = False):
    cache_b = W.cache_bytes_fp8(w.seq_lens) if fp8 else W.cache_bytes(w.seq_lens)
    fl = W.flops(w.seq_lens, w.s_q)
    hbm_peak = peaks["hbm_gbs"]
    main_gbs = cache_b / (main_ms * 1e-3) / 1e9
    main_tflops = fl / (main_ms * 1e-3) / 1e12
    hbm_frac = main_gbs / hbm_peak
    tensor_frac = main_tflops / peaks["bf16_tflops"]
    bound = "hbm" if hbm_frac >= tensor_frac else "tensor"
    return {"kernel": "mla_decode_main", "bound": bound,
            "achieved": main_gbs if bound == "hbm" else main_tflops,
            "peak": hbm_peak if bound == "hbm" else peaks["bf16_tflops"],
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": hbm_frac if bound == "hbm" else tensor_frac,
            "traffic": traffic, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": cache_b, "flops_per_launch": fl,
            "launch_ms": main_ms, "hbm_frac": hbm_frac, "tensor_frac": tensor_frac}


def run_native(args, rank, world, local):
    import torch
    import torch.distributed as dist
    import mla_decode_attention_02_gb300 as mla

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    peaks, peak_src = _peaks()

    w = W.workload(args.workload)
    fp8 = args.cache == "fp8"
    min_steps = args.steps if args.steps is not None else 20
    m = _measure(w, dev, world, min_steps, 1.5, not args.no_graph, args.warmup,
                 sampler_gpu=gpu_id if rank == 0 else False, fp8=fp8)
    step_ms, main_ms = m["step_ms"], m["main_ms"]
    steps = m["steps"]
    m_plan_us, m_comb_us, m_phase_us = m["plan_ms"] * 1e3, m["comb_ms"] * 1e3, m["phase_step_ms"] * 1e3
    m_clocks = m["clocks"]
    d, cpu, out, lse, ws, flush, mp = m["d"], m["cpu"], m["out"], m["lse"], m["ws"], m["flush"], m["mp"]
    S = w.s_q
    stream = torch.cuda.current_stream()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    cache_b = W.cache_bytes_fp8(w.seq_lens) if fp8 else W.cache_bytes(w.seq_lens)
    fl = W.flops(w.seq_lens, S)
    value = whole_job_tbs(world, cache_b, step_ms)

    # end to end through the public API: pinned host inputs -> device, step, result -> host.
    # As a serving loop runs it: step k's inputs are copied in on one stream while step
    # k - 1 computes on a second and step k - 2's results are copied out on a third (two
    # sets of device buffers, ordered by events).  The timed region is the whole K-step
    # loop, every step's copies and its L2 flush (on the compute stream, before the step)
    # included: e2e ms per step = elapsed / K.
    e2e = None
    if not args.no_e2e:
        names = ["q_latent", "q_rope", "block_table", "seq_lens"]
        host = {k: cpu[k].pin_memory() for k in names}
        dbuf = [{k: torch.empty_like(d[k]) for k in names} for _ in range(2)]
        outs = [(out, lse), (torch.empty_like(out), torch.empty_like(lse))]
        o_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        l_host = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
        h2d = sum(host[k].numel() * host[k].element_size() for k in names)
        d2h = o_host[0].numel() * o_host[0].element_size() + l_host[0].numel() * l_host[0].element_size()
        k_e2e = min(steps, 200)
        s_in, s_comp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

        def e2e_loop(K):
            """K pipelined steps; returns the last plan (for the status check)."""
            comp_done = [None] * K
            out_done = [None] * K
            p = None
            for k in range(K):
                b = k & 1
                ev_in = torch.cuda.Event()
                with torch.cuda.stream(s_in):
                    if k >= 2:
                        s_in.wait_event(comp_done[k - 2])    # step k - 2 is done with buffer set b
                    for nm in names:
                        dbuf[b][nm].copy_(host[nm], non_blocking=True)
                    ev_in.record(s_in)
                with torch.cuda.stream(s_comp):
                    s_comp.wait_event(ev_in)
                    if k >= 2:
                        s_comp.wait_event(out_done[k - 2])   # step k - 2's results are copied out
                    flush.fill_(k & 0xFF)
                    p = mla.plan(dbuf[b]["seq_lens"], s_q=S, max_pages_per_seq=mp, workspace=ws)
                    dec = mla.decode_fp8 if fp8 else mla.decode
                    dec(p, dbuf[b]["q_latent"], dbuf[b]["q_rope"], d["kv8"] if fp8 else d["kv_cache"],
                        dbuf[b]["block_table"], scale=d["scale"], out=outs[b][0], lse=outs[b][1])
                    comp_done[k] = torch.cuda.Event()
                    comp_done[k].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[k])
                    o_host[b].copy_(outs[b][0], non_blocking=True)
                    l_host[b].copy_(outs[b][1], non_blocking=True)
                    out_done[k] = torch.cuda.Event()
                    out_done[k].record(s_out)
            return p

        torch.cuda.synchronize()
        e2e_loop(4)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0, t1 = mk(), mk()
        t0.record(s_in)
        s_comp.wait_event(t0)
        s_out.wait_event(t0)
        p = e2e_loop(k_e2e)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_comp)
        t1.record(s_out)
        torch.cuda.synchronize()
        status = mla.check(p)
        if status != 0:
            raise RuntimeError(f"device status {status:#x} in the end-to-end region")
        e2e_ms = t0.elapsed_time(t1) / k_e2e
        e2e_ms = reduce_over_ranks([e2e_ms], "max", world, dev)[0]
        e2e = {"value": whole_job_tbs(world, cache_b, e2e_ms), "unit": "TB/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": k_e2e,
               "note": "per-step inputs (q_latent, q_rope, block_table, seq_lens) copied from "
                       "pinned host memory and o_latent + lse read back each step, on their own "
                       "streams, overlapped with the neighbouring steps' decode (two buffer sets); "
                       "elapsed time of the whole loop, L2 flush before every step included; the "
                       "KV cache is device-resident serving state"}

    roof = _roofline(w, main_ms, peaks, peak_src, None if fp8 else _ncu_traffic(w.name), fp8=fp8)
    t_roof = max(cache_b / (NOMINAL_HBM_TBS * 1e12), fl / (peaks["bf16_tflops"] * 1e12))
    t_roof_meas = max(cache_b / (peaks["hbm_gbs"] * 1e9), fl / (peaks["bf16_tflops"] * 1e12))
    del m, d, out, lse, ws, flush

    # the other workloads of the pages, measured the same way (shorter regions)
    per_workload = {}
    if not args.no_per_workload:
        for name in PER_WORKLOADS:
            # "<workload>+pow2": the same workload with power-of-two running maxima;
            # "<workload>+fp8": the same workload over the fp8 cache
            base, _, mode = name.partition("+")
            if base == w.name and mode == ("fp8" if fp8 else ""):
                continue
            wk = W.workload(base)
            r = _measure(wk, dev, world, 20, 0.3, not args.no_graph, 3, sampler_gpu=False,
                         pow2_max=mode == "pow2", fp8=mode == "fp8")
            rf = _roofline(wk, r["main_ms"], peaks, peak_src, _ncu_traffic(base) if not mode else None,
                           fp8=mode == "fp8")
            kb = W.cache_bytes_fp8(wk.seq_lens) if mode == "fp8" else W.cache_bytes(wk.seq_lens)
            per_workload[name] = {
                "config": _config(wk, mode == "fp8"), "steps": r["steps"], "us_per_step": r["step_ms"] * 1e3,
                "tb_s_step": whole_job_tbs(world, kb, r["step_ms"]),
                "phases_us": {"plan": r["plan_ms"] * 1e3, "main": r["main_ms"] * 1e3,
                              "combine": r["comb_ms"] * 1e3},
                "main_roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                     "hbm_frac", "tensor_frac", "traffic")},
                "step_roofline_frac_measured_peaks":
                    max(kb / (peaks["hbm_gbs"] * 1e9),
                        W.flops(wk.seq_lens, wk.s_q) / (peaks["bf16_tflops"] * 1e12)) / (r["step_ms"] * 1e-3)}
            del r
            torch.cuda.empty_cache()

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_base = _cpu_baseline(w, cpu, fp8=fp8)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
                "steps": steps, "warmup": args.warmup, "ms_per_step": step_ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": {**_config(w, fp8), "cache": args.cache},
                "tflops": world * fl / (step_ms * 1e-3) / 1e12,
                "us_per_step": step_ms * 1e3,
                "phases_us": {"plan": m_plan_us, "main": main_ms * 1e3, "combine": m_comb_us,
                              "step_with_phase_events": m_phase_us},
                "roofline_frac_8tbs": t_roof / (step_ms * 1e-3),
                "roofline_frac_measured_peaks": t_roof_meas / (step_ms * 1e-3),
                "e2e": e2e, "gpu_launches": STEP_KERNELS * steps, "roofline": roof,
                "cpu_baseline": cpu_base, "clocks": m_clocks, "per_workload": per_workload,
                "device": torch.cuda.get_device_name(dev), "units": mla.num_units(),
                "launch": "eager" if args.no_graph else "cuda_graph"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_prolog(args, rank, world, local):
    """--stage prolog: the prolog launch alone (absorbed q, RoPE, RMSNorm, cache append).

    The workload's new tokens (batch x s_q) with a pool holding just their pages;
    L2 is flushed (256 MiB written) before every timed launch, and each launch
    is bracketed by CUDA events on its stream.  value = algorithmic bytes per
    launch (every input read once, every output written once) / launch time.
    """
    import torch
    import mla_decode_attention_02_gb300 as mla

    if world > 1:
        raise SystemExit("--stage prolog runs on one GPU")
    w = W.workload(args.workload)
    B, S = w.batch, w.s_q
    if args.impl == "reference":
        from oracle import prolog as OP
        t = W.prolog_tensors(B, S, w.seed)
        c = W.sparse_cache(w.seq_lens, S, w.seed)
        times = []
        for _ in range(max(1, args.steps or 3)):
            t0 = time.perf_counter()
            OP.prolog(t["q_nope"], t["q_pe"], t["kv_latent"], t["k_pe"], t["w_uk"],
                      t["kv_norm_weight"], c["kv_cache"], c["block_table"], c["seq_lens"])
            times.append(time.perf_counter() - t0)
        sec = statistics.median(times)
        nbytes = W.prolog_bytes(B, S)
        print(json.dumps({"metric": PROLOG_METRIC, "stage": "prolog", "impl": "reference",
                          "value": nbytes / sec / 1e9, "unit": "GB/s", "us_per_launch": sec * 1e6,
                          "higher_is_better": True, "n_gpus": 1, "dtype": "f64",
                          "config": {"workload": w.name, "tokens": B * S}}), flush=True)
        return 0

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    t = {k: v.to(dev) for k, v in W.prolog_tensors(B, S, w.seed).items()}
    c_cpu = W.sparse_cache(w.seq_lens, S, w.seed)
    c = {k: v.to(dev) for k, v in c_cpu.items()}
    q_lat = torch.empty((B, S, W.NUM_HEADS, W.D_LATENT), dtype=torch.bfloat16, device=dev)
    q_rope = torch.empty((B, S, W.NUM_HEADS, W.D_ROPE), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    table = mla.rope_table(W.ROPE_BASE, dev)
    stream = torch.cuda.current_stream()

    def launch():
        mla.prolog(t["q_nope"], t["q_pe"], t["kv_latent"], t["k_pe"], t["w_uk"], t["kv_norm_weight"],
                   c["kv_cache"], c["block_table"], c["seq_lens"], table=table, q_latent=q_lat,
                   q_rope=q_rope, status=status)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        launch()
    torch.cuda.synchronize()
    steps = args.steps or 500
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(steps)]
    for e0, e1 in ev:
        e0.record(stream)
        e1.record(stream)
    torch.cuda.synchronize()

    def timed(external: bool):
        cur = torch.cuda.current_stream()
        for k in range(steps):
            flush.fill_(k & 0xFF)
            _record(ev[k][0], cur, external)
            launch()
            _record(ev[k][1], cur, external)

    # the K launches are one CUDA graph, so the GPU never waits for the host between them
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            timed(external=True)
        torch.cuda.synchronize()
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    time.sleep(0.5)
    t_start = time.time()
    if graph is not None:
        graph.replay()
    else:
        timed(external=False)
    torch.cuda.synchronize()
    t_end = time.time()
    clocks = sampler.summary(t_start, t_end)
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st:#x} in the prolog")
    us = [_event_ms(e0, e1) * 1e3 for e0, e1 in ev]
    us_mean = statistics.mean(us)
    nbytes = W.prolog_bytes(B, S)
    fl = W.prolog_flops(B, S)
    peaks, peak_src = _peaks()
    gbs = nbytes / (us_mean * 1e-6) / 1e9
    line = {"metric": PROLOG_METRIC, "stage": "prolog", "value": gbs, "unit": "GB/s",
            "us_per_launch": us_mean, "us_median": statistics.median(us), "us_min": min(us),
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "batch": B, "s_q": S, "tokens": B * S,
                       "l2": "flushed (256 MiB written) before every launch"},
            "tflops": fl / (us_mean * 1e-6) / 1e12,
            "roofline": {"kernel": "mla_prolog", "bound": "hbm", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "traffic": None, "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": nbytes, "flops_per_launch": fl},
            "gpu_launches": steps, "clocks": clocks, "launch": "eager" if args.no_graph else "cuda_graph",
            "device": torch.cuda.get_device_name(dev)}
    print(json.dumps(line), flush=True)
    return 0


def run_epilog(args, rank, world, local):
    """--stage epilog: the W_UV step and o_proj (two hand-written tcgen05 kernels).

    The workload's tokens (batch x s_q); L2 flushed (256 MiB written) before every
    step; events around each of the two launches, all K steps in one CUDA graph.
    value = algorithmic bytes of both / step time; the roofline is the W_UV kernel's.
    """
    import torch
    import mla_decode_attention_02_gb300 as mla

    if world > 1:
        raise SystemExit("--stage epilog runs on one GPU")
    w = W.workload(args.workload)
    B, S = w.batch, w.s_q
    T = B * S
    uv_b, op_b = W.epilog_bytes(T)
    if args.impl == "reference":
        from oracle import epilog as OE
        e = W.epilog_tensors(T, w.seed)
        times = []
        for _ in range(max(1, args.steps or 2)):
            t0 = time.perf_counter()
            OE.o_project(OE.uv_project(e["o_latent"], e["w_uv"]), e["w_o"])
            times.append(time.perf_counter() - t0)
        sec = statistics.median(times)
        print(json.dumps({"metric": EPILOG_METRIC, "stage": "epilog", "impl": "reference",
                          "value": (uv_b + op_b) / sec / 1e9, "unit": "GB/s", "us_per_step": sec * 1e6,
                          "higher_is_better": True, "n_gpus": 1, "dtype": "f64",
                          "config": {"workload": w.name, "tokens": T}}), flush=True)
        return 0

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    e = {k: v.to(dev) for k, v in W.epilog_tensors(T, w.seed).items()}
    o_lat = e["o_latent"].view(B, S, W.NUM_HEADS, W.D_LATENT)
    o_v = torch.empty((B, S, W.NUM_HEADS, W.D_V), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, W.HIDDEN), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        mla.epilog_uv(o_lat, e["w_uv"], o_v=o_v, status=status)
        mla.epilog_oproj(o_v, e["w_o"], out=out, status=status)
    torch.cuda.synchronize()
    steps = args.steps or 200
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk(), mk()) for _ in range(steps)]
    for trio in ev:
        for x in trio:
            x.record()
    torch.cuda.synchronize()

    def timed(external: bool):
        cur = torch.cuda.current_stream()
        for k in range(steps):
            flush.fill_(k & 0xFF)
            _record(ev[k][0], cur, external)
            mla.epilog_uv(o_lat, e["w_uv"], o_v=o_v, status=status)
            _record(ev[k][1], cur, external)
            mla.epilog_oproj(o_v, e["w_o"], out=out, status=status)
            _record(ev[k][2], cur, external)

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            timed(external=True)
        torch.cuda.synchronize()
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    time.sleep(0.5)
    t_start = time.time()
    if graph is not None:
        graph.replay()
    else:
        timed(external=False)
    torch.cuda.synchronize()
    t_end = time.time()
    clocks = sampler.summary(t_start, t_end)
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st:#x} in the epilog")
    uv_us = statistics.mean(_event_ms(a, b) * 1e3 for a, b, _ in ev)
    op_us = statistics.mean(_event_ms(b, c) * 1e3 for _, b, c in ev)
    step_us = uv_us + op_us
    peaks, peak_src = _peaks()
    uv_gbs = uv_b / (uv_us * 1e-6) / 1e9
    op_gbs = op_b / (op_us * 1e-6) / 1e9
    line = {"metric": EPILOG_METRIC, "stage": "epilog",
            "value": (uv_b + op_b) / (step_us * 1e-6) / 1e9, "unit": "GB/s", "us_per_step": step_us,
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "batch": B, "s_q": S, "tokens": T, "hidden": W.HIDDEN,
                       "l2": "flushed (256 MiB written) before every step"},
            "phases_us": {"uv": uv_us, "oproj": op_us},
            "oproj": {"kernel": "mla_epilog_oproj", "achieved_gbs": op_gbs, "frac": op_gbs / peaks["hbm_gbs"],
                      "algorithmic_bytes": op_b},
            "roofline": {"kernel": "mla_epilog_uv", "bound": "hbm", "achieved": uv_gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": uv_gbs / peaks["hbm_gbs"],
                         "traffic": None, "peak_source": peak_src, "algorithmic_bytes_per_launch": uv_b},
            "gpu_launches": steps, "clocks": clocks, "launch": "eager" if args.no_graph else "cuda_graph",
            "device": torch.cuda.get_device_name(dev)}
    print(json.dumps(line), flush=True)
    return 0


def _layer_reference(w):
    """The layer on the oracle: prolog and epilog whole, decode over a bounded sample of requests
    (~15 s, as the decode reference arm), its time scaled to the whole batch by cache bytes."""
    from oracle import epilog as OE
    from oracle import prolog as OP
    B, S = w.batch, w.s_q
    T = B * S
    inp = W.make_inputs(w)
    t = W.prolog_tensors(B, S, w.seed)
    e = W.epilog_tensors(T, w.seed)
    c = W.sparse_cache(w.seq_lens, S, w.seed)
    t0 = time.perf_counter()
    OP.prolog(t["q_nope"], t["q_pe"], t["kv_latent"], t["k_pe"], t["w_uk"], t["kv_norm_weight"],
              c["kv_cache"], c["block_table"], c["seq_lens"])
    t_prolog = time.perf_counter() - t0
    base = _cpu_baseline(w, inp)
    t_decode = W.cache_bytes(w.seq_lens) / (base["value"] * 1e12)
    t0 = time.perf_counter()
    OE.o_project(OE.uv_project(e["o_latent"], e["w_uv"]), e["w_o"])
    t_epilog = time.perf_counter() - t0
    uv_b, op_b = W.epilog_bytes(T)
    nbytes = W.prolog_bytes(B, S) + W.cache_bytes(w.seq_lens) + uv_b + op_b
    sec = t_prolog + t_decode + t_epilog
    print(json.dumps({"metric": LAYER_METRIC, "stage": "layer", "impl": "reference",
                      "value": nbytes / sec / 1e9, "unit": "GB/s", "us_per_step": sec * 1e6,
                      "higher_is_better": True, "n_gpus": 1, "dtype": "f64",
                      "config": {"workload": w.name, "tokens": T},
                      "phases_s": {"prolog": t_prolog, "decode_extrapolated": t_decode,
                                   "epilog": t_epilog},
                      "cpu_baseline": dict(base, value=nbytes / sec / 1e9, unit="GB/s")}), flush=True)
    return 0


def run_layer(args, rank, world, local):
    """--stage layer: the whole absorbed MLA layer of one decode step, on one stream.

    prolog (absorbed q, RoPE, cache append) -> plan -> main -> combine -> W_UV -> o_proj,
    each launch a programmatic dependent of the one before where the library allows it;
    L2 flushed before every step; K steps in one CUDA graph, events at the step
    boundaries.  value = algorithmic bytes of all stages / step time.
    """
    import torch
    import mla_decode_attention_02_gb300 as mla

    if world > 1:
        raise SystemExit("--stage layer runs on one GPU")
    w = W.workload(args.workload)
    B, S = w.batch, w.s_q
    T = B * S
    if args.impl == "reference":
        return _layer_reference(w)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in W.make_inputs(w).items()}
    t = {k: v.to(dev) for k, v in W.prolog_tensors(B, S, w.seed).items()}
    e = {k: v.to(dev) for k, v in W.epilog_tensors(1, w.seed).items() if k != "o_latent"}
    mp = d["block_table"].shape[1]
    table = mla.rope_table(W.ROPE_BASE, dev)
    q_lat = torch.empty((B, S, W.NUM_HEADS, W.D_LATENT), dtype=torch.bfloat16, device=dev)
    q_rope = torch.empty((B, S, W.NUM_HEADS, W.D_ROPE), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mla.workspace_size(B, S, mp), dtype=torch.uint8, device=dev)
    o = torch.empty((B, S, W.NUM_HEADS, W.D_LATENT), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, S, W.NUM_HEADS), dtype=torch.float32, device=dev)
    o_v = torch.empty((B, S, W.NUM_HEADS, W.D_V), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, W.HIDDEN), dtype=torch.bfloat16, device=dev)
    st_p = torch.zeros(1, dtype=torch.int32, device=dev)
    st_e = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        mla.prolog(t["q_nope"], t["q_pe"], t["kv_latent"], t["k_pe"], t["w_uk"], t["kv_norm_weight"],
                   d["kv_cache"], d["block_table"], d["seq_lens"], table=table, q_latent=q_lat,
                   q_rope=q_rope, status=st_p)
        p = mla.plan(d["seq_lens"], s_q=S, max_pages_per_seq=mp, workspace=ws)
        mla.decode(p, q_lat, q_rope, d["kv_cache"], d["block_table"], scale=d["scale"], out=o, lse=lse)
        mla.epilog_uv(o, e["w_uv"], o_v=o_v, status=st_e)
        mla.epilog_oproj(o_v, e["w_o"], out=out, status=st_e)
        return p

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        p = step()
    torch.cuda.synchronize()
    steps = args.steps or 100
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(steps)]
    for a_, b_ in ev:
        a_.record()
        b_.record()
    torch.cuda.synchronize()

    def timed(external: bool):
        cur = torch.cuda.current_stream()
        for k in range(steps):
            flush.fill_(k & 0xFF)
            _record(ev[k][0], cur, external)
            step()
            _record(ev[k][1], cur, external)

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            timed(external=True)
        torch.cuda.synchronize()
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    time.sleep(0.5)
    t_start = time.time()
    if graph is not None:
        graph.replay()
    else:
        timed(external=False)
    torch.cuda.synchronize()
    t_end = time.time()
    clocks = sampler.summary(t_start, t_end)
    for name, stv in (("prolog", int(st_p.item())), ("decode", mla.check(p)), ("epilog", int(st_e.item()))):
        if stv != 0:
            raise RuntimeError(f"device status {stv:#x} in the {name}")
    us = statistics.mean(_event_ms(a_, b_) * 1e3 for a_, b_ in ev)
    uv_b, op_b = W.epilog_bytes(T)
    nbytes = W.prolog_bytes(B, S) + W.cache_bytes(w.seq_lens) + uv_b + op_b
    print(json.dumps({"metric": LAYER_METRIC, "stage": "layer", "value": nbytes / (us * 1e-6) / 1e9,
                      "unit": "GB/s", "us_per_step": us, "n_gpus": 1, "steps": steps,
                      "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
                      "data": "synthetic",
                      "config": {"workload": w.name, "batch": B, "s_q": S, "tokens": T,
                                 "l2": "flushed (256 MiB written) before every step"},
                      "algorithmic_bytes_per_step": nbytes,
                      "gpu_launches": 6 * steps, "clocks": clocks,
                      "launch": "eager" if args.no_graph else "cuda_graph",
                      "device": torch.cuda.get_device_name(dev)}), flush=True)
    return 0


def main():
    args = _args()
    rank, world, local = _dist()
    if world != args.gpus and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.stage == "prolog":
        return run_prolog(args, rank, world, local)
    if args.stage == "epilog":
        return run_epilog(args, rank, world, local)
    if args.stage == "layer":
        return run_layer(args, rank, world, local)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_native(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
