#!/usr/bin/env python3
"""Benchmark of the paged heterogeneous-rank LoRA delta on GB300.

One step = one pass of the hot path over one batch: the token plan, the decode delta for
the batch's decode tokens and the tensor-core segment delta for its prefill segments,
for every projection of the workload.  Metric: LoRA-delta tokens/s per layer
(tokens x layers / step time), plus the dominant kernel's roofline fraction.

  python bench.py [--workload NAME] [--steps K] [--warmup W] [--gpus N]
  python bench.py --impl reference ...      # the fp64 CPU oracle on the host cores

The default workload is the 13B decode batch over a zoo of 2000 pooled adapters (ranks 8
to 64, 512 tokens, Zipf 0.5); the line also carries the 7B prefill batch, one layer of
the mixed prefill + decode iteration, and the headline batch through 8 layers (one call
per layer against the batch planned once for the step) as extra keys.

For N > 1 every rank serves its own batch (seed + rank): the delta has no cross-token
exchange, so ranks are independent replicas (weak scaling) and the only collectives are
the timing barrier and the max-over-ranks reduction.  Under torchrun the ranks come from
the environment; without it, ``--gpus N`` starts the N rank processes itself.

Timing: W untimed warm-up steps; K timed steps, each preceded by an L2 flush that evicts
the pool and inputs from L2: a buffer of twice the L2 is written, then another of that
size read, so that the L2 holds only clean lines of the second buffer (after a write alone
the L2 is full of dirty lines whose write-back would fall inside the timed step); the
flush is outside the per-step CUDA-event intervals; barrier + synchronize on both sides of
the timed region; max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rank_delta_paged_gb300 import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "decode_13b_zoo"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0 = about 2 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--prefetch", type=int, default=0, metavar="K",
                    help="also measure K later batches' adapter loads against the deltas (\"prefetch\")")
    ap.add_argument("--load-mode", choices=["zero_copy", "copy_engine"], default="zero_copy",
                    help="the pool's adapter load path for the end-to-end and load measurements")
    ap.add_argument("--bmm", action="store_true",
                    help="also time the padded batched-GEMM comparison path (decode-only workloads)")
    ap.add_argument("--pressure", type=int, default=0, metavar="K",
                    help="also run K batches of the zoo through acquire / apply / release (\"pressure\")")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers of the step (0 = the workload's own: 32 for mixed_iteration, 1 for decode_13b_zoo, "
                         "decode_7b and prefill_7b, whose layers are one projection each)")
    ap.add_argument("--pool-gib", type=float, default=0.0, help="mixed_iteration: pool size in GiB (0 = 40)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the extra prefill_7b and mixed-layer keys of the default line")
    ap.add_argument("--profile-calls", type=int, default=0, metavar="N",
                    help="for a profiler: N apply calls of the first layer, each after an L2 flush, "
                         "and nothing else (no timing, no line)")
    ap.add_argument("--dry-run", action="store_true",
                    help="start the ranks and print the line's skeleton without touching a GPU "
                         "(gloo; tests the launcher)")
    ap.add_argument("--apply", choices=["multi", "single"], default="multi",
                    help="multi: one slora_lora_apply_multi call per layer (all its projections); "
                         "single: one slora_lora_apply call per projection")
    return ap.parse_args()


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a workload's
# dominant kernel, each from one ncu capture (command below) of that kernel's sources as
# identified by ``sources_sha``.  When the sources have changed since the capture the line
# reports null: the counters describe a kernel that no longer exists.
TRAFFIC_CAPTURE = ("ncu --clock-control none --metrics dram__bytes_read.sum,dram__bytes_write.sum "
                   "-k regex:{kernel} -s 3 -c 1 python bench.py --workload {workload} --profile-calls 5")
TRAFFIC = {
    # workload name: (kernel, DRAM bytes per launch, sources_sha at capture)
    "decode_13b_h5120_a2000_t512_zipf0.5": ("delta_kernel", 264910080 + 3497728, "ea1fbf78de3ce652"),
    "decode_7b_h4096_a100_t256_zipf1": ("delta_kernel", 42062592 + 4608, "ea1fbf78de3ce652"),
}
KERNEL_SOURCES = {
    "delta_kernel": ("decode.cu", "ptx.h", "internal.h"),
    "prefill_kernel": ("prefill.cu", "ptx.h", "tcgen05.h", "internal.h"),
}


def code_of(text: str) -> str:
    """C++ / CUDA source without its comments, trailing blanks and empty lines (string
    literals in these files hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def sources_sha(kernel: str) -> str:
    """sha256 (first 16 hex digits) over the code of the kernel's source files: comments and
    blank lines do not count, so a capture stays valid across comment edits."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "rank_delta_paged_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_of(name: str):
    """(bytes or None, note) for a workload's dominant kernel."""
    if name not in TRAFFIC:
        return None, "no ncu capture for this workload"
    kernel, nbytes, sha = TRAFFIC[name]
    if sources_sha(kernel) != sha:
        return None, f"{kernel} sources changed since the ncu capture ({sha})"
    return nbytes, f"one ncu capture of {kernel} (sources {sha})"


def fp16_peak_tflops(dev) -> float:
    """Dense fp16 tensor throughput measured here: torch.matmul of 8192^3 fp16 matrices
    (2 N^3 flops), best of 10 CUDA-event-timed products after warm-up."""
    import torch
    n = 8192
    a = torch.randn(n, n, device=dev, dtype=torch.float16)
    b = torch.randn(n, n, device=dev, dtype=torch.float16)
    c = torch.empty(n, n, device=dev, dtype=torch.float16)
    for _ in range(3):
        torch.matmul(a, b, out=c)
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b, out=c)
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del a, b, c
    return 2.0 * n ** 3 / (best / 1e3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        return float(mp["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(w: W.Workload) -> float:
    """Per step: every used adapter's A^T and B rows once, x and y0 read, y written,
    for every projection (2 bytes per fp16 element)."""
    used = w.used_adapters()
    adapter = sum(4.0 * int(w.ranks[a]) * w.hidden for a in used)
    xy = 6.0 * w.hidden * w.T
    return w.n_proj * (adapter + xy)


def algorithmic_flops(w: W.Workload) -> float:
    idx = w.token_adapter_idx
    r = np.where(idx >= 0, w.ranks[np.maximum(idx, 0)], 0).astype(np.float64)
    return w.n_proj * 4.0 * w.hidden * float(r.sum())


# ---------------------------------------------------------------- clocks sampling
class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (ctypes; reading only), polled
    from a background thread every 0.5 ms, so that even a timed region of a few
    milliseconds is sampled while it runs."""
    # nvmlClocksEventReason bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    def __init__(self, uuid: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        # the NVML device whose UUID matches the CUDA device's (NVML may list GPUs that
        # CUDA does not see)
        norm = lambda t: t.lower().replace("gpu-", "").replace("-", "")
        want = norm(uuid)
        n = ctypes.c_uint()
        self.lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
        self.h = None
        for i in range(n.value):
            h = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h)) != 0:
                continue
            buf = ctypes.create_string_buffer(96)
            if self.lib.nvmlDeviceGetUUID(h, buf, 96) == 0 and want and norm(buf.value.decode()) == want:
                self.h = h
                break
        if self.h is None:
            raise RuntimeError("no NVML device with UUID " + uuid)
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))   # 1: SM clock
        self.max_mhz = float(mx.value)

    def sample(self):
        ct = self.ct
        mhz, mask = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) != 0:
            return None
        self.reasons_fn(self.h, ct.byref(mask))
        return float(mhz.value), int(mask.value)


class ClockSampler:
    """Clocks during the timed region: NVML polled every 0.5 ms when the library loads,
    else nvidia-smi every 100 ms."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.nvml = None
        self.samples = []
        self.source = "none"

    def _poll(self):
        import time
        while not self._stop.is_set():
            v = self.nvml.sample()
            if v is not None:
                self.samples.append(v)
            time.sleep(0.0005)

    def __enter__(self):
        try:
            self.nvml = NvmlClocks(self.uuid)
            import threading
            self._stop = threading.Event()
            self._thr = threading.Thread(target=self._poll, daemon=True)
            self._thr.start()
            self.source = "nvml"
            return self
        except Exception:
            self.nvml = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.nvml is not None:
            self._stop.set()
            self._thr.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        if self.nvml is not None:
            for mhz, mask in self.samples:
                sm.append(mhz)
                for n, bit in NvmlClocks.BITS.items():
                    if mask & bit:
                        reasons.add(n)
            mx = [self.nvml.max_mhz]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            if self.uuid and self.uuid not in f[0]:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "source": self.source}


class L2Flush:
    """Evicts the L2 before a timed step: writes a buffer of `nbytes`, then reads another of
    that size, so that the L2 holds only clean lines of the second buffer (a write alone
    would leave the written lines dirty, and their write-back would fall inside the next
    timed region)."""

    def __init__(self, nbytes: int, dev):
        import torch
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.ones(nbytes // 4, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)   # int32 in and out: no widened copy of the buffer


def planned_timing(rdp, sess, w, xs, ys, idx, seg, n_seg, per_layer, flush, stream, reps):
    """Median CUDA-event time of one step with the batch planned once for all its layers:
    slora_plan_remake, then slora_plan_apply for every layer (each step after an L2 flush,
    outside its events); the plan object is made before the timed steps."""
    import torch
    plan = rdp.slora_plan_create(sess.pool, per_layer, w.T, idx, seg, n_seg, None, stream)
    try:
        def step():
            rdp.slora_plan_remake(plan, idx, seg, None, stream)
            for l in range(w.n_layers):
                ps = list(range(l * per_layer, (l + 1) * per_layer))
                rdp.slora_plan_apply(plan, ps, [xs[p] for p in ps], [ys[p] for p in ps], stream)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        t = [a.elapsed_time(b) for a, b in ev]
    finally:
        rdp.slora_plan_destroy(plan)
    ms = statistics.median(t)
    return {"ms_per_step": ms, "value": w.T / (ms * 1e-3 / w.n_layers), "unit": "tokens/s/layer", "steps": reps,
            "includes": "slora_plan_remake (the plan kernel) once, then slora_plan_apply (the decode kernel, and "
                        "the segment kernel) for each of the step's layers"}


def graph_timing(step_on, flush, stream, reps):
    """Median and mean CUDA-event time of one step replayed from a CUDA graph, each replay
    preceded (outside its events) by a replay of a graph that flushes the L2."""
    import torch
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        gs, gf = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            step_on(side)      # warm the capture stream
            torch.cuda.current_stream().synchronize()
            with torch.cuda.graph(gf, stream=side):
                flush()
            with torch.cuda.graph(gs, stream=side):
                step_on(torch.cuda.current_stream())
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for a, b in ev:
                gf.replay()
                a.record(side)
                gs.replay()
                b.record(side)
            side.synchronize()
        stream.wait_stream(side)
        t = [a.elapsed_time(b) for a, b in ev]
        return {"ms_per_step": statistics.median(t), "mean_ms": statistics.fmean(t), "replays": reps,
                "l2": "flush graph replayed before every step replay, outside its events"}
    except Exception as e:   # a capture the runtime refuses is reported, not fatal
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_rate(w: W.Workload, seconds: float):
    """Tokens/s per layer of the fp64 oracle on a bounded token sample (projection 0)."""
    import oracle
    x, y0 = w.x(0), w.y0(0)
    rng = np.random.default_rng(1)
    per_call = min(w.T, 64)
    done, t_used, calls = 0, 0.0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        sel = np.sort(rng.choice(w.T, per_call, replace=False)).astype(np.int32)
        s = time.perf_counter()
        oracle.workload_reference(w, p=0, sel=sel, x=x, y0=y0)
        t_used += time.perf_counter() - s
        done += per_call
        calls += 1
    # one layer = n_proj / n_layers projections of the same work
    proj_per_layer = w.n_proj // w.n_layers
    rate = done / (t_used * proj_per_layer)
    sample = (f"{calls} oracle calls x {per_call} random tokens of projection 0 "
              f"({done} token-projections, {t_used:.1f} s), scaled to {proj_per_layer} "
              f"projection(s) per layer")
    return rate, oracle.threads(), sample


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = W.by_name(args.workload, seed=args.seed)
    steps = args.steps or 3
    warm = args.warmup
    # about a minute in all whatever K and W are (each step makes at least one oracle call)
    seconds = max(0.1, min(20.0, 60.0 / max(1, steps + warm)))
    for _ in range(warm):
        oracle_rate(w, 0.5)
    rates, cores, sample = [], 1, ""
    t0 = time.perf_counter()
    for _ in range(steps):
        r, cores, sample = oracle_rate(w, seconds)
        rates.append(r)
    wall = time.perf_counter() - t0
    value = statistics.mean(rates)
    line = {
        "impl": "reference", "metric": "lora_delta_tokens_per_s_per_layer", "value": value,
        "unit": "tokens/s/layer", "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": 1e3 * wall / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": config_of(w, "oracle bounded sample; no L2 concerns on the CPU"),
        "cpu_baseline": {"value": value, "unit": "tokens/s/layer", "cores": cores,
                         "kind": "oracle", "sample": f"each step: {sample}"},
        "e2e": {"value": value, "unit": "tokens/s/layer", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w: W.Workload, l2: str):
    used = w.used_adapters()
    return {"workload": w.name, "hidden": w.hidden, "projections": w.n_proj, "layers": w.n_layers,
            "tokens": w.T, "prefill_segments": w.n_seg, "adapters": w.n_adapters,
            "unique_adapters": int(used.size), "pool_pages": w.num_pages,
            "kv_pages": w.kv_pages, "l2": l2}


# ---------------------------------------------------------------- rank launcher
def launch_ranks(args) -> int:
    """Start ``args.gpus`` processes of this script, one per GPU, with the rank variables a
    torchrun launch would set; rank 0's output is the run's output.  If a rank fails the
    others are stopped (they would wait in a collective)."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    procs = []
    for r in range(args.gpus):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(args.gpus),
                   LOCAL_WORLD_SIZE=str(args.gpus), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + sys.argv[1:], env=env))
    rc = 0
    while procs:
        for p in list(procs):
            code = p.poll()
            if code is None:
                continue
            procs.remove(p)
            if code != 0:
                rc = rc or code
                for q in procs:
                    q.terminate()
        time.sleep(0.05)
    return rc


def dry_run(args, rank: int, world: int) -> int:
    """The launcher's path without a GPU: every rank joins a gloo group and counts itself."""
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("gloo")
    n = torch.ones(1)
    if world > 1:
        dist.all_reduce(n)
    if rank == 0:
        print(json.dumps({"metric": "lora_delta_tokens_per_s_per_layer", "value": None,
                          "unit": "tokens/s/layer", "n_gpus": world, "dry_run": True,
                          "ranks_started": int(n.item()), "impl": args.impl,
                          "config": {"workload": args.workload}}), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- extra workloads
def measure_extra(rdp, w, dev, flush, stream, hbm, fp16_tflops, reps=100):
    """One call per layer of workload ``w`` (all its projections in one call), timed with
    CUDA events after an L2 flush: the whole call as a caller runs it (its kernels chained
    by programmatic dependent launch), and, in a second pass, the kernels after the plan
    (the pool records an event between the plan and the rest, which breaks that chain)."""
    import torch
    from rank_delta_paged_gb300.harness import PoolSession
    sess = PoolSession(w, device=dev.index)
    try:
        sess.load(w.used_adapters(), stream)
        per_layer = w.n_proj // w.n_layers
        ins = [sess.device_inputs(p) for p in range(per_layer)]
        xs = [i[0] for i in ins]
        ys = [i[1].clone() for i in ins]
        idx, seg = ins[0][2], ins[0][3]

        def call(st):
            if per_layer > 1:
                rdp.slora_lora_apply_multi(sess.pool, list(range(per_layer)), xs, ys, w.T, idx, seg,
                                           w.n_seg, None, st)
            else:
                rdp.slora_lora_apply(sess.pool, 0, xs[0], ys[0], w.T, idx, seg, w.n_seg, None, st)

        for _ in range(3):
            call(stream)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
        for e in ev:
            for x in e:
                x.record(stream)
        torch.cuda.synchronize()
        for a, b, c in ev:
            flush()
            a.record(stream)
            call(stream)
            c.record(stream)
        torch.cuda.synchronize()
        call_ms = statistics.median(a.elapsed_time(c) for a, b, c in ev)
        for a, b, c in ev:
            flush()
            rdp.slora_pool_set_stage_event(sess.pool, b)
            call(stream)
            c.record(stream)
        torch.cuda.synchronize()
        rdp.slora_pool_set_stage_event(sess.pool, None)
        kern_ms = statistics.median(b.elapsed_time(c) for a, b, c in ev)
        status = sess.device_status()
    finally:
        sess.close()
    nbytes = algorithmic_bytes(w) / w.n_proj * per_layer
    flops = algorithmic_flops(w) / w.n_proj * per_layer
    t = kern_ms / 1e3
    attain = max(nbytes / (hbm * 1e9), flops / (fp16_tflops * 1e12))
    return {
        "workload": w.name, "tokens": w.T, "projections_per_call": per_layer, "prefill_segments": w.n_seg,
        "value": w.T / (call_ms / 1e3), "unit": "tokens/s/layer", "ms_per_call": call_ms,
        "kernel_ms": kern_ms, "status": status,
        "roofline": {"bound": "hbm", "achieved": nbytes / t / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": nbytes / t / 1e9 / hbm, "algorithmic_bytes_per_call": nbytes},
        "tensor": {"achieved_tflops": flops / t / 1e12, "peak_tflops": fp16_tflops,
                   "frac": flops / t / 1e12 / fp16_tflops, "flops_per_call": flops,
                   "peak_kind": "measured in this run: torch.matmul fp16 8192^3, best of 10"},
        "attainable_frac": attain / t,
        "timing": "median of %d calls, each after an L2 flush (2 x L2 written, then 2 x L2 read); ms_per_call: the call's "
                  "kernels chained as a caller runs them; kernel_ms: a second pass, from the event the pool records after "
                  "the plan to the end of the call" % reps,
    }


def measure_layers_extra(rdp, w, dev, flush, stream, hbm, reps=60):
    """An iteration of workload ``w``'s layers (one projection each), timed with CUDA events
    after an L2 flush: one slora_lora_apply per layer, and the batch planned once
    (slora_plan_remake, then slora_plan_apply per layer)."""
    import torch
    from rank_delta_paged_gb300.harness import PoolSession
    sess = PoolSession(w, device=dev.index)
    try:
        sess.load(w.used_adapters(), stream)
        ins = [sess.device_inputs(p) for p in range(w.n_proj)]
        xs = [i[0] for i in ins]
        ys = [i[1].clone() for i in ins]
        idx = ins[0][2]
        plan = rdp.slora_plan_create(sess.pool, 1, w.T, idx, None, 0, None, stream)
        try:
            def per_layer_calls():
                for p in range(w.n_proj):
                    rdp.slora_lora_apply(sess.pool, p, xs[p], ys[p], w.T, idx, None, 0, None, stream)

            def planned():
                rdp.slora_plan_remake(plan, idx, None, None, stream)
                for p in range(w.n_proj):
                    rdp.slora_plan_apply(plan, [p], [xs[p]], [ys[p]], stream)

            out = {}
            for name, step in (("calls", per_layer_calls), ("planned", planned)):
                for _ in range(3):
                    step()
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
                torch.cuda.synchronize()
                for a, b in ev:
                    flush()
                    a.record(stream)
                    step()
                    b.record(stream)
                torch.cuda.synchronize()
                out[name] = statistics.median(a.elapsed_time(b) for a, b in ev)
        finally:
            rdp.slora_plan_destroy(plan)
        status = sess.device_status()
    finally:
        sess.close()
    layer_bytes = algorithmic_bytes(w) / w.n_proj
    res = {"workload": w.name, "tokens": w.T, "layers": w.n_layers, "status": status,
           "timing": "median of %d steps, each after an L2 flush (2 x L2 written, then 2 x L2 read)" % reps}
    for name, ms in out.items():
        per_layer_s = ms / 1e3 / w.n_layers
        res[name] = {"ms_per_step": ms, "us_per_layer": per_layer_s * 1e6, "value": w.T / per_layer_s,
                     "unit": "tokens/s/layer",
                     "roofline_per_layer": {"achieved": layer_bytes / per_layer_s / 1e9, "peak": hbm, "unit": "GB/s",
                                            "frac": layer_bytes / per_layer_s / 1e9 / hbm,
                                            "algorithmic_bytes_per_layer": layer_bytes,
                                            "includes": "every kernel of the step (plans included), per layer"}}
    res["calls"]["includes"] = "one slora_lora_apply per layer (plan kernel + decode kernel each)"
    res["planned"]["includes"] = ("slora_plan_remake once (the plan kernel), then slora_plan_apply per layer "
                                  "(the decode kernel)")
    res["speedup"] = out["calls"] / out["planned"]
    return res


# ---------------------------------------------------------------- our arm
def main():
    args = parse()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch_ranks(args)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but {world} rank(s) were started", file=sys.stderr)
        return 2
    if args.dry_run:
        return dry_run(args, rank, world)
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist
    import rank_delta_paged_gb300 as rdp
    from rank_delta_paged_gb300.harness import PoolSession
    from rank_delta_paged_gb300.replicas import job_totals, replica_seed, tokens_per_s_per_layer

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    rdp.build.build()
    lib = rdp.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    wkw = {}
    if args.workload in ("mixed_iteration", "decode_13b_zoo", "decode_7b", "prefill_7b") and args.layers > 0:
        wkw["n_layers"] = args.layers
    if args.workload == "mixed_iteration":
        if args.pool_gib > 0:
            wkw["pool_bytes"] = int(args.pool_gib * (1 << 30))
    w = W.by_name(args.workload, seed=replica_seed(args.seed, rank), **wkw)
    used = w.used_adapters()
    sess = PoolSession(w, device=local)
    load_mode = {"zero_copy": rdp.SLORA_LOAD_ZERO_COPY, "copy_engine": rdp.SLORA_LOAD_COPY_ENGINE}[args.load_mode]
    rdp.slora_pool_set_load_mode(sess.pool, load_mode)
    stream = torch.cuda.current_stream()
    sess.load(used, stream)
    dev = torch.device("cuda", local)
    xs, ys, y0s = [], [], []
    for p in range(w.n_proj):
        x, y0, idx, seg = sess.device_inputs(p)
        xs.append(x)
        y0s.append(y0)
        ys.append(y0.clone())
    n_seg = w.n_seg
    l2 = int(torch.cuda.get_device_properties(local).L2_cache_size)
    flush = L2Flush(2 * max(l2, 64 << 20), dev)

    per_layer = w.n_proj // w.n_layers
    multi = args.apply == "multi" and per_layer > 1

    def apply_layer(l, st):
        ps = list(range(l * per_layer, (l + 1) * per_layer))
        if multi:
            rdp.slora_lora_apply_multi(sess.pool, ps, [xs[p] for p in ps], [ys[p] for p in ps], w.T, idx, seg,
                                       n_seg, None, st)
        else:
            for p in ps:
                rdp.slora_lora_apply(sess.pool, p, xs[p], ys[p], w.T, idx, seg, n_seg, None, st)

    def step():
        for l in range(w.n_layers):
            apply_layer(l, stream)

    if args.profile_calls > 0:
        for _ in range(args.profile_calls):
            flush()
            apply_layer(0, stream)
        torch.cuda.synchronize()
        status = sess.device_status()
        sess.close()
        return 0 if status == 0 else 3

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # size K so the timed region lasts about 2 s (clock sampling needs samples under load)
    if args.steps > 0:
        K = args.steps
    else:
        # device time of one flush + step, so that the timed region lasts about 2 s
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        per = float("inf")
        for _ in range(2):   # the faster of two passes: the first can include one-off costs
            g0.record(stream)
            for _ in range(5):
                flush()
                step()
            g1.record(stream)
            torch.cuda.synchronize()
            per = min(per, g0.elapsed_time(g1) / 5 / 1e3)
        K = int(min(20000, max(10, 2.0 / max(per, 1e-6))))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    launches0 = rdp.slora_pool_launch_count(sess.pool)
    uuid = ""
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(uuid) as clk:
        for k in range(K):
            flush()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize()
    barrier()
    launches = rdp.slora_pool_launch_count(sess.pool) - launches0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms, job_tokens = job_totals(float(sum(step_ms)), float(w.T), dev, world)
    ms_per_step = total_ms / K
    value = tokens_per_s_per_layer(job_tokens, w.n_layers, ms_per_step)

    # the same step replayed from a CUDA graph (no host launch cost): one graph zeroes the
    # flush buffer, the other holds the step; CUDA events bracket each step replay
    def step_on(st):
        for l in range(w.n_layers):
            apply_layer(l, st)

    graph = graph_timing(step_on, flush, stream, max(100, min(K, 2000)))
    planned = None
    if w.n_layers > 1:
        # the same step with the batch planned once for all its layers
        planned = planned_timing(rdp, sess, w, xs, ys, idx, seg, n_seg, per_layer, flush, stream,
                                 max(50, min(K, 500)))
        planned["speedup_vs_a_plan_per_layer"] = ms_per_step / planned["ms_per_step"]

    # dominant kernel roofline: the delta kernel(s) of one call (one projection, or one
    # layer's projections with --apply multi), timed on their own (the pool records an
    # event between the plan and the delta; that record serialises the two kernels, so
    # this pass is separate from the timed steps above)
    hbm, peak_kind = peaks()
    alg_bytes = algorithmic_bytes(w)
    call_projs = per_layer if multi else 1
    alg_bytes_launch = alg_bytes / w.n_proj * call_projs
    Kd = min(K, 200)
    d0 = [torch.cuda.Event(enable_timing=True) for _ in range(Kd)]
    d1 = [torch.cuda.Event(enable_timing=True) for _ in range(Kd)]
    for ev in d0 + d1:
        ev.record(stream)   # creates the events
    torch.cuda.synchronize()
    for k in range(Kd):
        flush()
        rdp.slora_pool_set_stage_event(sess.pool, d0[k])
        if multi:
            apply_layer(0, stream)
        else:
            rdp.slora_lora_apply(sess.pool, 0, xs[0], ys[0], w.T, idx, seg, n_seg, None, stream)
        d1[k].record(stream)
    torch.cuda.synchronize()
    rdp.slora_pool_set_stage_event(sess.pool, None)
    delta_ms = statistics.median(a.elapsed_time(b) for a, b in zip(d0, d1))
    t_d = torch.tensor([delta_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t_d, op=dist.ReduceOp.MAX)
    delta_ms = float(t_d.item())
    achieved = alg_bytes_launch / (delta_ms / 1e3) / 1e9
    step_achieved = alg_bytes / (ms_per_step / 1e3) / 1e9
    kernel_stats = rdp.slora_pool_kernel_stats(sess.pool) if hasattr(rdp, "slora_pool_kernel_stats") else None

    # the padded batched-GEMM comparison path on projection 0 (decode-only batches)
    bmm = None
    if args.bmm and n_seg == 0:
        nb = rdp.slora_bmm_workspace_bytes(sess.pool, w.T)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        yb = ys[0].clone()
        for _ in range(3):
            rdp.slora_lora_apply_bmm(sess.pool, 0, xs[0], yb, w.T, idx, ws, nb, None, stream)
        b0 = [torch.cuda.Event(enable_timing=True) for _ in range(Kd)]
        b1 = [torch.cuda.Event(enable_timing=True) for _ in range(Kd)]
        c0 = [torch.cuda.Event(enable_timing=True) for _ in range(Kd)]
        c1 = [torch.cuda.Event(enable_timing=True) for _ in range(Kd)]
        for k in range(Kd):
            flush()
            b0[k].record(stream)
            rdp.slora_lora_apply_bmm(sess.pool, 0, xs[0], yb, w.T, idx, ws, nb, None, stream)
            b1[k].record(stream)
            flush()
            c0[k].record(stream)
            rdp.slora_lora_apply(sess.pool, 0, xs[0], ys[0], w.T, idx, seg, n_seg, None, stream)
            c1[k].record(stream)
        torch.cuda.synchronize()
        bmm_ms = statistics.median(a.elapsed_time(b) for a, b in zip(b0, b1))
        cus_ms = statistics.median(a.elapsed_time(b) for a, b in zip(c0, c1))
        bmm = {"ms": bmm_ms, "custom_ms": cus_ms, "custom_speedup": bmm_ms / cus_ms, "workspace_bytes": int(nb),
               "padded_rank": int(nb // max(1, w.T * 4 * w.hidden + 2 * w.T)),
               "includes": "gather of every token's padded A^T and s*B from the pages + two cuBLAS strided "
                           "batched GEMMs (fp16 in, fp32 accumulation); custom = plan + delta kernels, one "
                           "projection, each after an L2 flush"}

    # ---- end to end through the C ABI from pinned host buffers --------------------
    hx = [torch.from_numpy(w.x(p).view(np.int16)).view(torch.float16).pin_memory() for p in range(w.n_proj)]
    hy0 = [torch.from_numpy(w.y0(p).view(np.int16)).view(torch.float16).pin_memory() for p in range(w.n_proj)]
    hidx = torch.from_numpy(w.token_adapter_idx).pin_memory()
    hseg = None if w.seg_indptr is None else torch.from_numpy(w.seg_indptr).pin_memory()
    hy = [torch.empty_like(h) for h in hy0]
    hy = [h.pin_memory() for h in hy]
    adapter_bytes = sum(4 * int(w.ranks[a]) * w.hidden * w.n_proj for a in used)
    h2d = sum(h.numel() * 2 for h in hx) + sum(h.numel() * 2 for h in hy0) + hidx.numel() * 4 + \
        (0 if hseg is None else hseg.numel() * 4) + adapter_bytes
    d2h = sum(h.numel() * 2 for h in hy)
    e2e_ms = []
    for k in range(args.e2e_steps + 2):
        sess.evict(used, stream)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        # the step's inputs go up before the adapter load is enqueued (the load makes the
        # stream wait for the adapters; the input copies need not)
        idx.copy_(hidx, non_blocking=True)
        if hseg is not None:
            seg.copy_(hseg, non_blocking=True)
        for p in range(w.n_proj):
            xs[p].copy_(hx[p], non_blocking=True)
            ys[p].copy_(hy0[p], non_blocking=True)
        sess.load(used, stream)
        for l in range(w.n_layers):
            apply_layer(l, stream)
            for p in range(l * per_layer, (l + 1) * per_layer):
                hy[p].copy_(ys[p], non_blocking=True)
        torch.cuda.synchronize()
        if k >= 2:
            e2e_ms.append(1e3 * (time.perf_counter() - t0))
    # the same end-to-end step with the batch's adapters already resident (a serving loop
    # whose adapters stayed in the pool): inputs up, apply, y down
    sess.load(used, stream)
    torch.cuda.synchronize()
    warm_ms = []
    for k in range(args.e2e_steps + 2):
        t0 = time.perf_counter()
        idx.copy_(hidx, non_blocking=True)
        if hseg is not None:
            seg.copy_(hseg, non_blocking=True)
        for p in range(w.n_proj):
            xs[p].copy_(hx[p], non_blocking=True)
            ys[p].copy_(hy0[p], non_blocking=True)
        for l in range(w.n_layers):
            apply_layer(l, stream)
            for p in range(l * per_layer, (l + 1) * per_layer):
                hy[p].copy_(ys[p], non_blocking=True)
        torch.cuda.synchronize()
        if k >= 2:
            warm_ms.append(1e3 * (time.perf_counter() - t0))
    # the load path alone: a cold load of the batch's adapters (host call + device work)
    load_wall, load_dev = [], []
    for k in range(5):
        sess.evict(used, stream)
        torch.cuda.synchronize()
        la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        la.record(stream)
        sess.load(used, stream)
        lb.record(stream)
        torch.cuda.synchronize()
        if k >= 1:
            load_wall.append(1e3 * (time.perf_counter() - t0))
            load_dev.append(la.elapsed_time(lb))
    load = {"adapters": len(used), "bytes": int(adapter_bytes),
            "wall_ms": statistics.median(load_wall), "stream_ms": statistics.median(load_dev),
            "gb_per_s": adapter_bytes / (statistics.median(load_wall) * 1e-3) / 1e9,
            "mode": args.load_mode,
            "includes": "host call (page allocation, page tables, launches) and the load path (" +
                        ("the load kernel reading the pinned store over the CPU-GPU link" if args.load_mode == "zero_copy"
                         else "one cudaMemcpyAsync per adapter into the staging ring, the load kernel from it") +
                        "); the directory update"}
    e2e_job_ms, _ = job_totals(statistics.mean(e2e_ms) if e2e_ms else float("nan"), float(w.T), dev, world)
    warm_job_ms, _ = job_totals(statistics.mean(warm_ms) if warm_ms else float("nan"), float(w.T), dev, world)
    e2e_value = tokens_per_s_per_layer(job_tokens, w.n_layers, e2e_job_ms)
    warm_value = tokens_per_s_per_layer(job_tokens, w.n_layers, warm_job_ms)
    prefetch = None
    if args.prefetch > 0 and w.n_seg == 0:
        from rank_delta_paged_gb300.harness import prefetch_overlap
        prefetch = {name: prefetch_overlap(sess, args.prefetch, stream, mode)
                    for name, mode in (("zero_copy", rdp.SLORA_LOAD_ZERO_COPY),
                                       ("copy_engine", rdp.SLORA_LOAD_COPY_ENGINE))}
        rdp.slora_pool_set_load_mode(sess.pool, load_mode)
        sess.load(used, stream)
    pressure = None
    if args.pressure > 0:
        from rank_delta_paged_gb300.harness import pressure_run
        sess.evict(used, stream)
        pressure = pressure_run(sess, args.pressure, stream)
    status = sess.device_status()
    if status != 0:
        print(f"device status {status} after the run", file=sys.stderr)
        return 3
    traffic, traffic_note = traffic_of(w.name)
    extras = None
    if args.workload == DEFAULT_WORKLOAD and not args.no_extras and rank == 0:
        fp16 = fp16_peak_tflops(dev)
        extras = {"fp16_dense_peak_tflops": fp16}
        for name, kw in (("prefill_7b", {}), ("mixed_layer", {"n_layers": 1, "pool_bytes": 2 << 30})):
            wx = W.by_name("mixed_iteration" if name == "mixed_layer" else name, seed=args.seed, **kw)
            extras[name] = measure_extra(rdp, wx, dev, flush, stream, hbm, fp16)
            if extras[name]["status"] != 0:
                print(f"device status {extras[name]['status']} in {name}", file=sys.stderr)
                return 3
        # the headline batch through 8 layers: one call per layer against one plan per step
        wl = W.by_name(args.workload, seed=args.seed, n_layers=8)
        extras["decode_13b_zoo_8_layers"] = measure_layers_extra(rdp, wl, dev, flush, stream, hbm)
        if extras["decode_13b_zoo_8_layers"]["status"] != 0:
            print("device status in the 8-layer step", file=sys.stderr)
            return 3

    line = {
        "metric": "lora_delta_tokens_per_s_per_layer", "value": value, "unit": "tokens/s/layer",
        "n_gpus": world, "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; random-init adapters, no dataset)",
        "config": dict(config_of(w, "flushed: 2 x L2 written, then another 2 x L2 read (the L2 left "
                                    "holding clean lines only), before every timed step, outside the "
                                    "per-step CUDA-event intervals"),
                       apply=(f"one slora_lora_apply_multi call per layer ({per_layer} projections)" if multi
                              else "one slora_lora_apply call per projection")),
        "gpu_launches": int(launches),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic, "traffic_source": traffic_note,
                     "kernel": "delta_kernel" + (" + prefill_kernel" if n_seg else "") +
                               (f" (one call of {call_projs} projections" if multi else " (one projection") +
                               "; median CUDA-event time between the plan and the end of the call)",
                     "launch_ms": delta_ms, "algorithmic_bytes_per_launch": alg_bytes_launch,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "step": {"achieved": step_achieved, "frac": step_achieved / hbm,
                              "algorithmic_bytes": alg_bytes, "includes": "plan + delta kernels"}},
        "e2e": {"value": e2e_value, "unit": "tokens/s/layer", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_job_ms,
                "includes": "H2D of x, y0, token map; cold load of the batch's adapters from the "
                            "pinned store (load path: " + args.load_mode + "); delta; D2H of y "
                            "(the eviction before each step is outside the timed part)",
                "warm": {"value": warm_value, "ms_per_step": warm_job_ms,
                         "h2d_bytes_per_step": int(h2d - adapter_bytes), "d2h_bytes_per_step": int(d2h),
                         "includes": "the same step with the batch's adapters already resident: H2D of x, "
                                     "y0, token map; delta; D2H of y"}},
        "graph": graph,
        **({"planned": planned} if planned is not None else {}),
        "load": load,
        "flops_per_step": algorithmic_flops(w),
        "clocks": clk.summary(),
    }
    if kernel_stats is not None:
        line["kernels"] = kernel_stats
    if prefetch is not None:
        line["prefetch"] = prefetch
    if pressure is not None:
        line["pressure"] = pressure
    if bmm is not None:
        line["bmm"] = bmm
    if extras is not None:
        line["extra_workloads"] = extras
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, sample = oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s/layer", "cores": cores,
                                "kind": "oracle", "sample": sample}
        import oracle
        oracle.set_threads(1)   # the same oracle on one core, a shorter sample
        r1, _, s1 = oracle_rate(w, max(1.0, args.cpu_seconds / 3))
        oracle.set_threads(cores)
        line["cpu_baseline"]["single_core"] = {"value": r1, "cores": 1, "sample": s1}
    if rank == 0:
        print(json.dumps(line), flush=True)
    sess.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
