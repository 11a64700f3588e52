#!/usr/bin/env python
"""Benchmark of the block-sparse decode step (lsa_decode_step) on GB300.

One step = one lsa_decode_step call over one batch of synthetic input: block
scores against the mean-key summaries, per-(request, KV head) top-k with the
sink / recent tokens forced, split-K attention over the selected blocks and
the log-sum-exp merge.  The metric is decode-step calls/s on the B=16 x 32K
workload (also reported: tokens/s = B x calls/s and achieved HBM GB/s of the
algorithmic bytes: candidate summaries + forced/selected K/V + page table +
q/out).

Timing: W warm-up steps, an untimed soak under load, then exactly K steps
replayed from CUDA graphs, bracketed by a barrier and a device synchronise,
timed with CUDA events on the launching stream.  L2 stays cold: the steps
rotate over R independent instances whose combined working set is several
times the 129 MB L2 (config key "l2").  Under torchrun each rank runs an
independent replica (the step has no cross-request exchange); the time is the
max over ranks and the value counts every rank's steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, algorithmic_bytes, make_inputs  # noqa: E402

METRIC = "sparse decode-step calls/s and achieved HBM GB/s vs GB300 peak (B=16, 32K)"
L2_BYTES = 129 * 1024 * 1024


# DRAM bytes per launch from one ncu capture of each kernel as it stands
# (read + write); a kernel changed since its capture has no entry.
# dram__bytes_read.sum + dram__bytes_write.sum per launch from the ncu capture
# summarised in profiles/; emptied whenever a kernel changes after its capture.
NCU_TRAFFIC = {
    "k_attn_flat (selects)": 68_524_544 + 700_416,
    "k_score": 67_334_912 + 305_152,
}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

class Instance:
    def __init__(self, w, seed_offset, dev):
        import sparse_attention_decode_block_gb300 as L
        self.w = w.replace(seed=w.seed + 1000 * seed_offset) if seed_offset else w
        self.g = make_inputs(self.w, dev)
        g = self.g
        B, Hkv = w.batch, w.num_kv_heads
        self.cache = L.make_cache(g["k_cache"], g["v_cache"])
        self.icache = None
        self.summ = torch.zeros((g["num_pages"], Hkv, w.dk), dtype=torch.bfloat16, device=dev)
        if w.c2f_candidates > 0:
            self.icache = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
            L.lsa_build_summaries(self.icache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.c2f_tokens
        else:
            L.lsa_build_summaries(self.cache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.k_blocks
        self.params = L.make_params(B, w.num_q_heads, g["max_blocks"], w.k_blocks, w.sink, w.recent,
                                    w.softmax_scale, w.c2f_candidates, w.c2f_tokens)
        self.ws = torch.zeros(max(16, L.lsa_decode_step_workspace_size(self.cache, self.params)),
                              dtype=torch.uint8, device=dev)
        self.idx = torch.empty((B, Hkv, max(1, nsel)), dtype=torch.int32, device=dev)
        self.out = torch.empty((B, w.num_q_heads, w.dv), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, w.num_q_heads), dtype=torch.float32, device=dev)
        self.L = L

    def step(self, q=None, pt=None, lens=None, stream=None):
        g = self.g
        self.L.lsa_decode_step(g["q"] if q is None else q, self.cache, self.summ, self.icache,
                               g["page_table"] if pt is None else pt, g["seq_lens"] if lens is None else lens,
                               self.params, self.idx, self.out, self.lse, self.ws, stream)



def fused_path(w) -> bool:
    """The library takes the persistent kernel when LSA_DECODE_PATH=fused and
    the shape is one it has an instance for (GQA groups of <= 8 heads, dk =
    dv in {64, 128}, block sizes 16 / 64, no coarse-to-fine pass)."""
    group = w.num_q_heads // w.num_kv_heads
    return (os.environ.get("LSA_DECODE_PATH") == "fused" and w.c2f_candidates == 0 and w.dk == w.dv
            and w.dk in (64, 128) and group <= 8 and w.block_size in (16, 64) and not w.v_aliased)


def selects_in_attention(w) -> bool:
    """The library lets the attention kernel select the blocks (no top-k
    launch) when the tensor-core attention with an even split applies:
    GQA groups of 2..8 (even), dk = dv in {64, 128}, no coarse-to-fine pass,
    rows of at most 8192 blocks, 0 < k <= 512."""
    group = w.num_q_heads // w.num_kv_heads
    max_blocks = -(-w.seq_len // w.block_size) if w.seq_len else None
    return (not fused_path(w) and w.c2f_candidates == 0 and not w.v_aliased and w.dk == w.dv
            and w.dk in (64, 128) and group % 2 == 0 and os.environ.get("LSA_ATTENTION_PATH") != "cuda_core"
            and max_blocks is not None and max_blocks <= 8192 and 0 < w.k_blocks <= 512)


def kernels_per_step(inst) -> int:
    import ctypes
    if fused_path(inst.w):
        return 1
    w = inst.w
    if selects_in_attention(w):
        return 2   # score, attention with the selection inside
    # score + top-k (+ fine score + fine top-k) + attention
    n = 2 + (2 if w.c2f_candidates > 0 else 0) + 1
    # the tensor-core attention (GQA groups of 2..8, dk = dv in {64, 128})
    # merges its parts itself; the CUDA-core kernel adds a merge launch when split
    group = w.num_q_heads // w.num_kv_heads
    tc = (w.c2f_candidates == 0 and not w.v_aliased and w.dk == w.dv and w.dk in (64, 128)
          and group % 2 == 0 and os.environ.get("LSA_ATTENTION_PATH") != "cuda_core")
    if not tc:
        lib = inst.L.load_library()
        ws_attn = lib.lsa_sparse_decode_workspace_size(ctypes.byref(inst.cache), ctypes.byref(inst.params))
        n += 1 if ws_attn > 0 else 0
    return n


def stage_times(insts, reps: int, stream) -> dict:
    """Average device time of each stage (score, top-k, attention + merge),
    each captured in a CUDA graph of `reps` calls through the individual entry
    points (the same kernels the fused call launches), rotating L2-cold over
    the instances."""
    w = insts[0].w
    if w.c2f_candidates > 0:
        return {}
    L = insts[0].L
    B, Hkv = w.batch, w.num_kv_heads
    bufs = []
    for it in insts:
        g = it.g
        dev = g["q"].device
        bufs.append(dict(
            scores=torch.empty((B * Hkv, g["max_blocks"]), dtype=torch.float32, device=dev),
            idx=torch.empty((B * Hkv, max(1, w.k_blocks)), dtype=torch.int32, device=dev),
            ws=torch.zeros(max(16, L.lsa_sparse_decode_workspace_size(it.cache, it.params)), dtype=torch.uint8,
                           device=dev)))
    R = len(insts)

    def score(i):
        it, b = insts[i % R], bufs[i % R]
        L.lsa_score(it.g["q"], it.cache, it.summ, it.g["page_table"], it.g["seq_lens"], it.params, b["scores"],
                    stream)

    def topk(i):
        b = bufs[i % R]
        L.lsa_topk(b["scores"], None, w.k_blocks, b["idx"], stream)

    def attn(i):
        it, b = insts[i % R], bufs[i % R]
        L.lsa_sparse_decode(it.g["q"], it.cache, it.g["page_table"], it.g["seq_lens"], b["idx"].view(B, Hkv, -1),
                            it.params, it.out, it.lse, b["ws"], stream)

    out = {}
    with torch.cuda.stream(stream):
        for i in range(R):
            score(i)
            topk(i)
            attn(i)
        stream.synchronize()
        for name, fn in (("score", score), ("topk", topk), ("attention", attn)):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for i in range(reps):
                    fn(i)
            gr.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
            stream.synchronize()
            out[name] = e0.elapsed_time(e1) / reps
    return out


def max_over_ranks(ms: float, dev, world: int) -> float:
    """The timed region's length as the slowest rank saw it (every rank gets it)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_calls_per_s(steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank's replica ran `steps` calls within `ms`."""
    return steps * world / (ms / 1e3)


def run_gpu(args, rank, world, dev):
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.config]
    import sparse_attention_decode_block_gb300 as L
    L.load_library()
    first = Instance(w, 0, dev)
    step_bytes = algorithmic_bytes(w, first.g["lens"])["total"]
    R = max(2, int(np.ceil(4 * L2_BYTES / max(step_bytes, 1))))
    R = min(R, 8) if args.instances <= 0 else args.instances
    insts = [first] + [Instance(w, i, dev) for i in range(1, R)]
    accs = [algorithmic_bytes(w, it.g["lens"]) for it in insts]
    acc = {k: sum(a[k] for a in accs) // R for k in accs[0]}
    step_bytes = acc["total"]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    L.lsa_get_device_status(clear=True)

    # warm-up (eager)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            insts[i % R].step(stream=stream)
    stream.synchronize()
    code, flags = L.lsa_get_device_status(clear=True)
    if code != 0:
        raise RuntimeError(f"device status after warm-up: {L.lsa_status_string(code)} ({flags:#x})")

    # CUDA graphs of `chunk` steps cycling over the instances
    chunk = R * max(1, 64 // R)

    def capture(nsteps):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(nsteps):
                insts[i % R].step(stream=stream)
        return gr

    K = args.steps
    g_full = capture(chunk) if K >= chunk else None
    rem = K % chunk
    g_rem = capture(rem) if rem else None
    n_full = K // chunk

    def replay_k():
        for _ in range(n_full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    # soak: keep the GPU under load for ~1 s before the timed region so the
    # clock samples describe the steady state
    with torch.cuda.stream(stream):
        t_end = time.time() + args.soak
        while time.time() < t_end:
            (g_full or g_rem).replay()
            stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        replay_k()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    code, flags = L.lsa_get_device_status(clear=True)
    if code != 0:
        raise RuntimeError(f"device status after timing: {L.lsa_status_string(code)} ({flags:#x})")
    ms = max_over_ranks(ms, dev, world)

    # per-stage split (separate untimed-for-value pass, L2 flushed before each)
    st = stage_times(insts, 8 * len(insts), stream)

    # end to end through the public call with host buffers: every step copies
    # q, page table and lengths from pinned host memory and reads back out/lse
    e2e = e2e_leg(insts, args, stream)

    return dict(ms=ms, step_bytes=step_bytes, acc=acc, R=R, clocks=clocks, stages=st, e2e=e2e,
                kernels=kernels_per_step(insts[0]), w=w)


def e2e_leg(insts, args, stream):
    inst = insts[0]
    g = inst.g
    hq = g["q"].cpu().pin_memory()
    hpt = g["page_table"].cpu().pin_memory()
    hl = g["seq_lens"].cpu().pin_memory()
    hout = torch.empty(inst.out.shape, dtype=inst.out.dtype).pin_memory()
    hlse = torch.empty(inst.lse.shape, dtype=inst.lse.dtype).pin_memory()
    dq, dpt, dl = torch.empty_like(g["q"]), torch.empty_like(g["page_table"]), torch.empty_like(g["seq_lens"])
    n = max(10, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):
            dq.copy_(hq, non_blocking=True)
            dpt.copy_(hpt, non_blocking=True)
            dl.copy_(hl, non_blocking=True)
            inst.step(dq, dpt, dl, stream)
            hout.copy_(inst.out, non_blocking=True)
            hlse.copy_(inst.lse, non_blocking=True)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            dq.copy_(hq, non_blocking=True)
            dpt.copy_(hpt, non_blocking=True)
            dl.copy_(hl, non_blocking=True)
            inst.step(dq, dpt, dl, stream)
            hout.copy_(inst.out, non_blocking=True)
            hlse.copy_(inst.lse, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / n
    h2d = hq.numel() * hq.element_size() + hpt.numel() * hpt.element_size() + hl.numel() * hl.element_size()
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
    return dict(ms_per_step=ms, h2d=h2d, d2h=d2h, steps=n)


# ---------------------------------------------------------------- CPU oracle

def cpu_baseline(w, budget_s: float = 15.0):
    """The oracle as it stands on the host cores, on a bounded sample: whole
    requests of the workload (all their KV heads), summaries precomputed by
    the oracle (they are built once per block, outside the step)."""
    import oracle
    inp = make_inputs(w.replace(batch=1, seq_lens=None if w.seq_lens is None else w.seq_lens[:1]), "cpu")
    c = oracle.Cache(inp["k_cache"], inp["v_cache"])
    kw = dict(num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink, recent=w.recent,
              scale=w.softmax_scale)
    if w.c2f_candidates > 0:
        ic = oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])
        isumm, _ = oracle.summaries(ic, inp["page_table"], inp["seq_lens"], use_index_keys=True)
        kw.update(index_cache=ic, index_summ=isumm, c2f_candidates=w.c2f_candidates, c2f_tokens=w.c2f_tokens)
        summ = None
    else:
        summ, _ = oracle.summaries(c, inp["page_table"], inp["seq_lens"])
    cores = os.cpu_count() or 1
    n, t0 = 0, time.time()
    while True:
        oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], summ=summ, nthreads=cores, **kw)
        n += 1
        if time.time() - t0 > budget_s or n >= 5000:
            break
    per_req = (time.time() - t0) / n
    calls = 1.0 / (per_req * w.batch)
    return {"value": calls, "unit": "calls/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} run(s) of 1 of {w.batch} requests (all {w.num_kv_heads} KV heads), fp64 oracle, "
                      f"summaries precomputed; calls/s = 1 / ({w.batch} x time per request)"}


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="b16_32k", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="lsa", choices=["lsa", "reference"])
    ap.add_argument("--soak", type=float, default=1.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--instances", type=int, default=0,
                    help="input instances rotated over to keep L2 cold (0: enough for 4x L2); "
                         "1 keeps the device footprint small for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.config]

    if args.impl == "reference":
        # the reference arm is the CPU oracle; rank 0 alone runs it
        if rank != 0:
            return
        t0 = time.time()
        cb = cpu_baseline(w, budget_s=20.0)
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "calls/s", "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / cb["value"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": w.name, "description": w.description},
                "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": "calls/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": round(time.time() - t0, 1)}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    res = run_gpu(args, rank, world, dev)
    ms_step = res["ms"] / args.steps
    calls = job_calls_per_s(args.steps, world, res["ms"])
    peak, peak_kind = peaks()
    gbs = res["step_bytes"] / (ms_step / 1e3) / 1e9
    st = res["stages"]
    acc = res["acc"]
    stage_bytes = {"score": acc["summaries"] + acc["page_table"] + acc["q_out"] // 2,
                   "attention": acc["kv"] + acc["q_out"] // 2 + acc["q_out"] // 2, "topk": 0}
    kernel_ms = {}
    if st and selects_in_attention(w):
        # the step is two launches: the score kernel and the attention kernel
        # that also selects the blocks; the latter's time is the step's time
        # minus the score kernel's (both CUDA-event timings)
        kernel_ms = {"k_score": st["score"], "k_attn_flat (selects)": max(ms_step - st["score"], 1e-9)}
        kbytes = {"k_score": stage_bytes["score"], "k_attn_flat (selects)": stage_bytes["attention"]}
    elif st:
        kernel_ms = dict(st)
        kbytes = stage_bytes
    dominant = None if fused_path(w) or not kernel_ms else max(kernel_ms, key=kernel_ms.get)
    if dominant:
        ach = kbytes[dominant] / (kernel_ms[dominant] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_kind": peak_kind,
                "duration_us": round(kernel_ms[dominant] * 1e3, 2),
                "timing": "step minus score kernel" if dominant.startswith("k_attn_flat") else "CUDA graph of the stage",
                "traffic": NCU_TRAFFIC.get(dominant) if w.name == "b16_32k" else None}
    else:
        # the persistent kernel is the whole step: its launch time is the step time
        roof = {"bound": "hbm", "kernel": "k_decode_fused", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(gbs / peak, 4), "peak_kind": peak_kind, "traffic": None}
    cb = None
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline(res["w"])
    e2e = res["e2e"]
    w = res["w"]
    line = {
        "metric": METRIC, "value": round(calls, 1), "unit": "calls/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "batch": w.batch,
                   "seq_len": w.seq_len or "ragged", "parallelism": f"replicas x{world}",
                   "path": "fused" if fused_path(w) else "pipeline",
                   "l2": (f"cold: {res['R']} rotating instances, " if res['R'] * res['step_bytes'] >= 2 * L2_BYTES
                          else f"NOT cold (profiling setting): {res['R']} instance(s), ")
                         + f"{res['R'] * res['step_bytes'] / 2**20:.0f} MiB touched per rotation vs 129 MB L2"},
        "tokens_per_s": round(calls * w.batch, 1),
        "step": {"algorithmic_bytes": res["step_bytes"], "bytes_split": acc, "gbs": round(gbs, 1),
                 "frac_of_peak": round(gbs / peak, 4), "frac_of_8tbs": round(gbs / 8000.0, 4)},
        "stages_ms": {k: round(v, 5) for k, v in st.items()},
        "kernels_ms": {k: round(v, 5) for k, v in kernel_ms.items()},
        "roofline": roof,
        "cpu_baseline": cb,
        "e2e": {"value": round(1e3 / e2e["ms_per_step"] * world, 1), "unit": "calls/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "note": "eager public-API calls from Python, pinned host buffers copied in and out every step"},
        "gpu_launches": res["kernels"] * args.steps,
        "clocks": res["clocks"],
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
