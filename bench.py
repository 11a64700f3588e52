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


# (workload, kernel) -> dram__bytes_read.sum + dram__bytes_write.sum per
# launch from the ncu capture summarised in profiles/; an entry is removed
# whenever its kernel changes after the capture.
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# each kernel the roofline may name, from one ncu capture of
# `python bench.py --config NAME --steps 8 --warmup 3 --soak 0
# --no-cpu-baseline --instances 1` (summaries in profiles/); an entry goes
# when its kernel changes until it is captured again.
NCU_TRAFFIC = {
    ("b16_32k", "k_attn_flat (selects)"): 68554837, ("b16_32k", "k_score"): 67405483,
    ("ragged", "k_attn_flat (selects)"): 526917717, ("ragged", "k_score"): 139504299,
    ("b16_32k_quest", "k_attn_flat (selects)"): 68547755, ("b16_32k_quest", "k_score_quest"): 135514197,
    ("c2f", "k_c2f_fine"): 9007488, ("c2f", "k_score"): 8614912, ("c2f_wrelu", "k_c2f_fine"): 9009067,
    ("mla", "k_score"): 76397312, ("mla", "k_topk"): 303104, ("mla", "k_sparse_attn_umma"): 9537920,
    ("c2f", "k_sparse_attn_umma"): 4430720,
    ("c2f_pq", "k_pq_scores"): 67523021, ("c2f_pq", "k_pq_hist + k_pq_select"): 25293645,
}


def peaks(kind: str = "hbm"):
    """(peak, "measured" | "fallback"): HBM GB/s, or dense bf16 TFLOP/s
    (the burst figure: the kernel is timed on its own)."""
    key, fallback = ("hbm_gbs", 6800.0) if kind == "hbm" else ("bf16_tflops", 1900.0)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p[key]), "measured"
    except Exception:
        return fallback, "fallback"


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
        if w.summary_kind == 1:
            self.summ = torch.zeros((g["num_pages"], Hkv, 2, w.dk), dtype=torch.bfloat16, device=dev)
        else:
            self.summ = torch.zeros((g["num_pages"], Hkv, w.dk), dtype=torch.bfloat16, device=dev)
        if w.pq_candidates > 0:
            self.icache = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
            nsel = w.c2f_tokens
        elif w.c2f_candidates > 0:
            self.icache = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
            L.lsa_build_summaries(self.icache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.c2f_tokens
        elif w.summary_kind == 1:
            L.lsa_build_minmax_summaries(self.cache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.k_blocks
        else:
            L.lsa_build_summaries(self.cache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.k_blocks
        self.params = L.make_params(B, w.num_q_heads, g["max_blocks"], w.k_blocks, w.sink, w.recent,
                                    w.softmax_scale, w.c2f_candidates, w.c2f_tokens,
                                    summary_kind=w.summary_kind, fine_head_weights=g.get("fine_weights"),
                                    pq_candidates=w.pq_candidates, pq_codes=g.get("pq_codes"),
                                    pq_codebook=g.get("pq_codebook"), pq_hit=g.get("pq_hit"))
        self.ws = torch.zeros(max(16, L.lsa_decode_step_workspace_size(self.cache, self.params)),
                              dtype=torch.uint8, device=dev)
        self.idx = torch.empty((B, Hkv, max(1, nsel)), dtype=torch.int32, device=dev)
        self.out = torch.empty((B, w.num_q_heads, w.dv), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, w.num_q_heads), dtype=torch.float32, device=dev)
        self.L = L

    def step(self, q=None, pt=None, lens=None, stream=None, out=None, lse=None):
        g = self.g
        self.L.lsa_decode_step(g["q"] if q is None else q, self.cache, self.summ, self.icache,
                               g["page_table"] if pt is None else pt, g["seq_lens"] if lens is None else lens,
                               self.params, self.idx, self.out if out is None else out,
                               self.lse if lse is None else lse, self.ws, stream)



def selects_in_attention(w) -> bool:
    """The library lets the attention kernel select the blocks (no top-k
    launch) when the tensor-core attention with an even split applies:
    GQA groups of 2..8 (even), dk = dv in {64, 128}, no coarse-to-fine pass,
    rows of at most 8192 blocks, 0 < k <= 512."""
    group = w.num_q_heads // w.num_kv_heads
    max_blocks = -(-max(w.seq_len, (w.seq_len_range or (0, 0))[1]) // w.block_size)
    return (w.c2f_candidates == 0 and not w.v_aliased and w.dk == w.dv
            and w.dk in (64, 128) and 2 <= group <= 8 and group % 2 == 0
            and os.environ.get("LSA_ATTENTION_PATH") != "cuda_core"
            and 0 < max_blocks <= 8192 and 0 < w.k_blocks <= 512)


def kernels_per_step(inst) -> int:
    """Kernel launches of one step, as the library's planner makes them."""
    n = inst.L.lsa_decode_step_launches(inst.cache, inst.icache, inst.params)
    assert n > 0, "invalid step shapes"
    return n


def pq_stage_times(insts, reps: int, stream) -> dict:
    """The PQ32 coarse-to-fine step's stages through their entry points:
    the coarse scores (lsa_pq_scores) and attention over each instance's
    own selection (lsa_sparse_decode); the selection kernels are the step's
    time minus these."""
    w = insts[0].w
    L = insts[0].L
    R = len(insts)
    bufs = []
    with torch.cuda.stream(stream):
        for it in insts:
            it.step(stream=stream)   # each instance's own selection
        stream.synchronize()
    for it in insts:
        T = it.g["max_blocks"] * w.block_size
        bufs.append(dict(coarse=torch.empty((w.batch, T), dtype=torch.float32, device=it.g["q"].device),
                         ws=torch.zeros(max(16, L.lsa_sparse_decode_workspace_size(it.cache, it.params)),
                                        dtype=torch.uint8, device=it.g["q"].device)))

    def pq_scores(i):
        it, b = insts[i % R], bufs[i % R]
        L.lsa_pq_scores(it.g["q"], it.icache, it.g["page_table"], it.g["seq_lens"], it.params, b["coarse"], stream)

    def attn(i):
        it, b = insts[i % R], bufs[i % R]
        L.lsa_sparse_decode(it.g["q"], it.cache, it.g["page_table"], it.g["seq_lens"], it.idx, it.params, it.out,
                            it.lse, b["ws"], stream)

    out = {}
    with torch.cuda.stream(stream):
        for fn in (pq_scores, attn):
            for i in range(R):
                fn(i)
        stream.synchronize()
        out["pq_scores"] = graph_ms(pq_scores, reps, stream)
        out["attention"] = graph_ms(attn, reps, stream)
    return out


def stage_times(insts, reps: int, stream) -> dict:
    """Average device time of each stage of the step, each captured in a CUDA
    graph of `reps` calls through its own entry point (the kernels the step
    launches), rotating L2-cold over the instances: score (lsa_score), top-k
    (lsa_topk), the coarse-to-fine fine pass (lsa_fine_topk) and attention
    with its merge (lsa_sparse_decode over the stage's own selection)."""
    w = insts[0].w
    if w.pq_candidates > 0:
        return pq_stage_times(insts, reps, stream)
    L = insts[0].L
    B, Hkv = w.batch, w.num_kv_heads
    c2f = w.c2f_candidates > 0
    bufs = []
    for it in insts:
        g = it.g
        dev = g["q"].device
        k1 = w.c2f_candidates if c2f else max(1, w.k_blocks)
        b = dict(scores=torch.empty((B * Hkv, g["max_blocks"]), dtype=torch.float32, device=dev),
                 idx=torch.empty((B * Hkv, k1), dtype=torch.int32, device=dev),
                 ws=torch.zeros(max(16, L.lsa_sparse_decode_workspace_size(it.cache, it.params)),
                                dtype=torch.uint8, device=dev))
        if c2f:
            b["tok"] = torch.empty((B, Hkv, w.c2f_tokens), dtype=torch.int32, device=dev)
            b["fws"] = torch.empty(B * Hkv * w.c2f_candidates * w.block_size * 4 + 256, dtype=torch.uint8,
                                   device=dev)
        bufs.append(b)
    R = len(insts)

    def score(i):
        it, b = insts[i % R], bufs[i % R]
        cache = it.icache if c2f else it.cache
        L.lsa_score(it.g["q"], cache, it.summ, it.g["page_table"], it.g["seq_lens"], it.params, b["scores"],
                    stream)

    def topk(i):
        b = bufs[i % R]
        L.lsa_topk(b["scores"], None, b["idx"].shape[1], b["idx"], stream)

    def fine(i):
        it, b = insts[i % R], bufs[i % R]
        L.lsa_fine_topk(it.g["q"], it.icache, it.g["page_table"], it.g["seq_lens"], b["idx"].view(B, Hkv, -1),
                        it.params, b["tok"], b["fws"], stream)

    def attn(i):
        it, b = insts[i % R], bufs[i % R]
        sel = b["tok"] if c2f else b["idx"].view(B, Hkv, -1)
        L.lsa_sparse_decode(it.g["q"], it.cache, it.g["page_table"], it.g["seq_lens"], sel, it.params, it.out,
                            it.lse, b["ws"], stream)

    stages = [("score", score), ("topk", topk)] + ([("fine", fine)] if c2f else []) + [("attention", attn)]
    out = {}
    with torch.cuda.stream(stream):
        for i in range(R):
            for _, fn in stages:
                fn(i)
        stream.synchronize()
        for name, fn in stages:
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
        # the opt-in approximate top-k on the same score rows (stochastic
        # early exit): its time, and its recall of the exact selection
        def topk_approx(i):
            b = bufs[i % R]
            L.lsa_topk_approx(b["scores"], None, b["idx"].shape[1], 7 + i, b["idx"], stream)

        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(reps):
                topk_approx(i)
        gr.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gr.replay()
        e1.record(stream)
        stream.synchronize()
        approx_ms = e0.elapsed_time(e1) / reps
        recall, mass = topk_recall(bufs, topk, topk_approx, stream)
        # tie-heavy rows (the scores' signs: two values, the boundary bucket
        # crowded), where the exact selection needs its bisection
        for b in bufs:
            sc = b["scores"]
            b["scores"] = torch.where(torch.isneginf(sc), sc, torch.sign(sc))
        tie_exact = graph_ms(topk, reps, stream)
        tie_approx = graph_ms(topk_approx, reps, stream)
        tie_recall, tie_mass = topk_recall(bufs, topk, topk_approx, stream)
    out["_topk_approx"] = {"rows": int(bufs[0]["scores"].shape[0]), "cols": int(bufs[0]["scores"].shape[1]),
                           "k": int(bufs[0]["idx"].shape[1]), "exact_us": round(out["topk"] * 1e3, 2),
                           "approx_us": round(approx_ms * 1e3, 2),
                           "speedup": round(out["topk"] / max(approx_ms, 1e-9), 3),
                           "recall": round(recall, 5), "score_mass": round(mass, 6),
                           "tie_heavy": {"exact_us": round(tie_exact * 1e3, 2), "approx_us": round(tie_approx * 1e3, 2),
                                         "speedup": round(tie_exact / max(tie_approx, 1e-9), 3),
                                         "recall": round(tie_recall, 5), "score_mass": round(tie_mass, 6),
                                         "rows": "sign of the step's scores (-inf kept)"},
                           "note": "lsa_topk vs lsa_topk_approx on the step's score rows, each a CUDA graph "
                                   "rotating over the instances; recall = exact selections kept"}
    return out


def graph_ms(fn, reps: int, stream) -> float:
    """Device time of one call of fn(i), from a CUDA graph of reps calls."""
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
    return e0.elapsed_time(e1) / reps


def topk_recall(bufs, topk, topk_approx, stream):
    """(fraction of the exact top-k selections the approximate one keeps,
    the approximate selection's score mass over the exact one's): equal
    scores make the first low and leave the second at 1."""
    hit = tot = 0
    mass_a = mass_e = 0.0
    for i in range(len(bufs)):
        b = bufs[i]
        topk(i)
        exact = b["idx"].clone()
        topk_approx(i)
        stream.synchronize()
        ex, ap = exact.cpu().numpy(), b["idx"].cpu().numpy()
        sc = b["scores"].double().cpu().numpy()
        for r in range(ex.shape[0]):
            er, ar = ex[r][ex[r] >= 0], ap[r][ap[r] >= 0]
            hit += len(set(er.tolist()) & set(ar.tolist()))
            tot += len(er)
            base = sc[r][er].min() if len(er) else 0.0     # shift so the masses compare positive parts
            mass_e += float((sc[r][er] - base).sum())
            mass_a += float((sc[r][ar] - base).sum())
    return hit / max(tot, 1), (mass_a / mass_e if mass_e > 0 else 1.0)


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
    mem0 = torch.cuda.memory_allocated(dev)
    first = Instance(w, 0, dev)
    inst_bytes = max(torch.cuda.memory_allocated(dev) - mem0, 1)
    step_bytes = algorithmic_bytes(w, first.g["lens"])["total"]
    R = max(2, int(np.ceil(4 * L2_BYTES / max(step_bytes, 1))))
    # at most 16 instances and 96 GB of them (the small-step workloads touch
    # a few tens of MB of a cache of a GB or more per step)
    R = min(R, 16, max(2, int(96e9 // inst_bytes))) if args.instances <= 0 else args.instances
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

    pq_tokens = 0
    if w.pq_candidates > 0:
        # encoded candidate tokens of the first instance (every instance has the same lengths)
        for Lr in first.g["lens"]:
            se = min(w.sink, Lr)
            rs = max(Lr - w.recent, se)
            pq_tokens += sum(w.block_size for j in range(Lr // w.block_size)
                             if j * w.block_size >= se and (j + 1) * w.block_size <= rs)
    return dict(ms=ms, step_bytes=step_bytes, acc=acc, R=R, clocks=clocks, stages=st, e2e=e2e,
                kernels=kernels_per_step(insts[0]), w=w, pq_tokens=pq_tokens)


def _packed(tensors, pinned: bool, dev=None):
    """One uint8 buffer holding the tensors back to back at 16-byte aligned
    offsets (pinned host memory, or device memory when dev is given), and
    views of it shaped like each tensor."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += -(-t.numel() * t.element_size() // 16) * 16
    buf = (torch.empty(n, dtype=torch.uint8).pin_memory() if pinned
           else torch.empty(n, dtype=torch.uint8, device=dev))
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def e2e_leg(insts, args, stream):
    """The same step through the public call with HOST buffers: every step
    copies its q, page table and lengths from pinned host memory to the
    device, runs lsa_decode_step, and copies out and lse back to pinned host
    memory.  A caller's inputs of one step sit in one pinned staging buffer
    (q, page table, lengths at 16-byte aligned offsets) and its results in
    another, so that a step is one copy in and one copy out.  The copies and
    the call are captured in CUDA graphs of `chunk` steps rotating over the
    instances (as the device-side timing does), so that the number is the
    library's cost plus the copies, not Python's.  Before timing, each
    instance's results through this path are checked to equal, bit for bit,
    the device-resident step's."""
    R = len(insts)
    host = []
    for it in insts:
        g = it.g
        hin, (hq, hpt, hl) = _packed([g["q"], g["page_table"], g["seq_lens"]], pinned=True)
        hq.copy_(g["q"].cpu())
        hpt.copy_(g["page_table"].cpu())
        hl.copy_(g["seq_lens"].cpu())
        din, (dq, dpt, dl) = _packed([g["q"], g["page_table"], g["seq_lens"]], pinned=False, dev=g["q"].device)
        dout, (do, dlse) = _packed([it.out, it.lse], pinned=False, dev=g["q"].device)
        hout, (ho, hlse) = _packed([it.out, it.lse], pinned=True)
        host.append(dict(hin=hin, din=din, dq=dq, dpt=dpt, dl=dl, dout=dout, do=do, dlse=dlse,
                         hout=hout, ho=ho, hlse=hlse))

    def one(i):
        it, h = insts[i % R], host[i % R]
        h["din"].copy_(h["hin"], non_blocking=True)
        it.step(h["dq"], h["dpt"], h["dl"], stream, out=h["do"], lse=h["dlse"])
        h["hout"].copy_(h["dout"], non_blocking=True)

    chunk = R * max(1, 32 // R)
    n = max(chunk, min(args.steps, 4000) // chunk * chunk)
    with torch.cuda.stream(stream):
        for i in range(R):
            insts[i].step(stream=stream)
            one(i)
        stream.synchronize()
        for it, h in zip(insts, host):
            if not (torch.equal(h["ho"].view(torch.int16), it.out.cpu().view(torch.int16))
                    and torch.equal(h["hlse"], it.lse.cpu())):
                raise RuntimeError("the host-buffer step differs from the device-resident step")
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(chunk):
                one(i)
        gr.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n // chunk):
            gr.replay()
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / n
    h = host[0]
    return dict(ms_per_step=ms, h2d=h["hin"].numel(), d2h=h["hout"].numel(), steps=n)


# ---------------------------------------------------------------- CPU oracle

def cpu_model() -> str:
    """The host CPU's model name; on Arm, the implementer and part numbers
    from /proc/cpuinfo with the name of the few known parts."""
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
    except OSError:
        return "unknown"
    for ln in txt.splitlines():
        if ln.startswith("model name"):
            return ln.split(":", 1)[1].strip()
    fields = {}
    for ln in txt.splitlines():
        if ":" in ln:
            k, v = ln.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    parts = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
             ("0x41", "0xd0c"): "Arm Neoverse N1", ("0x41", "0xd49"): "Arm Neoverse N2"}
    imp, part = fields.get("CPU implementer"), fields.get("CPU part")
    if part:
        return parts.get((imp, part), f"implementer {imp} part {part}")
    return "unknown"


def cpu_baseline(w, budget_s: float = 12.0):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload: whole requests (every KV head of each), as many as it takes to
    give every core a (request, KV head) unit where the batch allows, with
    the summaries precomputed by the oracle (they are built once per block,
    outside the step).  Timed with OpenMP over all cores and single-threaded;
    calls/s = 1 / (B x time per request)."""
    import oracle
    cores = os.cpu_count() or 1
    nreq = min(w.batch, max(1, -(-cores // w.num_kv_heads)))
    sw = w.replace(batch=nreq, seq_lens=None if w.seq_lens is None else w.seq_lens[:nreq])
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    inp = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in make_inputs(sw, gen).items()}
    c = oracle.Cache(inp["k_cache"], None if w.v_aliased else inp["v_cache"], dv=w.dv if w.v_aliased else None)
    kw = dict(num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink, recent=w.recent,
              scale=w.softmax_scale)
    if w.pq_candidates > 0:
        ic = oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])
        kw.update(index_cache=ic, c2f_tokens=w.c2f_tokens, fine_weights=inp["fine_weights"],
                  pq_candidates=w.pq_candidates, pq_codes=inp["pq_codes"], pq_codebook=inp["pq_codebook"],
                  pq_hit=inp["pq_hit"])
        summ = None
    elif w.c2f_candidates > 0:
        ic = oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])
        isumm, _ = oracle.summaries(ic, inp["page_table"], inp["seq_lens"], use_index_keys=True)
        kw.update(index_cache=ic, index_summ=isumm, c2f_candidates=w.c2f_candidates, c2f_tokens=w.c2f_tokens,
                  fine_weights=inp.get("fine_weights"))
        summ = None
    elif w.summary_kind == 1:
        summ, _ = oracle.quest_summaries(c, inp["page_table"], inp["seq_lens"])
        kw.update(summary_kind=1)
    else:
        summ, _ = oracle.summaries(c, inp["page_table"], inp["seq_lens"])

    def timed(nthreads, budget):
        n, t0 = 0, time.time()
        while True:
            oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], summ=summ, nthreads=nthreads, **kw)
            n += 1
            if time.time() - t0 > budget or n >= 5000:
                break
        return (time.time() - t0) / n / nreq, n   # seconds per request

    units = nreq * w.num_kv_heads
    used = min(cores, units)
    per_req, n_all = timed(cores, budget_s)
    per_req1, n_one = timed(1, budget_s / 2)
    return {"value": round(1.0 / (per_req * w.batch), 3), "unit": "calls/s", "cores": used, "kind": "oracle",
            "nproc": cores, "cpu_model": cpu_model(),
            "single_thread": {"value": round(1.0 / (per_req1 * w.batch), 4), "unit": "calls/s", "cores": 1},
            "sample": f"{n_all} run(s) ({n_one} single-threaded) of {nreq} of {w.batch} requests with all "
                      f"{w.num_kv_heads} KV heads each ({units} (request, KV head) units, OpenMP over them on "
                      f"{used} of {cores} cores), fp64 oracle, summaries precomputed; "
                      f"calls/s = 1 / ({w.batch} x time per request)"}


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
    st = dict(res["stages"])
    approx = st.pop("_topk_approx", None)
    acc = res["acc"]
    # algorithmic bytes of each stage: the score reads the candidate
    # summaries, page table and q; the fine pass the candidates' FP8 keys and
    # scales; attention the selected and forced K/V, q and the output; top-k
    # moves no algorithmic bytes (its input and output are intermediates)
    stage_bytes = {"score": acc["summaries"] + acc["page_table"] + acc["q_out"] // 2, "topk": 0,
                   "fine": acc["fine"], "attention": acc["kv"] + acc["q_out"]}
    if st and w.pq_candidates > 0:
        # four launches: coarse scores and bucket counts, the selection
        # cluster kernel, attention; the selection's time is the step's
        # minus the coarse scores' and attention's
        kernel_ms = {"k_pq_scores": st["pq_scores"], "attention": st["attention"],
                     "k_pq_hist + k_pq_select": max(ms_step - st["pq_scores"] - st["attention"], 1e-9)}
        kbytes = {"k_pq_scores": stage_bytes["score"], "attention": stage_bytes["attention"],
                  "k_pq_hist + k_pq_select": acc["fine"]}
    elif st and selects_in_attention(w):
        # the step is two launches: the score kernel and the attention kernel
        # that also selects the blocks; the latter's time is the step's time
        # minus the score kernel's (both CUDA-event timings)
        sk = "k_score_quest" if w.summary_kind == 1 else "k_score"
        kernel_ms = {sk: st["score"], "k_attn_flat (selects)": max(ms_step - st["score"], 1e-9)}
        kbytes = {sk: stage_bytes["score"], "k_attn_flat (selects)": stage_bytes["attention"]}
    elif st and w.c2f_candidates > 0 and res["kernels"] == 3:
        # coarse scores, the cluster kernel (coarse top-C, FP8 rescoring,
        # token top-k), attention; the cluster kernel's time is the step's
        # minus the other two
        kernel_ms = {"k_score": st["score"], "k_c2f_fine": max(ms_step - st["score"] - st["attention"], 1e-9),
                     "k_sparse_attn_umma": st["attention"]}
        kbytes = {"k_score": stage_bytes["score"], "k_c2f_fine": stage_bytes["fine"],
                  "k_sparse_attn_umma": stage_bytes["attention"]}
    else:
        # one kernel per stage (scores, top-k, attention): each stage's
        # entry point launches the step's own kernel for it
        names = {"score": "k_score_quest" if w.summary_kind == 1 else "k_score",
                 "topk": "k_topk", "attention": "k_sparse_attn_umma" if w.num_q_heads // w.num_kv_heads == 64
                 else "attention"}
        kernel_ms = {names.get(k, k): v for k, v in st.items()}
        kbytes = {names.get(k, k): v for k, v in stage_bytes.items()}
    # the dominant kernel: the longest stage that moves algorithmic bytes
    moving = {k: v for k, v in kernel_ms.items() if kbytes.get(k, 0) > 0}
    dominant = max(moving, key=moving.get)
    if dominant == "k_pq_scores":
        # a dense contraction: every encoded candidate token's 64 x 128 dots
        flops = 2.0 * w.num_q_heads * w.dk * res["pq_tokens"]
        tpeak, tkind = peaks("tensor")
        ach = flops / (kernel_ms[dominant] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dominant, "achieved": round(ach, 1), "peak": tpeak, "unit": "TFLOP/s",
                "frac": round(ach / tpeak, 4), "peak_kind": tkind, "duration_us": round(kernel_ms[dominant] * 1e3, 2),
                "algorithmic_flops": flops, "algorithmic_bytes": kbytes[dominant],
                "hbm_frac": round(kbytes[dominant] / (kernel_ms[dominant] / 1e3) / 1e9 / peak, 4),
                "timing": "CUDA graph of the stage's entry point",
                "traffic": NCU_TRAFFIC.get((w.name, dominant))}
    else:
        ach = kbytes[dominant] / (kernel_ms[dominant] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_kind": peak_kind,
                "duration_us": round(kernel_ms[dominant] * 1e3, 2),
                "algorithmic_bytes": kbytes[dominant],
                "timing": ("step minus score kernel" if dominant.startswith("k_attn_flat")
                           else "step minus the other kernels" if dominant.startswith(("k_pq_hist", "k_c2f_fine"))
                           else "CUDA graph of the stage's entry point"),
                "traffic": NCU_TRAFFIC.get((w.name, dominant))}
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
                   "l2": (f"cold: {res['R']} rotating instances, " if res['R'] * res['step_bytes'] >= 2 * L2_BYTES
                          else f"NOT cold (profiling setting): {res['R']} instance(s), ")
                         + f"{res['R'] * res['step_bytes'] / 2**20:.0f} MiB touched per rotation vs 129 MB L2"},
        "tokens_per_s": round(calls * w.batch, 1),
        "step": {"algorithmic_bytes": res["step_bytes"], "bytes_split": acc, "gbs": round(gbs, 1),
                 "frac_of_peak": round(gbs / peak, 4), "frac_of_8tbs": round(gbs / 8000.0, 4)},
        "stages_ms": {k: round(v, 5) for k, v in st.items()},
        "kernels_ms": {k: round(v, 5) for k, v in kernel_ms.items()},
        "topk_approx": approx,
        "roofline": roof,
        "cpu_baseline": cb,
        "e2e": {"value": round(1e3 / e2e["ms_per_step"] * world, 1), "unit": "calls/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e["ms_per_step"], 5),
                "note": "lsa_decode_step on host inputs: each step copies one pinned staging buffer "
                        "(q, page table, lengths) in and one (out, lse) back, the copies and the call "
                        "captured in CUDA graphs; results checked equal to the device-resident step's"},
        "gpu_launches": res["kernels"] * args.steps,
        "clocks": res["clocks"],
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
