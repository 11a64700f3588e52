"""Shared helpers of the GPU parity tests: run the library through its C-ABI
binding, run the oracle on the same seeded inputs, and compare.

Tolerances
  selection: bit-exact against the oracle, except where the oracle's own
    fp64 scores put two blocks closer than the fp32 rounding bound of the
    GPU scorer at the selection boundary (an "epsilon tie": both choices are
    correct to within rounding); such rows are counted, their selection is
    checked to lie inside the tie band, and their attention is checked with
    the oracle run on that selection.
  attention: |o - o_ref| <= 2e-2 + 1e-2 * |o_ref| element-wise (bf16 inputs,
    fp32 accumulation); lse: |l - l_ref| <= 1e-3 + 1e-3 * |l_ref|.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import sparse_attention_decode_block_gb300 as L
from workloads import Workload

ATOL, RTOL = 2e-2, 1e-2
LSE_ATOL, LSE_RTOL = 1e-3, 1e-3


def to_dev(inp: dict, dev="cuda") -> dict:
    """Move an instance to the device, keeping a latent cache's V a view of K."""
    out = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    k, v = inp["k_cache"], inp["v_cache"]
    if v.data_ptr() == k.data_ptr():
        out["v_cache"] = out["k_cache"][..., : v.shape[-1]]
    return out


def f64(bits) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def subset(inp: dict, reqs) -> dict:
    """CPU copy of the requests `reqs` with their pages gathered into a
    compact cache (page table remapped); values are unchanged."""
    pt = inp["page_table"]
    rows = pt[list(reqs)]
    used = rows[rows >= 0].long()
    uniq, inv = torch.unique(used, return_inverse=True)
    new_rows = torch.full_like(rows, -1)
    new_rows[rows >= 0] = inv.to(torch.int32)
    out = dict(q=inp["q"][list(reqs)].cpu(), page_table=new_rows.cpu(),
               seq_lens=inp["seq_lens"][list(reqs)].cpu(), lens=[inp["lens"][r] for r in reqs],
               num_pages=int(uniq.numel()), max_blocks=inp["max_blocks"])
    out["k_cache"] = inp["k_cache"][uniq.to(inp["k_cache"].device)].cpu()
    if inp["v_cache"].data_ptr() == inp["k_cache"].data_ptr():
        out["v_cache"] = out["k_cache"][..., : inp["v_cache"].shape[-1]]
    else:
        out["v_cache"] = inp["v_cache"][uniq.to(inp["v_cache"].device)].cpu()
    if "idx_keys" in inp:
        out["idx_keys"] = inp["idx_keys"][uniq.to(inp["idx_keys"].device)].cpu()
        out["idx_scale"] = inp["idx_scale"][uniq.to(inp["idx_scale"].device)].cpu()
    if "fine_weights" in inp:
        out["fine_weights"] = inp["fine_weights"][list(reqs)].cpu()
    return out


def oracle_cache(inp: dict) -> oracle.Cache:
    return oracle.Cache(inp["k_cache"], inp["v_cache"])


def oracle_index(inp: dict) -> oracle.Cache:
    return oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])


def oracle_decode(w: Workload, cpu: dict, nthreads: int = os.cpu_count() or 1, **over):
    kw = dict(num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink, recent=w.recent,
              scale=w.softmax_scale, nthreads=nthreads)
    if w.c2f_candidates > 0:
        ic = oracle_index(cpu)
        isumm, _ = oracle.summaries(ic, cpu["page_table"], cpu["seq_lens"], use_index_keys=True)
        kw.update(index_cache=ic, index_summ=isumm, c2f_candidates=w.c2f_candidates,
                  c2f_tokens=w.c2f_tokens, fine_weights=cpu.get("fine_weights"))
    kw.update(over)
    c = oracle_cache(cpu)
    summ = None
    if w.c2f_candidates == 0:
        if w.summary_kind == 1:
            summ, _ = oracle.quest_summaries(c, cpu["page_table"], cpu["seq_lens"])
            kw["summary_kind"] = 1
        else:
            summ, _ = oracle.summaries(c, cpu["page_table"], cpu["seq_lens"])
    return oracle.decode(cpu["q"], c, cpu["page_table"], cpu["seq_lens"], summ=summ, **kw)


# ---------------------------------------------------------------- GPU side

class GpuStep:
    """Device buffers and descriptors for one workload instance."""

    def __init__(self, w: Workload, g: dict, num_splits: int = 0):
        self.w, self.g = w, g
        dev = g["q"].device
        self.cache = L.make_cache(g["k_cache"], g["v_cache"])
        self.icache = None
        B, Hkv = w.batch, w.num_kv_heads
        if w.pq_candidates > 0:
            self.icache = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
            self.summ = torch.zeros((1, 1, w.dk), dtype=torch.bfloat16, device=dev)   # not read
            nsel = w.c2f_tokens
        elif w.c2f_candidates > 0:
            self.icache = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
            self.summ = torch.zeros((g["num_pages"], Hkv, w.dk), dtype=torch.bfloat16, device=dev)
            L.lsa_build_summaries(self.icache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.c2f_tokens
        elif w.summary_kind == 1:
            self.summ = torch.zeros((g["num_pages"], Hkv, 2, w.dk), dtype=torch.bfloat16, device=dev)
            L.lsa_build_minmax_summaries(self.cache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.k_blocks
        else:
            self.summ = torch.zeros((g["num_pages"], Hkv, w.dk), dtype=torch.bfloat16, device=dev)
            L.lsa_build_summaries(self.cache, g["page_table"], g["seq_lens"], self.summ)
            nsel = w.k_blocks
        self.params = L.make_params(B, w.num_q_heads, g["max_blocks"], w.k_blocks, w.sink, w.recent,
                                    w.softmax_scale, w.c2f_candidates, w.c2f_tokens, num_splits,
                                    summary_kind=w.summary_kind, fine_head_weights=g.get("fine_weights"),
                                    pq_candidates=w.pq_candidates, pq_codes=g.get("pq_codes"),
                                    pq_codebook=g.get("pq_codebook"), pq_hit=g.get("pq_hit"))
        ws = L.lsa_decode_step_workspace_size(self.cache, self.params)
        assert ws > 0 or w.batch == 0 or True
        self.ws = torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev)
        self.idx = torch.full((B, Hkv, max(nsel, 1)), -7, dtype=torch.int32, device=dev)
        self.out = torch.empty((B, w.num_q_heads, w.dv), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, w.num_q_heads), dtype=torch.float32, device=dev)

    def run(self, stream=None):
        g = self.g
        L.lsa_decode_step(g["q"], self.cache, self.summ, self.icache, g["page_table"], g["seq_lens"],
                          self.params, self.idx, self.out, self.lse, self.ws, stream)


def check_status_clean():
    torch.cuda.synchronize()
    code, flags = L.lsa_get_device_status(clear=True)
    assert code == 0, f"device status {L.lsa_status_string(code)} flags={flags:#x}"


# ---------------------------------------------------------------- comparisons

def assert_attention_close(o_gpu: torch.Tensor, o_ref_bits: np.ndarray, what: str = ""):
    o = o_gpu.detach().float().cpu().numpy().astype(np.float64)
    r = f64(o_ref_bits)
    err = np.abs(o - r)
    ok = err <= ATOL + RTOL * np.abs(r)
    if not ok.all():
        i = np.unravel_index(np.argmax(err - (ATOL + RTOL * np.abs(r))), err.shape)
        raise AssertionError(f"{what}: {(~ok).sum()} elements out of tolerance; worst at {i}: "
                             f"gpu={o[i]} ref={r[i]} (max abs err {err.max():.3g})")
    big = np.abs(r) > 1e-3
    rel = (err[big] / np.abs(r[big])).max() if big.any() else 0.0
    return float(err.max()), float(rel)


def assert_lse_close(lse_gpu: torch.Tensor, lse_ref: np.ndarray, what: str = ""):
    l = lse_gpu.detach().cpu().numpy().astype(np.float64)
    both_inf = np.isneginf(l) & np.isneginf(lse_ref)
    with np.errstate(invalid="ignore"):   # -inf - -inf where both are empty; masked below
        d = np.where(both_inf, 0.0, np.abs(l - lse_ref))
    lim = LSE_ATOL + LSE_RTOL * np.where(both_inf, 0.0, np.abs(lse_ref))
    assert np.all(d <= lim), f"{what}: lse max err {np.nanmax(d):.3g}"


def quest_score_bound(q_bits: np.ndarray, mx_f64: np.ndarray, mn_f64: np.ndarray, dk: int) -> np.ndarray:
    """Upper bound on |fp32 GPU Quest score - exact score| per block: each
    head's sum of dk rounded products (each max(q M, q m) exact up to one
    product rounding) is off by at most 2 dk 2^-24 sum_i |q_i| max(|M_i|,
    |m_i|); the maximum over heads is exact.  Twice that, for safety."""
    q = np.abs(f64(q_bits))                        # [G, dk]
    a = np.maximum(np.abs(mx_f64), np.abs(mn_f64))   # [nblocks, dk]
    return 4 * dk * 2.0 ** -24 * (a @ q.T).max(axis=1)


def score_bound(q_bits: np.ndarray, summ_f64: np.ndarray, G: int, dk: int) -> np.ndarray:
    """Upper bound on |fp32 GPU score - exact score| per block: the group's
    queries are summed in fp32 (G terms) and dotted with the summary in fp32
    (dk terms); each rounding is at most 2^-24 relative, so the error is at
    most (G + dk) * 2^-23 * sum_i sum_g |q_gi| |S_i| (twice the first-order
    bound, for safety)."""
    qa = np.abs(f64(q_bits)).sum(axis=0)          # [dk]
    return (G + dk) * 2.0 ** -23 * (np.abs(summ_f64) @ qa)


def compare_selection(sel_gpu: np.ndarray, sel_ref: np.ndarray, scores_ref: np.ndarray, tau: np.ndarray):
    """Returns 'equal' or 'tie' (valid alternative within the tie band), or
    raises.  scores_ref: oracle fp64 scores of the row (-inf = non-candidate);
    tau: per-column score error bound."""
    if np.array_equal(sel_gpu, sel_ref):
        return "equal"
    a = set(sel_gpu[sel_gpu >= 0].tolist())
    b = set(sel_ref[sel_ref >= 0].tolist())
    assert len(a) == len(b), f"selection sizes differ: {sorted(a)} vs {sorted(b)}"
    cand = np.flatnonzero(np.isfinite(scores_ref))
    order = cand[np.lexsort((cand, -scores_ref[cand]))]
    kth = scores_ref[order[len(b) - 1]]
    band = 2 * tau.max()
    for j in a.symmetric_difference(b):
        assert np.isfinite(scores_ref[j]), f"non-candidate {j} selected"
        assert abs(scores_ref[j] - kth) <= band, (
            f"selection differs outside the rounding band: block {j} score {scores_ref[j]} vs k-th {kth} "
            f"(band {band:.3g})")
    return "tie"
