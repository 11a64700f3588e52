"""Seeded synthetic inputs for the block-sparse decode step.

This module is shared by the tests, the bench and the smoke check.  It draws
queries, paged K/V caches, page tables, lengths and (for the coarse-to-fine
workload) FP8 index keys, and nothing else: it holds none of the method's
arithmetic (no summaries, scores, selection or attention).

Workload shapes follow the pages' workloads:
  * block top-k with mean-key summaries, 16-token blocks, paged cache
    (Vortex blog post, "Block top-k attention", Figure 1 and Figure 2);
  * 8B-class GQA heads (32 query / 8 KV heads, d=128) at 16 x 32K
    (Vortex blog post, "Why Long Generations Are Expensive");
  * a 64-head FP8 indexer with a 2K->k coarse-to-fine search (LeanSparse,
    Section 5 "Coarse-to-fine decode indexing");
  * an MLA-shaped latent cache, 576-d keys with the first 512 dims as values
    (Vortex blog post, "Designing for a new architecture").

Draw order for every workload, from one ``torch.Generator`` seeded with the
workload's seed: lengths -> page permutation -> q -> K -> V -> per-(request,
KV head) shifted blocks -> FP8 index keys -> indexer head weights.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

__all__ = ["Workload", "WORKLOADS", "small_workloads", "make_inputs", "get"]


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    dk: int
    dv: int
    block_size: int
    # Either a fixed context length, or a (lo, hi) inclusive uniform range.
    seq_len: int = 0
    seq_len_range: Optional[tuple] = None
    # Explicit lengths override both (used by edge-case tests).
    seq_lens: Optional[tuple] = None
    sink: int = 0
    recent: int = 0
    k_blocks: int = 0
    scale: float = 0.0          # 0 -> 1/sqrt(dk)
    contiguous_pages: bool = False
    shift_frac: float = 0.0     # fraction of each request's blocks shifted per KV head
    shift_sigma: float = 0.0    # shift magnitude along the group's mean-query direction
    v_aliased: bool = False     # V = K[..., :dv] (latent cache)
    c2f_candidates: int = 0
    c2f_tokens: int = 0
    summary_kind: int = 0       # 0: mean keys; 1: Quest's max and min keys
    fine_weighted: bool = False  # coarse-to-fine: weighted-ReLU fine score with drawn head weights
    pq_candidates: int = 0      # PQ32 coarse-to-fine: token candidates of the coarse pass
    pq_hit_frac: float = 0.5    # ... fraction of tokens whose original index key is cached
    pq_noise: float = 0.35      # ... key = its codes' centroids + N(0, pq_noise^2) per dim
    extra_pages: int = 0        # unused pages appended to the pool
    description: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / math.sqrt(self.dk)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        name="tiny", seed=0, batch=1, num_q_heads=4, num_kv_heads=1, dk=64, dv=64,
        block_size=16, seq_len=1024, sink=16, recent=16, k_blocks=6, scale=1.0 / 8.0,
        contiguous_pages=True,
        description="B=1, 4q/1kv, d=64, L=1024, block 16, top-8 blocks incl. first and last"),
    "b16_32k": Workload(
        name="b16_32k", seed=1, batch=16, num_q_heads=32, num_kv_heads=8, dk=128, dv=128,
        block_size=16, seq_len=32768, sink=16, recent=16, k_blocks=62,
        shift_frac=0.05, shift_sigma=2.0,
        description="B=16, 32q/8kv, d=128, L=32768, block 16, top-64 blocks incl. first and "
                    "last, 5% of blocks shifted +2 sigma along the group's mean query"),
    "b16_32k_quest": Workload(
        name="b16_32k_quest", seed=1, batch=16, num_q_heads=32, num_kv_heads=8, dk=128, dv=128,
        block_size=16, seq_len=32768, sink=16, recent=16, k_blocks=62,
        shift_frac=0.05, shift_sigma=2.0, summary_kind=1,
        description="the B=16 x 32K workload with Quest's min/max key summaries and bound scores"),
    "ragged": Workload(
        name="ragged", seed=2, batch=64, num_q_heads=32, num_kv_heads=8, dk=128, dv=128,
        block_size=64, seq_len_range=(4096, 131072), sink=4, recent=512, k_blocks=23,
        description="64 requests, L ~ U{4K..128K}, 32q/8kv, d=128, page 64, token budget "
                    "2048 incl. 4 sink + 512 recent"),
    "c2f": Workload(
        name="c2f", seed=3, batch=4, num_q_heads=64, num_kv_heads=1, dk=128, dv=128,
        block_size=64, seq_len=524288, sink=0, recent=0, k_blocks=0,
        c2f_candidates=256, c2f_tokens=2048,
        description="B=4, L=512K, block 64, coarse top-256 blocks, fine FP8 top-2048 tokens, "
                    "64q/1kv, d=128"),
    "c2f_wrelu": Workload(
        name="c2f_wrelu", seed=3, batch=4, num_q_heads=64, num_kv_heads=1, dk=128, dv=128,
        block_size=64, seq_len=524288, sink=0, recent=0, k_blocks=0,
        c2f_candidates=256, c2f_tokens=2048, fine_weighted=True,
        description="the coarse-to-fine workload with the weighted-ReLU indexer fine score "
                    "(head weights ~ U[0, 1))"),
    "c2f_pq": Workload(
        name="c2f_pq", seed=5, batch=4, num_q_heads=64, num_kv_heads=1, dk=128, dv=128,
        block_size=64, seq_len=524288, sink=0, recent=0, k_blocks=0,
        c2f_tokens=2048, pq_candidates=8192,
        description="B=4, L=512K, 64-head FP8 indexer with PQ32 codes: coarse top-8192 tokens by the "
                    "PQ weighted-ReLU score, miss filter (half the tokens' keys cached), exact "
                    "weighted-ReLU top-2048 tokens, 64q/1kv d=128"),
    "mla": Workload(
        name="mla", seed=4, batch=4, num_q_heads=64, num_kv_heads=1, dk=576, dv=512,
        block_size=64, seq_len=1048576, sink=4, recent=128, k_blocks=29, v_aliased=True,
        description="B=4, L=1M, 64q/1 latent kv, dk=576/dv=512 (V aliased), block 64, "
                    "token budget 2048 incl. 4 sink + 128 recent"),
}


def small_workloads() -> dict:
    """Scaled-down versions of every workload: same structure (heads, dims,
    block size, forced ranges, shift, FP8 index, aliasing), sizes that the
    oracle finishes in seconds, with ragged tails (lengths not multiples of
    the block size) and several tiles per row."""
    W = WORKLOADS
    return {
        "tiny": W["tiny"],
        "b16_small": W["b16_32k"].replace(
            name="b16_small", seed=11, batch=3, seq_len=0, seq_lens=(4096, 3001, 777)),
        "ragged_small": W["ragged"].replace(
            name="ragged_small", seed=12, batch=5, seq_len_range=(100, 9000)),
        "c2f_small": W["c2f"].replace(
            name="c2f_small", seed=13, batch=2, seq_len=0, seq_lens=(16384 + 37, 9000),
            c2f_candidates=32, c2f_tokens=512, recent=37),
        "mla_small": W["mla"].replace(
            name="mla_small", seed=14, batch=2, seq_len=0, seq_lens=(20000, 6001)),
        "c2f_wrelu_small": W["c2f_wrelu"].replace(
            name="c2f_wrelu_small", seed=16, batch=2, seq_len=0, seq_lens=(16384 + 37, 9000),
            c2f_candidates=32, c2f_tokens=512, recent=37),
        "c2f_pq_small": W["c2f_pq"].replace(
            name="c2f_pq_small", seed=17, batch=2, seq_len=0, seq_lens=(16384 + 37, 9000),
            pq_candidates=1024, c2f_tokens=256, recent=37),
        "quest_small": W["b16_32k_quest"].replace(
            name="quest_small", seed=15, batch=3, seq_len=0, seq_lens=(4096, 3001, 777)),
    }


def get(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    sw = small_workloads()
    if name in sw:
        return sw[name]
    raise KeyError(name)


def _lengths(w: Workload, g: torch.Generator) -> list:
    if w.seq_lens is not None:
        assert len(w.seq_lens) == w.batch
        return [int(x) for x in w.seq_lens]
    if w.seq_len_range is not None:
        lo, hi = w.seq_len_range
        t = torch.randint(lo, hi + 1, (w.batch,), generator=g, device=g.device)
        return [int(x) for x in t.cpu().tolist()]
    return [w.seq_len] * w.batch


def make_inputs(w: Workload, device: str = "cpu", lens: Optional[Sequence[int]] = None) -> dict:
    """Draw one instance of workload ``w`` on ``device``.

    Returns a dict of tensors, all on ``device``:
      q          [B, Hq, dk] bf16
      k_cache    [P, Hkv, b, dk] bf16  (page, head, token-in-block, dim)
      v_cache    [P, Hkv, b, dv] bf16  (a view of k_cache[..., :dv] when aliased)
      page_table [B, max_blocks] int32, -1 past each request's last page
      seq_lens   [B] int32 (tokens in cache, the current step's token included)
      idx_keys   [P, Hkv, b, dk] uint8 (FP8 e4m3 bit patterns)   -- coarse-to-fine only
      idx_scale  [P, Hkv, b] fp32 per-token dequantisation scale -- coarse-to-fine only
    plus the python ints/lists ``lens``, ``num_pages``, ``max_blocks``.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    B, Hq, Hkv, b = w.batch, w.num_q_heads, w.num_kv_heads, w.block_size
    drawn = _lengths(w, g)
    if lens is None:
        lens = drawn
    lens = [int(x) for x in lens]
    nblk = [(L + b - 1) // b for L in lens]
    max_blocks = max(1, max(nblk) if nblk else 1)
    num_pages = sum(nblk) + w.extra_pages
    num_pages = max(num_pages, 1)

    # page permutation
    if w.contiguous_pages:
        perm = torch.arange(num_pages, dtype=torch.int64, device=dev)
    else:
        perm = torch.randperm(num_pages, generator=g, device=dev)
    pt = torch.full((B, max_blocks), -1, dtype=torch.int32, device=dev)
    off = 0
    for r in range(B):
        if nblk[r]:
            pt[r, : nblk[r]] = perm[off: off + nblk[r]].to(torch.int32)
        off += nblk[r]

    q = torch.randn((B, Hq, w.dk), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    k_cache = torch.randn((num_pages, Hkv, b, w.dk), generator=g, device=dev,
                          dtype=torch.float32).to(torch.bfloat16)
    if w.v_aliased:
        v_cache = k_cache[..., : w.dv]
    else:
        v_cache = torch.randn((num_pages, Hkv, b, w.dv), generator=g, device=dev,
                              dtype=torch.float32).to(torch.bfloat16)

    if w.shift_frac > 0 and w.shift_sigma != 0:
        G = w.group
        for r in range(B):
            nb = nblk[r]
            n_shift = int(round(w.shift_frac * nb))
            if n_shift == 0:
                continue
            for h in range(Hkv):
                u = q[r, h * G:(h + 1) * G].float().mean(dim=0)
                u = u / u.norm().clamp_min(1e-12)
                blocks = torch.randperm(nb, generator=g, device=dev)[:n_shift]
                pages = pt[r, blocks].long()
                blk = k_cache[pages, h].float() + (w.shift_sigma * u)
                k_cache[pages, h] = blk.to(torch.bfloat16)

    out = dict(q=q, k_cache=k_cache, v_cache=v_cache, page_table=pt,
               seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev),
               lens=lens, num_pages=num_pages, max_blocks=max_blocks)

    if w.pq_candidates > 0:
        # PQ32 index keys: a codebook of 256 centroids per 4-dim subspace,
        # a code per (token, subspace), the key its centroids plus noise
        cbk = torch.randn((32, 256, 4), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
        codes = torch.randint(0, 256, (num_pages, Hkv, b, 32), generator=g, device=dev, dtype=torch.int64)
        kk = cbk.float()[torch.arange(32, device=dev), codes].reshape(num_pages, Hkv, b, w.dk)
        kk += w.pq_noise * torch.randn((num_pages, Hkv, b, w.dk), generator=g, device=dev, dtype=torch.float32)
        out["pq_codebook"] = cbk.contiguous()
        out["pq_codes"] = codes.to(torch.uint8).contiguous()
    elif w.c2f_candidates > 0:
        kk = torch.randn((num_pages, Hkv, b, w.dk), generator=g, device=dev, dtype=torch.float32)
    if w.c2f_candidates > 0 or w.pq_candidates > 0:
        amax = kk.abs().amax(dim=-1).clamp_min(1e-30)
        scale = (amax / 448.0).to(torch.float32)
        k8 = (kk / scale.unsqueeze(-1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        out["idx_keys"] = k8.view(torch.uint8)
        out["idx_scale"] = scale.contiguous()
        if w.fine_weighted or w.pq_candidates > 0:
            # indexer head weights of the weighted-ReLU fine score
            out["fine_weights"] = torch.rand((B, Hq), generator=g, device=dev, dtype=torch.float32)
        if w.pq_candidates > 0:
            out["pq_hit"] = (torch.rand((num_pages, Hkv, b), generator=g, device=dev) < w.pq_hit_frac).to(torch.uint8)
    return out


def algorithmic_bytes(w: Workload, lens: Sequence[int]) -> dict:
    """Bytes one decode step must move at minimum: summaries of candidate
    blocks, forced + selected K/V, page-table entries read, q and out.

    The byte account follows the ByteCross page's decode-step read model
    (KV bytes = 2 * heads * head_dim * tokens * element size, Section 3.1,
    Eq. 4), applied to the entries a sparse step actually reads.
    """
    b, Hkv, Hq = w.block_size, w.num_kv_heads, w.num_q_heads
    summ = sel = fine = pt = 0
    for L in lens:
        nb_full = L // b
        sink_end = min(w.sink, L)
        rec_start = max(L - w.recent, sink_end)
        forced = sink_end + (L - rec_start)
        ncand = 0
        for j in range(nb_full):
            lo, hi = j * b, (j + 1) * b
            if not (lo < sink_end or hi > rec_start):
                ncand += 1
        nblk = (L + b - 1) // b
        pt += nblk * 4
        if w.pq_candidates > 0:
            # the PQ32 codes of every candidate token (32 bytes), the FP8
            # keys and scales of at most C candidates plus the tail, their
            # hit flags
            summ += ncand * b * Hkv * 32
            ntail = L - nb_full * b
            nfine = min(w.pq_candidates, ncand * b)
            fine += (nfine + ntail) * Hkv * (w.dk * 1 + 4) + nfine * Hkv
            ntok = forced + min(w.c2f_tokens, nfine + ntail)
        elif w.c2f_candidates > 0:
            summ += ncand * Hkv * w.dk * 2
            ncb = min(w.c2f_candidates, ncand)
            fine += ncb * b * Hkv * (w.dk * 1 + 4)
            ntok = forced + min(w.c2f_tokens, ncb * b)
        else:
            summ += ncand * Hkv * w.dk * 2 * (2 if w.summary_kind == 1 else 1)
            ntok = forced + min(w.k_blocks, ncand) * b
        kv_row = w.dk * 2 + (0 if w.v_aliased else w.dv * 2)
        sel += ntok * Hkv * kv_row
    qo = len(lens) * Hq * (w.dk * 2 + w.dv * 2)
    total = summ + sel + fine + pt + qo
    return dict(summaries=summ, kv=sel, fine=fine, page_table=pt, q_out=qo, total=total)
