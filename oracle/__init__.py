"""Python shim over the plain-C CPU oracle (``lsa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and
the bench's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or calls anything here, and nothing here imports the CUDA
library.  Inputs are host numpy arrays (bf16 as uint16 bit patterns, FP8 as
uint8 bit patterns) or CPU torch tensors; every result is computed in fp64 by
the C code from those inputs.

Parity status per function (what pins each one is listed in the tests):
  bf16_round, e4m3_decode, summaries, block_scores, topk, attend_tokens,
  lse_merge, decode (single stage and coarse-to-fine), dense -- all pinned.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lsa_oracle.c")
_LIB = os.path.join(_HERE, "liblsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math; OpenMP when the
    compiler supports it).  Returns the path of the shared library."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", _LIB + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


class _Cache(C.Structure):
    _fields_ = [("num_pages", C.c_int32), ("num_kv_heads", C.c_int32),
                ("block_size", C.c_int32), ("dk", C.c_int32), ("dv", C.c_int32),
                ("k", C.c_void_p), ("v", C.c_void_p), ("k8", C.c_void_p),
                ("k8_scale", C.c_void_p)]


class _Params(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_q_heads", C.c_int32), ("max_blocks", C.c_int32),
                ("k_blocks", C.c_int32), ("sink", C.c_int32), ("recent", C.c_int32),
                ("scale", C.c_double), ("c2f_candidates", C.c_int32),
                ("c2f_tokens", C.c_int32), ("summary_kind", C.c_int32), ("fine_weights", C.c_void_p),
                ("pq_candidates", C.c_int32), ("pq_codes", C.c_void_p), ("pq_codebook", C.c_void_p),
                ("pq_hit", C.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P, I = C.c_void_p, C.c_int32
            lib.orc_bf16_to_f64.argtypes = [C.c_uint16]
            lib.orc_bf16_to_f64.restype = C.c_double
            lib.orc_f64_to_bf16.argtypes = [C.c_double]
            lib.orc_f64_to_bf16.restype = C.c_uint16
            lib.orc_e4m3_to_f64.argtypes = [C.c_uint8]
            lib.orc_e4m3_to_f64.restype = C.c_double
            lib.orc_summaries.argtypes = [P, C.c_int, P, P, I, I, P, P]
            lib.orc_quest_summaries.argtypes = [P, P, P, I, I, P, P]
            lib.orc_block_scores.argtypes = [P, P, C.c_int, P, P, P, P, P]
            lib.orc_topk.argtypes = [P, I, I, P]
            lib.orc_pq_scores.argtypes = [P, P, P, P, C.c_int, C.c_int, C.c_int64, C.c_int64, P]
            lib.orc_pq_scores.restype = C.c_int
            lib.orc_pq_encode.argtypes = [P, P, C.c_int64, P, P]
            lib.orc_pq_encode.restype = C.c_int
            lib.orc_token_scores_wrelu.argtypes = [P, P, P, P, C.c_int, C.c_int, C.c_int64, P, P]
            lib.orc_token_scores_wrelu.restype = C.c_int
            lib.orc_miss_filter.argtypes = [P, P, C.c_int64, C.c_int64, P, P]
            lib.orc_miss_filter.restype = C.c_int
            lib.orc_pq_select.argtypes = [P, P, P, P, P, C.c_int, C.c_int, P, P, P, P]
            lib.orc_pq_select.restype = C.c_int
            lib.orc_splitmix64.argtypes = [C.c_uint64, C.c_uint64]
            lib.orc_splitmix64.restype = C.c_uint64
            lib.orc_topk_approx.argtypes = [P, I, I, I, C.c_uint64, C.c_int64, P]
            lib.orc_topk_approx.restype = C.c_int
            lib.orc_fine_scores.argtypes = [P, P, P, P, C.c_int, C.c_int, C.c_int64, P, P, P]
            lib.orc_decode.argtypes = [P, P, P, P, P, P, P, P, C.c_int, P, P, P, P]
            lib.orc_dense.argtypes = [P, P, P, P, P, P, P]
            lib.orc_attend_tokens.argtypes = [P, P, P, C.c_int64, P, C.c_int, C.c_double, P, P]
            lib.orc_lse_merge.argtypes = [C.c_int, C.c_int, P, P, P, P]
            lib.orc_attend_selection.argtypes = [P, P, P, P, P, P, I, C.c_int, P, P]
            lib.orc_lse_merge.restype = None
            for f in ("orc_summaries", "orc_quest_summaries", "orc_block_scores", "orc_topk", "orc_fine_scores",
                      "orc_decode", "orc_dense", "orc_attend_tokens", "orc_attend_selection"):
                getattr(lib, f).restype = C.c_int
            _lib = lib
    return _lib


_ERR = {1: "page id out of range", 2: "invalid argument", 3: "out of memory"}


def _check(rc: int):
    if rc != 0:
        raise RuntimeError(f"oracle error {rc}: {_ERR.get(rc, '?')}")


def _np(x, dtype) -> np.ndarray:
    """Host, C-contiguous numpy view/copy of a numpy array or torch tensor.
    bf16 tensors become uint16 bit patterns, fp8 tensors uint8 patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach()
            if t.device.type != "cpu":
                t = t.cpu()
            if t.dtype == torch.bfloat16:
                t = t.contiguous().view(torch.int16)
            elif t.dtype in (torch.float8_e4m3fn,):
                t = t.contiguous().view(torch.uint8)
            x = t.contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype != dtype:
        if dtype == np.uint16 and a.dtype == np.int16:
            a = a.view(np.uint16)
        else:
            a = a.astype(dtype)
    return a


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


class Cache:
    """Host copy of a paged cache: k [P, Hkv, b, dk] bf16, v [P, Hkv, b, dv]
    bf16 (V aliased on a latent cache is passed as the copy k[..., :dv]),
    optional FP8 index keys k8 [P, Hkv, b, dk] and scales [P, Hkv, b]."""

    def __init__(self, k, v=None, k8=None, k8_scale=None, dv: Optional[int] = None):
        self.k = _np(k, np.uint16) if k is not None else None
        if v is None and k is not None and dv is not None:
            v = self.k[..., :dv]
        self.v = _np(v, np.uint16) if v is not None else None
        self.k8 = _np(k8, np.uint8) if k8 is not None else None
        self.k8_scale = _np(k8_scale, np.float32) if k8_scale is not None else None
        ref = self.k if self.k is not None else self.k8
        P, H, b, dk = ref.shape
        self.shape = (P, H, b, dk)
        self.dv = self.v.shape[-1] if self.v is not None else dk
        self._c = _Cache(P, H, b, dk, self.dv, _p(self.k), _p(self.v), _p(self.k8),
                         _p(self.k8_scale))

    @property
    def ref(self):
        return C.byref(self._c)


def _params(batch, num_q_heads, max_blocks, k_blocks=0, sink=0, recent=0, scale=1.0,
            c2f_candidates=0, c2f_tokens=0, summary_kind=0, fine_weights=None,
            pq_candidates=0, pq_codes=None, pq_codebook=None, pq_hit=None):
    """fine_weights, pq_codes, pq_codebook, pq_hit: C-contiguous numpy arrays
    (kept alive by the caller) or None."""
    ptr = lambda a: None if a is None else a.ctypes.data
    return _Params(batch, num_q_heads, max_blocks, k_blocks, sink, recent, float(scale),
                   c2f_candidates, c2f_tokens, summary_kind, ptr(fine_weights),
                   pq_candidates, ptr(pq_codes), ptr(pq_codebook), ptr(pq_hit))


# ---------------------------------------------------------------- formats

def bf16_round(x: float) -> int:
    """double -> bf16 bit pattern, round to nearest even (one rounding)."""
    return int(_load().orc_f64_to_bf16(float(x)))


def bf16_value(bits: int) -> float:
    return float(_load().orc_bf16_to_f64(int(bits) & 0xFFFF))


def e4m3_decode(code: int) -> float:
    return float(_load().orc_e4m3_to_f64(int(code) & 0xFF))


# ---------------------------------------------------------------- steps

def summaries(cache: Cache, page_table, seq_lens, use_index_keys: bool = False):
    """bf16 mean-key summaries [P, Hkv, dk] (uint16 bits) of every full
    block the page tables reference, and the [P] mask of pages written."""
    lib = _load()
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    P, H, b, dk = cache.shape
    out = np.zeros((P, H, dk), dtype=np.uint16)
    valid = np.zeros((P,), dtype=np.uint8)
    _check(lib.orc_summaries(cache.ref, int(use_index_keys), _p(pt), _p(lens), pt.shape[0],
                             pt.shape[1], _p(out), _p(valid)))
    return out, valid.astype(bool)


def quest_summaries(cache: Cache, page_table, seq_lens):
    """Quest summaries [P, Hkv, 2, dk] (uint16 bf16 bits): the element-wise
    maximum then minimum of the keys of every full block the page tables
    reference, and the [P] mask of pages written."""
    lib = _load()
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    P, H, b, dk = cache.shape
    out = np.zeros((P, H, 2, dk), dtype=np.uint16)
    valid = np.zeros((P,), dtype=np.uint8)
    _check(lib.orc_quest_summaries(cache.ref, _p(pt), _p(lens), pt.shape[0], pt.shape[1], _p(out), _p(valid)))
    return out, valid.astype(bool)


def block_scores(q, cache: Cache, summ, page_table, seq_lens, num_q_heads, sink, recent,
                 use_index_keys: bool = False, summary_kind: int = 0):
    """fp64 block scores [B, Hkv, max_blocks]; -inf for non-candidates.
    ``summ`` = oracle summaries (uint16 bits; Quest summaries when
    summary_kind = 1) or None to compute from keys."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    s = None if summ is None else _np(summ, np.uint16)
    B, maxb = pt.shape
    prm = _params(B, num_q_heads, maxb, 0, sink, recent, summary_kind=summary_kind)
    out = np.empty((B, cache.shape[1], maxb), dtype=np.float64)
    _check(lib.orc_block_scores(_p(qa), cache.ref, int(use_index_keys), _p(s), _p(pt), _p(lens),
                                C.byref(prm), _p(out)))
    return out


def topk(scores, k: int) -> np.ndarray:
    """Row-wise top-k of a [rows, n] array by (score desc, index asc), -inf
    and NaN excluded; indices ascending, -1 padded.  Scores are taken as fp64
    (an fp32 input converts exactly)."""
    lib = _load()
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float64))
    if s.shape[-1] == 0:
        return np.full(s.shape[:-1] + (k,), -1, dtype=np.int32)
    s2 = s.reshape(-1, s.shape[-1])
    out = np.empty((s2.shape[0], k), dtype=np.int32)
    for i in range(s2.shape[0]):
        row = np.ascontiguousarray(s2[i])
        o = np.empty((k,), dtype=np.int32)
        _check(lib.orc_topk(_p(row), row.shape[0], k, _p(o)))
        out[i] = o
    return out.reshape(s.shape[:-1] + (k,))


def splitmix64(seed: int, n: int) -> int:
    """Output n (n >= 1) of SplitMix64 seeded with ``seed``."""
    return int(_load().orc_splitmix64(seed & (2**64 - 1), n & (2**64 - 1)))


def topk_approx(scores, k: int, seed: int, nbins: int = 2048, row0: int = 0) -> np.ndarray:
    """Row-wise approximate top-k with the stochastic early exit (the
    boundary bucket sampled): rows of fp32 scores, row i drawing
    splitmix64(seed, row0 + i + 1).  Indices ascending, -1 padded."""
    lib = _load()
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    s2 = s.reshape(-1, s.shape[-1])
    out = np.empty((s2.shape[0], k), dtype=np.int32)
    for i in range(s2.shape[0]):
        row = np.ascontiguousarray(s2[i])
        o = np.empty((max(k, 1),), dtype=np.int32)
        _check(lib.orc_topk_approx(_p(row), row.shape[0], k, nbins, seed & (2**64 - 1), row0 + i, _p(o)))
        out[i] = o[:k]
    return out.reshape(s.shape[:-1] + (k,))


def fine_scores(q, index_cache: Cache, page_table, num_q_heads, r: int, h: int, blocks, fine_weights=None):
    """fp64 FP8 rescoring of every token of ``blocks`` (request r, KV head h):
    returns (scores, token positions).  fine_weights [B, Hq]: the weighted
    ReLU head aggregation instead of the head sum."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    bl = np.ascontiguousarray(np.asarray(blocks, dtype=np.int64))
    b = index_cache.shape[2]
    fw = None if fine_weights is None else _np(fine_weights, np.float32)
    prm = _params(pt.shape[0], num_q_heads, pt.shape[1], fine_weights=fw)
    f = np.empty((bl.shape[0] * b,), dtype=np.float64)
    t = np.empty((bl.shape[0] * b,), dtype=np.int64)
    _check(lib.orc_fine_scores(_p(qa), index_cache.ref, _p(pt), C.byref(prm), r, h, bl.shape[0],
                               _p(bl), _p(f), _p(t)))
    return f, t


def pq_scores(q, index_cache: Cache, page_table, num_q_heads, fine_weights, pq_codes, pq_codebook,
              r: int, h: int, t0: int, n: int):
    """fp64 PQ32 coarse scores (LeanSparse Eq. 6) of tokens [t0, t0+n) of
    request r, KV head h."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    fw = _np(fine_weights, np.float32)
    codes = _np(pq_codes, np.uint8)
    cbk = _np(pq_codebook, np.uint16)
    prm = _params(pt.shape[0], num_q_heads, pt.shape[1], fine_weights=fw, pq_candidates=1,
                  pq_codes=codes, pq_codebook=cbk)
    out = np.empty((n,), dtype=np.float64)
    _check(lib.orc_pq_scores(_p(qa), index_cache.ref, _p(pt), C.byref(prm), r, h, int(t0), int(n), _p(out)))
    return out


def pq_encode(index_cache: Cache, pq_codebook, slots):
    """PQ32 codes [n, 32] of the index keys at flattened slots p * b + t
    (one KV head): nearest centroid per 4-dim subvector, fp32 distances."""
    lib = _load()
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    cbk = _np(pq_codebook, np.uint16)
    codes = np.empty((sl.shape[0], 32), dtype=np.uint8)
    _check(lib.orc_pq_encode(index_cache.ref, _p(cbk), sl.shape[0], _p(sl), _p(codes)))
    return codes


def token_scores_wrelu(q, index_cache: Cache, page_table, num_q_heads, fine_weights, r: int, h: int, tokens):
    """fp64 weighted-ReLU index scores (the exact keys) of explicit tokens."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    fw = _np(fine_weights, np.float32)
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    prm = _params(pt.shape[0], num_q_heads, pt.shape[1], fine_weights=fw)
    out = np.empty((tok.shape[0],), dtype=np.float64)
    _check(lib.orc_token_scores_wrelu(_p(qa), index_cache.ref, _p(pt), C.byref(prm), int(r), int(h), tok.shape[0],
                                      _p(tok), _p(out)))
    return out


def miss_filter(scores, hit, k: int):
    """LeanSparse's miss filter over candidate coarse scores: (keep mask, tau)."""
    lib = _load()
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float64))
    hh = np.ascontiguousarray(np.asarray(hit, dtype=np.uint8))
    keep = np.empty((s.shape[0],), dtype=np.uint8)
    tau = np.empty((1,), dtype=np.float64)
    _check(lib.orc_miss_filter(_p(s), _p(hh), s.shape[0], int(k), _p(keep), _p(tau)))
    return keep.astype(bool), float(tau[0])


def pq_select(q, index_cache: Cache, page_table, seq_lens, *, num_q_heads, sink, recent, fine_weights,
              pq_codes, pq_codebook, pq_hit, pq_candidates: int, tokens: int, r: int, h: int):
    """The PQ coarse-to-fine selection of (r, h): dict(sel [tokens], cand
    [C], kept [C] bool, tau)."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    fw = _np(fine_weights, np.float32)
    codes = _np(pq_codes, np.uint8)
    cbk = _np(pq_codebook, np.uint16)
    hit = None if pq_hit is None else _np(pq_hit, np.uint8)
    prm = _params(pt.shape[0], num_q_heads, pt.shape[1], 0, sink, recent, 1.0, 0, tokens, 0, fw,
                  pq_candidates, codes, cbk, hit)
    sel = np.empty((max(tokens, 1),), dtype=np.int32)
    cand = np.empty((max(pq_candidates, 1),), dtype=np.int32)
    kept = np.empty((max(pq_candidates, 1),), dtype=np.uint8)
    tau = np.empty((1,), dtype=np.float64)
    _check(lib.orc_pq_select(_p(qa), index_cache.ref, _p(pt), _p(lens), C.byref(prm), int(r), int(h),
                             _p(sel), _p(cand), _p(kept), _p(tau)))
    return dict(sel=sel[:tokens], cand=cand[:pq_candidates], kept=kept[:pq_candidates].astype(bool),
                tau=float(tau[0]))


def decode(q, cache: Cache, page_table, seq_lens, *, num_q_heads, k_blocks, sink, recent, scale,
           summ=None, index_cache: Optional[Cache] = None, index_summ=None,
           c2f_candidates: int = 0, c2f_tokens: int = 0, nthreads: int = 1, summary_kind: int = 0,
           fine_weights=None, pq_candidates: int = 0, pq_codes=None, pq_codebook=None, pq_hit=None):
    """The whole decode step.  Returns dict(out [B,Hq,dv] uint16 bf16 bits,
    lse [B,Hq] fp64, sel [B,Hkv,ksel] int32, cand [B,Hkv,C] int32 or None)
    (C: the coarse block candidates, or with pq_candidates the PQ coarse
    token candidates)."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    s = None if summ is None else _np(summ, np.uint16)
    isum = None if index_summ is None else _np(index_summ, np.uint16)
    B, maxb = pt.shape
    Hkv = cache.shape[1]
    fw = None if fine_weights is None else _np(fine_weights, np.float32)
    codes = None if pq_codes is None else _np(pq_codes, np.uint8)
    cbk = None if pq_codebook is None else _np(pq_codebook, np.uint16)
    hit = None if pq_hit is None else _np(pq_hit, np.uint8)
    prm = _params(B, num_q_heads, maxb, k_blocks, sink, recent, scale, c2f_candidates, c2f_tokens,
                  summary_kind, fw, pq_candidates, codes, cbk, hit)
    ksel = c2f_tokens if (c2f_candidates > 0 or pq_candidates > 0) else k_blocks
    ncand = pq_candidates if pq_candidates > 0 else c2f_candidates
    out = np.zeros((B, num_q_heads, cache.dv), dtype=np.uint16)
    lse = np.zeros((B, num_q_heads), dtype=np.float64)
    sel = np.zeros((B, Hkv, max(ksel, 0)), dtype=np.int32)
    cand = np.zeros((B, Hkv, ncand), dtype=np.int32) if ncand > 0 else None
    _check(lib.orc_decode(_p(qa), cache.ref, _p(s), index_cache.ref if index_cache else None,
                          _p(isum), _p(pt), _p(lens), C.byref(prm), int(nthreads), _p(out),
                          _p(lse), _p(sel), _p(cand)))
    return dict(out=out, lse=lse, sel=sel, cand=cand)


def dense(q, cache: Cache, page_table, seq_lens, *, num_q_heads, scale):
    """Dense attention over all L tokens (bf16 bits out, fp64 lse)."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    B, maxb = pt.shape
    prm = _params(B, num_q_heads, maxb, scale=scale)
    out = np.zeros((B, num_q_heads, cache.dv), dtype=np.uint16)
    lse = np.zeros((B, num_q_heads), dtype=np.float64)
    _check(lib.orc_dense(_p(qa), cache.ref, _p(pt), _p(lens), C.byref(prm), _p(out), _p(lse)))
    return dict(out=out, lse=lse)


def attend_tokens(q_head, cache: Cache, page_table_row, tokens, h: int, scale: float):
    """fp64 attention of one query head (fp64 vector) over explicit tokens."""
    lib = _load()
    qd = np.ascontiguousarray(np.asarray(q_head, dtype=np.float64))
    ptr = _np(page_table_row, np.int32)
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    o = np.empty((cache.dv,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    _check(lib.orc_attend_tokens(_p(qd), cache.ref, _p(ptr), tok.shape[0], _p(tok), int(h),
                                 float(scale), _p(o), _p(lse)))
    return o, float(lse[0])


def attend_selection(q, cache: Cache, page_table, seq_lens, sel, *, num_q_heads, sink, recent, scale,
                     token_mode: bool = False):
    """Attention over forced tokens plus a given selection ([B, Hkv, n]
    block indices, or token positions in token mode).  Returns dict(out, lse)."""
    lib = _load()
    qa = _np(q, np.uint16)
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    s = _np(sel, np.int32)
    B, maxb = pt.shape
    prm = _params(B, num_q_heads, maxb, s.shape[-1], sink, recent, scale)
    out = np.zeros((B, num_q_heads, cache.dv), dtype=np.uint16)
    lse = np.zeros((B, num_q_heads), dtype=np.float64)
    _check(lib.orc_attend_selection(_p(qa), cache.ref, _p(pt), _p(lens), C.byref(prm), _p(s), s.shape[-1],
                                    int(token_mode), _p(out), _p(lse)))
    return dict(out=out, lse=lse)


def lse_merge(o_parts, lse_parts):
    lib = _load()
    o = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    n, dv = o.shape
    oo = np.empty((dv,), dtype=np.float64)
    lo = np.empty((1,), dtype=np.float64)
    lib.orc_lse_merge(n, dv, _p(o), _p(l), _p(oo), _p(lo))
    return oo, float(lo[0])


def bf16_bits_to_f64(a) -> np.ndarray:
    """Decode a uint16 bf16 bit-pattern array to fp64 (bit shift only)."""
    a = np.asarray(a).astype(np.uint32) << 16
    return a.view(np.float32).astype(np.float64)
