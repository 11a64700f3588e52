"""Thin ctypes binding of liblsa.so.

Every function has the name and argument order of its C counterpart in
include/lsa.h and only marshals arguments: torch tensors become device
pointers and strides, the stream defaults to torch's current stream, and a
non-OK status raises LsaError.  All computation happens in the library's CUDA
kernels; there is no fallback.  If liblsa.so is missing the first call fails
with an error naming the build step.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("LSA_LIBRARY") or os.path.join(_HERE, "liblsa.so")

LSA_OK = 0
LSA_ERR_INVALID_ARG = 1
LSA_ERR_UNSUPPORTED = 2
LSA_ERR_WORKSPACE = 3
LSA_ERR_BOUNDS = 4
LSA_ERR_TIMEOUT = 5
LSA_ERR_CUDA = 6
LSA_ERR_NAN = 7
LSA_KEYS_BF16 = 0
LSA_KEYS_E4M3 = 1
LSA_SUMMARY_MEAN = 0
LSA_SUMMARY_MINMAX = 1

EXPORTED = ["lsa_status_string", "lsa_get_device_status", "lsa_build_summaries", "lsa_append_block",
            "lsa_build_minmax_summaries", "lsa_append_block_minmax",
            "lsa_score", "lsa_topk", "lsa_topk_approx", "lsa_fine_topk", "lsa_pq_encode", "lsa_pq_scores",
            "lsa_decode_step_launches", "lsa_sparse_decode_workspace_size",
            "lsa_sparse_decode", "lsa_decode_step_workspace_size", "lsa_decode_step",
            "lsa_sparse_decode_static_scratch"]


class LsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lsa_status_string(code)} (status {code})")


class lsa_cache(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p),
                ("k_page_stride", C.c_int64), ("k_head_stride", C.c_int64), ("k_token_stride", C.c_int64),
                ("v_page_stride", C.c_int64), ("v_head_stride", C.c_int64), ("v_token_stride", C.c_int64),
                ("num_pages", C.c_int32), ("block_size", C.c_int32), ("num_kv_heads", C.c_int32),
                ("dk", C.c_int32), ("dv", C.c_int32), ("key_format", C.c_int32),
                ("k_scale", C.c_void_p), ("scale_page_stride", C.c_int64), ("scale_head_stride", C.c_int64)]


class lsa_params(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_q_heads", C.c_int32), ("max_blocks", C.c_int32),
                ("k_blocks", C.c_int32), ("sink_tokens", C.c_int32), ("recent_tokens", C.c_int32),
                ("softmax_scale", C.c_float), ("c2f_candidates", C.c_int32), ("c2f_tokens", C.c_int32),
                ("num_splits", C.c_int32), ("summary_kind", C.c_int32),
                ("fine_head_weights", C.c_void_p), ("pq_candidates", C.c_int32),
                ("pq_codes", C.c_void_p), ("pq_codebook", C.c_void_p), ("pq_hit", C.c_void_p)]


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None):
    """Load liblsa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -c \"import __graft_entry__ as g; "
                               f"g.build()\"` (nvcc, sm_103a)")
        lib = C.CDLL(p)
        V, P, I, S = C.c_void_p, C.POINTER, C.c_int32, C.c_size_t
        cache_p, params_p = P(lsa_cache), P(lsa_params)
        sig = {
            "lsa_status_string": ([C.c_int], C.c_char_p),
            "lsa_get_device_status": ([P(C.c_uint32), C.c_int], C.c_int),
            "lsa_build_summaries": ([cache_p, V, V, I, I, V, V], C.c_int),
            "lsa_append_block": ([cache_p, V, V, V, V, I, I, V, V], C.c_int),
            "lsa_build_minmax_summaries": ([cache_p, V, V, I, I, V, V], C.c_int),
            "lsa_append_block_minmax": ([cache_p, V, V, V, V, I, I, V, V], C.c_int),
            "lsa_score": ([V, cache_p, V, V, V, params_p, V, V], C.c_int),
            "lsa_topk": ([V, V, I, I, I, V, V], C.c_int),
            "lsa_topk_approx": ([V, V, I, I, I, C.c_uint64, V, V], C.c_int),
            "lsa_pq_encode": ([cache_p, V, V, V, I, I, V, V], C.c_int),
            "lsa_decode_step_launches": ([cache_p, cache_p, params_p], C.c_int32),
            "lsa_pq_scores": ([V, cache_p, V, V, params_p, V, V], C.c_int),
            "lsa_fine_topk": ([V, cache_p, V, V, V, params_p, V, V, S, V], C.c_int),
            "lsa_sparse_decode_workspace_size": ([cache_p, params_p], S),
            "lsa_sparse_decode": ([V, cache_p, V, V, V, params_p, V, V, V, S, V], C.c_int),
            "lsa_sparse_decode_static_scratch": ([V, cache_p, V, V, V, params_p, V, V, V], C.c_int),
            "lsa_decode_step_workspace_size": ([cache_p, params_p], S),
            "lsa_decode_step": ([V, cache_p, V, cache_p, V, V, params_p, V, V, V, V, S, V], C.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def lsa_status_string(code: int) -> str:
    return load_library().lsa_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != LSA_OK:
        raise LsaError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def make_cache(k: torch.Tensor, v: Optional[torch.Tensor] = None, *, k_scale: Optional[torch.Tensor] = None,
               num_pages: Optional[int] = None) -> lsa_cache:
    """Describe a paged cache.  ``k``: [P, Hkv, b, dk] bf16 (or uint8 /
    float8_e4m3fn index keys, with ``k_scale`` [P, Hkv, b] fp32); ``v``:
    [P, Hkv, b, dv] bf16, a view of ``k`` for a latent cache, or None for an
    index cache.  Strides are taken from the tensors (in elements)."""
    c = lsa_cache()
    P, H, b, dk = k.shape
    c.k = k.data_ptr()
    c.k_page_stride, c.k_head_stride, c.k_token_stride = k.stride(0), k.stride(1), k.stride(2)
    c.num_pages = num_pages if num_pages is not None else P
    c.block_size, c.num_kv_heads, c.dk = b, H, dk
    if k.dtype in (torch.uint8, torch.float8_e4m3fn):
        c.key_format = LSA_KEYS_E4M3
        assert k_scale is not None and k_scale.dtype == torch.float32
        c.k_scale = k_scale.data_ptr()
        c.scale_page_stride, c.scale_head_stride = k_scale.stride(0), k_scale.stride(1)
    else:
        assert k.dtype == torch.bfloat16
        c.key_format = LSA_KEYS_BF16
    if v is not None:
        assert v.dtype == torch.bfloat16
        c.v = v.data_ptr()
        c.v_page_stride, c.v_head_stride, c.v_token_stride = v.stride(0), v.stride(1), v.stride(2)
        c.dv = v.shape[-1]
    return c


def make_params(batch, num_q_heads, max_blocks, k_blocks=0, sink_tokens=0, recent_tokens=0,
                softmax_scale=0.0, c2f_candidates=0, c2f_tokens=0, num_splits=0, summary_kind=0,
                fine_head_weights: Optional[torch.Tensor] = None, pq_candidates=0,
                pq_codes: Optional[torch.Tensor] = None, pq_codebook: Optional[torch.Tensor] = None,
                pq_hit: Optional[torch.Tensor] = None) -> lsa_params:
    """fine_head_weights: device fp32 [batch, num_q_heads]; pq_codes uint8
    [num_pages, 1, b, 32], pq_codebook bf16 [32, 256, 4], pq_hit uint8
    [num_pages, 1, b] (device).  The caller keeps the tensors alive while the
    parameters are in use."""
    return lsa_params(int(batch), int(num_q_heads), int(max_blocks), int(k_blocks), int(sink_tokens),
                      int(recent_tokens), float(softmax_scale), int(c2f_candidates), int(c2f_tokens),
                      int(num_splits), int(summary_kind), _ptr(fine_head_weights), int(pq_candidates),
                      _ptr(pq_codes), _ptr(pq_codebook), _ptr(pq_hit))


def lsa_get_device_status(clear: bool = True):
    """(status code, raw flag bits) of the current device; synchronises."""
    flags = C.c_uint32(0)
    code = load_library().lsa_get_device_status(C.byref(flags), int(bool(clear)))
    return code, int(flags.value)


def lsa_build_summaries(cache: lsa_cache, page_table, seq_lens, summaries, stream=None):
    B, maxb = page_table.shape
    _check(load_library().lsa_build_summaries(C.byref(cache), _ptr(page_table), _ptr(seq_lens), B, maxb,
                                              _ptr(summaries), _stream(stream)), "lsa_build_summaries")


def lsa_build_minmax_summaries(cache: lsa_cache, page_table, seq_lens, summaries, stream=None):
    B, maxb = page_table.shape
    _check(load_library().lsa_build_minmax_summaries(C.byref(cache), _ptr(page_table), _ptr(seq_lens), B, maxb,
                                                     _ptr(summaries), _stream(stream)), "lsa_build_minmax_summaries")


def lsa_append_block_minmax(cache: lsa_cache, k_new, v_new, page_table, seq_lens, summaries, stream=None):
    B, maxb = page_table.shape
    _check(load_library().lsa_append_block_minmax(C.byref(cache), _ptr(k_new), _ptr(v_new), _ptr(page_table),
                                                  _ptr(seq_lens), B, maxb, _ptr(summaries), _stream(stream)),
           "lsa_append_block_minmax")


def lsa_append_block(cache: lsa_cache, k_new, v_new, page_table, seq_lens, summaries, stream=None):
    B, maxb = page_table.shape
    _check(load_library().lsa_append_block(C.byref(cache), _ptr(k_new), _ptr(v_new), _ptr(page_table),
                                           _ptr(seq_lens), B, maxb, _ptr(summaries), _stream(stream)),
           "lsa_append_block")


def lsa_score(q, cache: lsa_cache, summaries, page_table, seq_lens, params: lsa_params, scores, stream=None):
    _check(load_library().lsa_score(_ptr(q), C.byref(cache), _ptr(summaries), _ptr(page_table), _ptr(seq_lens),
                                    C.byref(params), _ptr(scores), _stream(stream)), "lsa_score")


def lsa_topk(scores, num_cols, k: int, idx, stream=None):
    rows, cols = scores.shape
    _check(load_library().lsa_topk(_ptr(scores), _ptr(num_cols), rows, cols, int(k), _ptr(idx), _stream(stream)),
           "lsa_topk")


def lsa_topk_approx(scores, num_cols, k: int, seed: int, idx, stream=None):
    rows, cols = scores.shape
    _check(load_library().lsa_topk_approx(_ptr(scores), _ptr(num_cols), rows, cols, int(k),
                                          int(seed) & (2**64 - 1), _ptr(idx), _stream(stream)),
           "lsa_topk_approx")


def lsa_decode_step_launches(cache: lsa_cache, index_cache: Optional[lsa_cache], params: lsa_params) -> int:
    return int(load_library().lsa_decode_step_launches(C.byref(cache), C.byref(index_cache) if index_cache else None,
                                                       C.byref(params)))


def lsa_pq_encode(index_cache: lsa_cache, codebook, page_table, seq_lens, codes, stream=None):
    B, maxb = page_table.shape
    _check(load_library().lsa_pq_encode(C.byref(index_cache), _ptr(codebook), _ptr(page_table), _ptr(seq_lens), B,
                                        maxb, _ptr(codes), _stream(stream)), "lsa_pq_encode")


def lsa_pq_scores(q, index_cache: lsa_cache, page_table, seq_lens, params: lsa_params, scores, stream=None):
    _check(load_library().lsa_pq_scores(_ptr(q), C.byref(index_cache), _ptr(page_table), _ptr(seq_lens),
                                        C.byref(params), _ptr(scores), _stream(stream)), "lsa_pq_scores")


def lsa_fine_topk(q, index_cache: lsa_cache, page_table, seq_lens, cand, params: lsa_params, tok_idx,
                  workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().lsa_fine_topk(_ptr(q), C.byref(index_cache), _ptr(page_table), _ptr(seq_lens),
                                        _ptr(cand), C.byref(params), _ptr(tok_idx), _ptr(workspace), nbytes,
                                        _stream(stream)), "lsa_fine_topk")


def lsa_sparse_decode_workspace_size(cache: lsa_cache, params: lsa_params) -> int:
    return int(load_library().lsa_sparse_decode_workspace_size(C.byref(cache), C.byref(params)))


def lsa_sparse_decode(q, cache: lsa_cache, page_table, seq_lens, idx, params: lsa_params, out, lse, workspace,
                      stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().lsa_sparse_decode(_ptr(q), C.byref(cache), _ptr(page_table), _ptr(seq_lens), _ptr(idx),
                                            C.byref(params), _ptr(out), _ptr(lse), _ptr(workspace), nbytes,
                                            _stream(stream)), "lsa_sparse_decode")


def lsa_sparse_decode_static_scratch(q, cache: lsa_cache, page_table, seq_lens, idx, params: lsa_params, out, lse,
                                     stream=None):
    _check(load_library().lsa_sparse_decode_static_scratch(_ptr(q), C.byref(cache), _ptr(page_table),
                                                           _ptr(seq_lens), _ptr(idx), C.byref(params), _ptr(out),
                                                           _ptr(lse), _stream(stream)),
           "lsa_sparse_decode_static_scratch")


def lsa_decode_step_workspace_size(cache: lsa_cache, params: lsa_params) -> int:
    return int(load_library().lsa_decode_step_workspace_size(C.byref(cache), C.byref(params)))


def lsa_decode_step(q, cache: lsa_cache, summaries, index_cache: Optional[lsa_cache], page_table, seq_lens,
                    params: lsa_params, idx_out, out, lse, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().lsa_decode_step(_ptr(q), C.byref(cache), _ptr(summaries),
                                          C.byref(index_cache) if index_cache is not None else None,
                                          _ptr(page_table), _ptr(seq_lens), C.byref(params), _ptr(idx_out),
                                          _ptr(out), _ptr(lse), _ptr(workspace), nbytes, _stream(stream)),
           "lsa_decode_step")
