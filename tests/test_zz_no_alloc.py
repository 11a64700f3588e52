"""lsa_sparse_decode_static_scratch: the attention call that takes no caller
workspace and allocates nothing (its scratch is the library's static device
buffer).  Compared against lsa_sparse_decode on the same inputs, two calls in
a row each, and checked to reject shapes whose scratch would not fit.

Kept last in collection order so that it also runs after every other GPU
test of the session has used the library.
"""
import pytest
import torch

import sparse_attention_decode_block_gb300 as L
from helpers import check_status_clean, to_dev
from workloads import WORKLOADS, make_inputs, small_workloads

pytestmark = pytest.mark.gpu

STATIC_BYTES = 8 << 20   # LSA_STATIC_SCRATCH_BYTES in include/lsa.h


def _select_on_gpu(w, g, cache, summ, prm):
    """The GPU's own block selection for the inputs (lsa_score + lsa_topk)."""
    B, Hkv = w.batch, w.num_kv_heads
    scores = torch.empty((B, Hkv, g["max_blocks"]), dtype=torch.float32, device="cuda")
    L.lsa_score(g["q"], cache, summ, g["page_table"], g["seq_lens"], prm, scores)
    idx = torch.empty((B, Hkv, w.k_blocks), dtype=torch.int32, device="cuda")
    L.lsa_topk(scores.view(B * Hkv, -1), None, w.k_blocks, idx.view(B * Hkv, -1))
    return idx


@pytest.mark.parametrize("name", ["b16_small", "ragged_small", "b16_32k"])
def test_static_scratch_matches_workspace_call_twice(name):
    w = WORKLOADS[name] if name in WORKLOADS else small_workloads()[name]
    g = make_inputs(w, "cuda") if name in WORKLOADS else to_dev(make_inputs(w, "cpu"))
    cache = L.make_cache(g["k_cache"], g["v_cache"])
    prm = L.make_params(w.batch, w.num_q_heads, g["max_blocks"], w.k_blocks, w.sink, w.recent, w.softmax_scale)
    need = L.lsa_sparse_decode_workspace_size(cache, prm)
    assert need <= STATIC_BYTES
    summ = torch.zeros((g["num_pages"], w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_summaries(cache, g["page_table"], g["seq_lens"], summ)
    idx = _select_on_gpu(w, g, cache, summ, prm)

    ws = torch.zeros(max(16, need), dtype=torch.uint8, device="cuda")
    shape = (w.batch, w.num_q_heads)
    ref_out = torch.empty(shape + (w.dv,), dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(shape, dtype=torch.float32, device="cuda")
    L.lsa_sparse_decode(g["q"], cache, g["page_table"], g["seq_lens"], idx, prm, ref_out, ref_lse, ws)

    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        L.lsa_sparse_decode_static_scratch(g["q"], cache, g["page_table"], g["seq_lens"], idx, prm, out, lse)
        torch.cuda.synchronize()
        check_status_clean()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)


def test_static_scratch_follows_the_attention_plan(monkeypatch):
    """Calls of one shape whose attention plan alternates (LSA_ATTENTION_PATH
    picks the CUDA-core split-K kernel, whose partials fill the buffer, or
    the default tensor-core even split, whose per-row counters must start at
    zero): each call equals lsa_sparse_decode on a fresh workspace under the
    same plan."""
    w = small_workloads()["b16_small"]
    g = to_dev(make_inputs(w, "cpu"))
    cache = L.make_cache(g["k_cache"], g["v_cache"])
    prm = L.make_params(w.batch, w.num_q_heads, g["max_blocks"], w.k_blocks, w.sink, w.recent, w.softmax_scale)
    summ = torch.zeros((g["num_pages"], w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_summaries(cache, g["page_table"], g["seq_lens"], summ)
    idx = _select_on_gpu(w, g, cache, summ, prm)
    shape = (w.batch, w.num_q_heads)
    for path in ["cuda_core", "tensor_core", "cuda_core", "tensor_core", "tensor_core"]:
        if path == "cuda_core":
            monkeypatch.setenv("LSA_ATTENTION_PATH", "cuda_core")
        else:
            monkeypatch.delenv("LSA_ATTENTION_PATH", raising=False)
        need = L.lsa_sparse_decode_workspace_size(cache, prm)
        assert 0 < need <= STATIC_BYTES
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        ref_out = torch.empty(shape + (w.dv,), dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty(shape, dtype=torch.float32, device="cuda")
        L.lsa_sparse_decode(g["q"], cache, g["page_table"], g["seq_lens"], idx, prm, ref_out, ref_lse, ws)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        L.lsa_sparse_decode_static_scratch(g["q"], cache, g["page_table"], g["seq_lens"], idx, prm, out, lse)
        torch.cuda.synchronize()
        check_status_clean()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), path
        assert torch.equal(lse, ref_lse), path


def test_static_scratch_rejects_bad_pointers_before_touching_the_buffer():
    w = small_workloads()["tiny"]
    g = to_dev(make_inputs(w, "cpu"))
    cache = L.make_cache(g["k_cache"], g["v_cache"])
    prm = L.make_params(w.batch, w.num_q_heads, g["max_blocks"], w.k_blocks, w.sink, w.recent, w.softmax_scale)
    out = torch.empty((w.batch, w.num_q_heads, w.dv), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.LsaError) as e:
        L.lsa_sparse_decode_static_scratch(g["q"], cache, g["page_table"], g["seq_lens"], None, prm, out, None)
    assert e.value.code == L.LSA_ERR_INVALID_ARG


def test_static_scratch_rejects_shapes_that_do_not_fit():
    # many requests with many split parts: the partials exceed the static buffer
    B, hq, hkv, d, b, nb = 512, 32, 8, 128, 16, 4
    pages = B * nb
    k = torch.zeros((pages, hkv, b, d), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    q = torch.zeros((B, hq, d), dtype=torch.bfloat16, device="cuda")
    pt = torch.arange(pages, dtype=torch.int32, device="cuda").view(B, nb)
    lens = torch.full((B,), nb * b, dtype=torch.int32, device="cuda")
    idx = torch.zeros((B, hkv, 1), dtype=torch.int32, device="cuda")
    out = torch.empty((B, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    cache = L.make_cache(k, v)
    prm = L.make_params(B, hq, nb, 1, 16, 16, d ** -0.5, num_splits=4)
    assert L.lsa_sparse_decode_workspace_size(cache, prm) > STATIC_BYTES
    with pytest.raises(L.LsaError) as e:
        L.lsa_sparse_decode_static_scratch(q, cache, pt, lens, idx, prm, out, lse)
    assert e.value.code == L.LSA_ERR_WORKSPACE
    torch.cuda.synchronize()
    check_status_clean()
