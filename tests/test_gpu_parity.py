"""GPU parity: every C-ABI entry point against the CPU oracle on the same
seeded inputs (small workloads spanning several tiles with ragged tails,
edge cases, and the full-size workloads on sampled requests)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_decode_block_gb300 as L
from helpers import (GpuStep, assert_attention_close, assert_lse_close, bits, check_status_clean,
                     compare_selection, f64, oracle_cache, oracle_decode, oracle_index, quest_score_bound,
                     score_bound, subset, to_dev)
from workloads import WORKLOADS, make_inputs, small_workloads

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")
SMALL = ["tiny", "b16_small", "ragged_small", "mla_small"]
QUEST = ["quest_small"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    L.lsa_get_device_status(clear=True)
    yield


def small(name, **kw):
    w = small_workloads()[name]
    return w.replace(**kw) if kw else w


# ---------------------------------------------------------------- summaries

@pytest.mark.parametrize("name", SMALL + ["c2f_small"])
def test_summaries_bit_exact(name):
    w = small(name)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    if w.c2f_candidates:
        c = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
        oc, use8 = oracle_index(cpu), True
    else:
        c = L.make_cache(g["k_cache"], g["v_cache"])
        oc, use8 = oracle_cache(cpu), False
    summ = torch.zeros((cpu["num_pages"], w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_summaries(c, g["page_table"], g["seq_lens"], summ)
    check_status_clean()
    ref, valid = oracle.summaries(oc, cpu["page_table"], cpu["seq_lens"], use_index_keys=use8)
    got = bits(summ)
    assert valid.any()
    assert np.array_equal(got[valid], ref[valid])
    assert np.all(got[~valid] == 0)          # pages with no full block untouched


def test_summaries_bit_exact_block_48():
    """A block size that is not a power of two: the mean is a correctly
    rounded fp64 division on both sides, then one bf16 rounding."""
    w = small("b16_small", block_size=48, seq_lens=(4096, 3001, 777), k_blocks=20)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    c = L.make_cache(g["k_cache"], g["v_cache"])
    summ = torch.zeros((cpu["num_pages"], w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_summaries(c, g["page_table"], g["seq_lens"], summ)
    check_status_clean()
    ref, valid = oracle.summaries(oracle_cache(cpu), cpu["page_table"], cpu["seq_lens"])
    got = bits(summ)
    assert valid.any()
    assert np.array_equal(got[valid], ref[valid])
    # and the whole step at b = 48 (three 16-token items per block)
    run_and_compare_step(w, cpu, g)


def test_quest_summaries_bit_exact_and_append_matches_bulk():
    """Quest's max / min key summaries: bit-exact against the oracle, and
    appending tokens one by one builds the same summaries as the bulk call."""
    w = small("quest_small")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    c = L.make_cache(g["k_cache"], g["v_cache"])
    summ = torch.zeros((cpu["num_pages"], w.num_kv_heads, 2, w.dk), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_minmax_summaries(c, g["page_table"], g["seq_lens"], summ)
    check_status_clean()
    ref, valid = oracle.quest_summaries(oracle_cache(cpu), cpu["page_table"], cpu["seq_lens"])
    got = bits(summ)
    assert valid.any()
    assert np.array_equal(got[valid], ref[valid])
    assert np.all(got[~valid] == 0)
    # append: the last 40 tokens of each request one at a time
    lens0 = [L_ - 40 for L_ in cpu["lens"]]
    kc = g["k_cache"].clone()
    vc = g["v_cache"].clone()
    cache2 = L.make_cache(kc, vc)
    lens = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    summ2 = torch.zeros_like(summ)
    L.lsa_build_minmax_summaries(cache2, g["page_table"], lens, summ2)
    pt = cpu["page_table"]
    b = w.block_size
    for step in range(40):
        kn = torch.empty((w.batch, w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
        vn = torch.empty_like(kn)
        for r in range(w.batch):
            t = lens0[r] + step
            p = int(pt[r, t // b])
            kn[r] = g["k_cache"][p, :, t % b]
            vn[r] = g["v_cache"][p, :, t % b]
        L.lsa_append_block_minmax(cache2, kn, vn, g["page_table"], lens, summ2)
    check_status_clean()
    assert lens.tolist() == list(cpu["lens"])
    assert torch.equal(summ2.view(torch.int16), summ.view(torch.int16))


def test_quest_scores_within_rounding_and_topk_bit_exact():
    w = small("quest_small")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    c = L.make_cache(g["k_cache"], g["v_cache"])
    summ = torch.zeros((cpu["num_pages"], w.num_kv_heads, 2, w.dk), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_minmax_summaries(c, g["page_table"], g["seq_lens"], summ)
    prm = L.make_params(w.batch, w.num_q_heads, cpu["max_blocks"], w.k_blocks, w.sink, w.recent,
                        summary_kind=L.LSA_SUMMARY_MINMAX)
    scores = torch.empty((w.batch, w.num_kv_heads, cpu["max_blocks"]), dtype=torch.float32, device="cuda")
    L.lsa_score(g["q"], c, summ, g["page_table"], g["seq_lens"], prm, scores)
    check_status_clean()
    oc = oracle_cache(cpu)
    osumm, _ = oracle.quest_summaries(oc, cpu["page_table"], cpu["seq_lens"])
    ref = oracle.block_scores(cpu["q"], oc, osumm, cpu["page_table"], cpu["seq_lens"], w.num_q_heads, w.sink,
                              w.recent, summary_kind=1)
    got = scores.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    S = f64(osumm)
    G = w.group
    for r in range(w.batch):
        pg = np.maximum(cpu["page_table"][r].numpy(), 0)
        for h in range(w.num_kv_heads):
            fin = np.isfinite(ref[r, h])
            tau = quest_score_bound(bits(cpu["q"][r, h * G:(h + 1) * G]), S[pg, h, 0], S[pg, h, 1], w.dk)
            assert np.all(np.abs(got[r, h][fin] - ref[r, h][fin]) <= tau[fin] + 1e-30)
    idx = torch.empty((w.batch * w.num_kv_heads, w.k_blocks), dtype=torch.int32, device="cuda")
    L.lsa_topk(scores.view(w.batch * w.num_kv_heads, -1), None, w.k_blocks, idx)
    check_status_clean()
    want = oracle.topk(got.reshape(w.batch * w.num_kv_heads, -1), w.k_blocks)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_append_matches_bulk_build():
    w = small("b16_small", seq_lens=(100, 33, 18))
    cpu = make_inputs(w, "cpu", lens=[100 + 40, 33 + 40, 18 + 40])   # room for 40 appended tokens
    g = to_dev(cpu)
    L0 = torch.tensor([100, 33, 18], dtype=torch.int32, device="cuda")
    k_full, v_full = g["k_cache"].clone(), g["v_cache"].clone()
    k_cache = torch.zeros_like(k_full)
    v_cache = torch.zeros_like(v_full)
    # copy the first L0 tokens of every request, then append the rest one by one
    pt = cpu["page_table"]
    b = w.block_size
    for r in range(w.batch):
        for t in range(int(L0[r])):
            p = int(pt[r, t // b])
            k_cache[p, :, t % b] = k_full[p, :, t % b]
            v_cache[p, :, t % b] = v_full[p, :, t % b]
    cache = L.make_cache(k_cache, v_cache)
    summ = torch.zeros((cpu["num_pages"], w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
    lens = L0.clone()
    L.lsa_build_summaries(cache, g["page_table"], lens, summ)
    for step in range(40):
        kn = torch.empty((w.batch, w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
        vn = torch.empty_like(kn)
        for r in range(w.batch):
            t = int(L0[r]) + step
            p = int(pt[r, t // b])
            kn[r] = k_full[p, :, t % b]
            vn[r] = v_full[p, :, t % b]
        L.lsa_append_block(cache, kn, vn, g["page_table"], lens, summ)
    check_status_clean()
    assert lens.tolist() == [140, 73, 58]
    ref = torch.zeros_like(summ)
    L.lsa_build_summaries(L.make_cache(k_full, v_full), g["page_table"], lens, ref)
    torch.cuda.synchronize()
    assert torch.equal(summ.view(torch.int16), ref.view(torch.int16))
    for r in range(w.batch):
        for t in range(140 if r == 0 else (73 if r == 1 else 58)):
            p = int(pt[r, t // b])
            assert torch.equal(k_cache[p, :, t % b], k_full[p, :, t % b])
            assert torch.equal(v_cache[p, :, t % b], v_full[p, :, t % b])


# ---------------------------------------------------------------- scores / top-k

@pytest.mark.parametrize("name", SMALL + ["c2f_small"])
def test_scores_within_rounding_and_topk_bit_exact(name):
    w = small(name)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    use8 = w.c2f_candidates > 0
    c = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"]) if use8 else L.make_cache(g["k_cache"], g["v_cache"])
    oc = oracle_index(cpu) if use8 else oracle_cache(cpu)
    summ = torch.zeros((cpu["num_pages"], w.num_kv_heads, w.dk), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_summaries(c, g["page_table"], g["seq_lens"], summ)
    prm = L.make_params(w.batch, w.num_q_heads, cpu["max_blocks"], w.k_blocks, w.sink, w.recent)
    scores = torch.empty((w.batch, w.num_kv_heads, cpu["max_blocks"]), dtype=torch.float32, device="cuda")
    L.lsa_score(g["q"], c, summ, g["page_table"], g["seq_lens"], prm, scores)
    osumm, _ = oracle.summaries(oc, cpu["page_table"], cpu["seq_lens"], use_index_keys=use8)
    ref = oracle.block_scores(cpu["q"], oc, osumm, cpu["page_table"], cpu["seq_lens"], w.num_q_heads, w.sink,
                              w.recent, use_index_keys=use8)
    got = scores.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    S = f64(osumm)
    G = w.group
    for r in range(w.batch):
        for h in range(w.num_kv_heads):
            pg = cpu["page_table"][r].numpy()
            fin = np.isfinite(ref[r, h])
            tau = score_bound(bits(cpu["q"][r, h * G:(h + 1) * G]), S[np.maximum(pg, 0), h], G, w.dk)
            assert np.all(np.abs(got[r, h][fin] - ref[r, h][fin]) <= tau[fin] + 1e-30)
    # top-k over the GPU's fp32 scores: bit-exact against the oracle's top-k of the same values
    k = w.k_blocks if not use8 else w.c2f_candidates
    idx = torch.empty((w.batch * w.num_kv_heads, k), dtype=torch.int32, device="cuda")
    L.lsa_topk(scores.view(w.batch * w.num_kv_heads, -1), None, k, idx)
    check_status_clean()
    want = oracle.topk(got.reshape(w.batch * w.num_kv_heads, -1), k)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_topk_vortex_figure1_golden_gpu():
    gold = json.load(open(os.path.join(GOLD, "vortex_fig1_block_topk.json")))
    s = torch.tensor([gold["scores"]], dtype=torch.float32, device="cuda")
    idx = torch.empty((1, gold["k"]), dtype=torch.int32, device="cuda")
    L.lsa_topk(s, None, gold["k"], idx)
    assert idx.cpu().tolist()[0] == gold["selected_ascending"]


@pytest.mark.parametrize("cols,k", [(1, 1), (7, 3), (64, 62), (2048, 62), (2048, 1), (5000, 256),
                                    (16384, 2048), (16381, 29), (32768, 100), (100, 200)])
def test_topk_random_rows_with_ties(cols, k):
    gen = torch.Generator().manual_seed(cols * 7 + k)
    rows = 6
    s = torch.randint(-40, 40, (rows, cols), generator=gen).float() / 8     # many exact ties
    s[1] = torch.randn(cols, generator=gen)                                  # distinct values
    s[2] = 0.0
    s[2, ::3] = -0.0                                                         # -0 and +0 tie
    s[3, torch.rand(cols, generator=gen) < 0.5] = -math.inf                  # non-candidates
    s[4] = -math.inf
    s[5] = torch.randn(cols, generator=gen) * 1e30
    ncols = torch.tensor([cols, cols, cols, cols, cols, max(0, cols - 3)], dtype=torch.int32)
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    L.lsa_topk(s.cuda(), ncols.cuda(), k, idx)
    check_status_clean()
    want = np.stack([oracle.topk(s[i:i + 1, : int(ncols[i])].numpy(), k)[0] for i in range(rows)])
    assert np.array_equal(idx.cpu().numpy(), want)


@pytest.mark.parametrize("cols", [2048, 8192])
@pytest.mark.parametrize("k", [32, 62, 64, 65, 128])
def test_topk_clustered_rows_take_every_selection_path(cols, k):
    """Rows whose largest keys sit in few threads' columns: the candidate
    set at the k-th largest thread maximum grows past 128 (ranked through
    sorted runs) and past 512 (bisection), on both sides of k = 64, where
    the bound switches from the top-64 tree to the general search."""
    gen = torch.Generator().manual_seed(cols * 131 + k)
    rows = 5
    s = torch.randn(rows, cols, generator=gen)
    s[0, 500:700] += 20.0                                    # one contiguous cluster
    s[1] = torch.arange(cols, dtype=torch.float32)           # increasing: the last columns win
    s[2, ::16] += 10.0                                       # one high key every 16 columns
    s[3, 100:100 + 3 * k] = 7.0                              # a tie run longer than k at the top
    s[4, cols // 2:] = torch.randn(cols - cols // 2, generator=gen).abs() + 3.0   # upper half above the rest
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    L.lsa_topk(s.cuda(), None, k, idx)
    check_status_clean()
    want = oracle.topk(s.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), want)


@pytest.mark.parametrize("path", ["rows", "cluster"])
@pytest.mark.parametrize("cols,k", [(4097, 1), (8192, 256), (16381, 29), (16384, 2048), (32768, 100),
                                    (32768, 4000)])
def test_topk_row_and_cluster_kernels(cols, k, path, monkeypatch):
    """Few long rows: one CTA per row, or one cluster of CTAs per row
    sharing counts through distributed shared memory; both bit-exact,
    through the boundary-bucket ranking and the bisection for heavy ties."""
    monkeypatch.setenv("LSA_TOPK_PATH", path)
    gen = torch.Generator().manual_seed(cols * 3 + k)
    rows = 4
    s = torch.randn(rows, cols, generator=gen)
    s[1] = torch.randint(-6, 6, (cols,), generator=gen).float()       # ties far past the boundary cap
    s[2, : cols // 3] = -math.inf
    s[3, 100:100 + 2 * k] = 9.0                                       # a tie run longer than k at the top
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    L.lsa_topk(s.cuda(), None, k, idx)
    check_status_clean()
    assert np.array_equal(idx.cpu().numpy(), oracle.topk(s.numpy(), k))


@pytest.mark.parametrize("path", ["rows", "cluster"])
@pytest.mark.parametrize("cols,k", [(7, 3), (2048, 62), (5000, 256), (16381, 29), (16384, 2048), (32768, 100)])
def test_topk_approx_matches_oracle(cols, k, path, monkeypatch):
    """The stochastic early exit equals the oracle's, bit for bit, for the
    same seed and row numbers: exact winners above the boundary bucket and
    the same circular sample of it (fp32 bucket decisions on both sides)."""
    monkeypatch.setenv("LSA_TOPK_PATH", path)
    gen = torch.Generator().manual_seed(cols * 5 + k)
    rows = 5
    s = torch.randn(rows, cols, generator=gen)
    s[1] = torch.randint(-20, 20, (cols,), generator=gen).float() / 4     # crowded buckets
    s[2, torch.rand(cols, generator=gen) < 0.5] = -math.inf
    s[3] = 0.0
    s[4] = torch.randn(cols, generator=gen) * 1e30
    ncols = torch.tensor([cols, cols, cols, max(0, cols - 5), cols], dtype=torch.int32)
    for seed in (0, 12345, 2**64 - 1):
        idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
        L.lsa_topk_approx(s.cuda(), ncols.cuda(), k, seed, idx)
        check_status_clean()
        want = np.stack([oracle.topk_approx(s[i:i + 1, : int(ncols[i])].numpy(), k, seed, row0=i)[0]
                         for i in range(rows)])
        assert np.array_equal(idx.cpu().numpy(), want), seed


def test_topk_nan_is_skipped_and_flagged():
    s = torch.tensor([[0.5, float("nan"), 2.0, 1.0]], device="cuda")
    idx = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    L.lsa_topk(s, None, 2, idx)
    torch.cuda.synchronize()
    code, flags = L.lsa_get_device_status(clear=True)
    assert code == L.LSA_ERR_NAN
    assert idx.cpu().tolist()[0] == [2, 3]


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("engine", ["tensor_core", "cuda_core"])
@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_sparse_decode_with_oracle_selection(name, splits, engine, monkeypatch):
    """Attention over the oracle's selection: the tensor-core kernels (GQA
    groups of 2..8 heads: the even split over the GPU without a split count,
    split-K with one) and the split-K CUDA-core kernel."""
    if engine == "cuda_core":
        monkeypatch.setenv("LSA_ATTENTION_PATH", "cuda_core")
    w = small(name)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    ref = oracle_decode(w, cpu)
    cache = L.make_cache(g["k_cache"], g["v_cache"])
    prm = L.make_params(w.batch, w.num_q_heads, cpu["max_blocks"], w.k_blocks, w.sink, w.recent,
                        w.softmax_scale, num_splits=splits)
    ws = torch.zeros(max(16, L.lsa_sparse_decode_workspace_size(cache, prm)), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.batch, w.num_q_heads, w.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device="cuda")
    sel = torch.from_numpy(ref["sel"]).cuda()
    L.lsa_sparse_decode(g["q"], cache, g["page_table"], g["seq_lens"], sel, prm, out, lse, ws)
    check_status_clean()
    assert_attention_close(out, ref["out"], name)
    assert_lse_close(lse, ref["lse"], name)


def compare_step_rows(st, w, cpu, reqs):
    """Checks requests `reqs` of a finished GpuStep against the oracle run on
    those requests alone (selection, then attention and lse)."""
    reqs = list(reqs)
    sub = subset(cpu, reqs) if len(reqs) != w.batch else cpu
    wr = w.replace(batch=len(reqs), seq_lens=tuple(sub["lens"]), seq_len_range=None)
    ref = oracle_decode(wr, sub)
    sel_gpu = st.idx.cpu().numpy()[reqs]
    # oracle scores for the tie rule
    use8 = w.c2f_candidates > 0
    ties = 0
    if not use8:
        oc = oracle_cache(sub)
        quest = w.summary_kind == 1
        osumm, _ = (oracle.quest_summaries if quest else oracle.summaries)(oc, sub["page_table"], sub["seq_lens"])
        sc = oracle.block_scores(sub["q"], oc, osumm, sub["page_table"], sub["seq_lens"], w.num_q_heads, w.sink,
                                 w.recent, summary_kind=w.summary_kind)
        S = f64(osumm)
        G = w.group
        for i in range(len(reqs)):
            for h in range(w.num_kv_heads):
                pg = np.maximum(sub["page_table"][i].cpu().numpy(), 0)
                qb = bits(sub["q"][i, h * G:(h + 1) * G])
                tau = (quest_score_bound(qb, S[pg, h, 0], S[pg, h, 1], w.dk) if quest
                       else score_bound(qb, S[pg, h], G, w.dk))
                kind = compare_selection(sel_gpu[i, h], ref["sel"][i, h], sc[i, h], tau)
                ties += kind == "tie"
    else:
        assert np.array_equal(sel_gpu, ref["sel"]), "fine token selection differs"
    out = st.out[reqs]
    lse = st.lse[reqs]
    if ties:
        # rows whose selection is an equally valid alternative (checked above):
        # the expected output is the oracle's attention on that selection
        ref = oracle.attend_selection(sub["q"], oracle_cache(sub), sub["page_table"], sub["seq_lens"], sel_gpu,
                                      num_q_heads=w.num_q_heads, sink=w.sink, recent=w.recent,
                                      scale=w.softmax_scale)
        print(f"{w.name}: {ties} epsilon-tie rows")
    err = assert_attention_close(out, ref["out"], w.name)
    assert_lse_close(lse, ref["lse"], w.name)
    return err


def run_and_compare_step(w, cpu, g, reqs=None, num_splits=0):
    st = GpuStep(w, g, num_splits)
    st.run()
    check_status_clean()
    return compare_step_rows(st, w, cpu, range(w.batch) if reqs is None else reqs)


@pytest.mark.parametrize("name", SMALL + ["c2f_small", "c2f_wrelu_small"] + QUEST)
def test_decode_step_end_to_end(name):
    w = small(name)
    cpu = make_inputs(w, "cpu")
    run_and_compare_step(w, cpu, to_dev(cpu))


def test_step_repeats_bit_identical():
    """Five calls on one workspace give identical bits (the counters the
    step needs at zero are left at zero by every call)."""
    w = small("b16_small")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    outs = []
    for _ in range(5):
        st.run()
        outs.append((st.idx.clone(), st.out.clone(), st.lse.clone()))
    check_status_clean()
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0])
        assert torch.equal(o[1].view(torch.int16), outs[0][1].view(torch.int16))
        assert torch.equal(o[2], outs[0][2])
    ref = oracle_decode(w, cpu)
    assert np.array_equal(outs[0][0].cpu().numpy(), ref["sel"])
    assert_attention_close(outs[0][1], ref["out"], "repeat")


def test_one_workspace_serves_different_inputs():
    """Two calls with different inputs on one workspace: the second equals a
    call on a fresh workspace (nothing of the first call is left behind)."""
    w = small("b16_small")
    ga = to_dev(make_inputs(w, "cpu"))
    gb = to_dev(make_inputs(w.replace(seed=w.seed + 7), "cpu"))
    st = GpuStep(w, ga)
    st.run()
    shared_ws = st.ws
    fresh = GpuStep(w, gb)
    fresh.run()
    again = GpuStep(w, gb)
    again.ws = shared_ws
    again.run()
    check_status_clean()
    assert torch.equal(again.idx, fresh.idx)
    assert torch.equal(again.out.view(torch.int16), fresh.out.view(torch.int16))
    assert torch.equal(again.lse, fresh.lse)


@pytest.mark.parametrize("splits", [1, 2, 5, 1000])
def test_decode_step_split_count_does_not_change_result(splits):
    w = small("ragged_small")
    cpu = make_inputs(w, "cpu")
    run_and_compare_step(w, cpu, to_dev(cpu), num_splits=splits)


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("lens", [(0, 1, 5), (16, 17, 31), (33, 47, 1000)])
def test_short_and_empty_requests(lens):
    w = small("b16_small", seq_lens=lens)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    st.run()
    check_status_clean()
    ref = oracle_decode(w, cpu)
    assert np.array_equal(st.idx.cpu().numpy(), ref["sel"])
    assert_attention_close(st.out, ref["out"], "short")
    assert_lse_close(st.lse, ref["lse"], "short")
    for r, Lr in enumerate(lens):
        if Lr == 0:
            assert torch.all(st.out[r].float() == 0) and torch.all(torch.isneginf(st.lse[r]))


@pytest.mark.parametrize("name", ["c2f_small", "c2f_wrelu_small"])
@pytest.mark.parametrize("lens,ncand,ntok", [((0, 30, 64 * 5, 64 * 20 + 5), 32, 512),
                                             ((64 * 40, 64 * 3 + 1, 64 * 9), 5, 100),
                                             ((64 * 70, 64 * 66), 64, 4096), ((64 * 300, 64 * 260), 256, 2048)])
def test_coarse_to_fine_short_requests_and_few_candidates(name, lens, ncand, ntok):
    """Requests with fewer full blocks than candidates or fewer tokens than
    the token budget, and candidate counts that leave most of a cluster's
    CTAs without a block (or give each the most it takes)."""
    w = small(name, seq_lens=lens, batch=len(lens), c2f_candidates=ncand, c2f_tokens=ntok)
    cpu = make_inputs(w, "cpu")
    run_and_compare_step(w, cpu, to_dev(cpu))


def test_topk_covering_all_blocks_equals_dense():
    lens = (4105, 3001, 777)
    w = small("b16_small", seq_lens=lens, k_blocks=300, sink=16, recent=25)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    st.run()
    check_status_clean()
    d = oracle.dense(cpu["q"], oracle_cache(cpu), cpu["page_table"], cpu["seq_lens"], num_q_heads=w.num_q_heads,
                     scale=w.softmax_scale)
    assert_attention_close(st.out, d["out"], "dense")
    assert_lse_close(st.lse, d["lse"], "dense")


def test_only_forced_tokens_when_k_is_zero():
    w = small("ragged_small", k_blocks=0)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    st.run()
    check_status_clean()
    ref = oracle_decode(w, cpu)
    assert_attention_close(st.out, ref["out"], "k=0")


def test_empty_batch_is_a_no_op():
    w = small("tiny")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    cache = L.make_cache(g["k_cache"], g["v_cache"])
    prm = L.make_params(0, w.num_q_heads, cpu["max_blocks"], w.k_blocks, w.sink, w.recent)
    out = torch.empty((1, 4, 64), dtype=torch.bfloat16, device="cuda")
    L.lsa_decode_step(g["q"], cache, g["k_cache"], None, g["page_table"], g["seq_lens"], prm, None, out, None, None)
    check_status_clean()


def test_vortex_figure2_shared_pages_gpu():
    gold = json.load(open(os.path.join(GOLD, "vortex_fig2_paged_layout.json")))
    P, H, b, d, Hq = gold["num_pages"], 2, 16, 64, 8
    gen = torch.Generator().manual_seed(21)
    k = torch.randn((P, H, b, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((P, H, b, d), generator=gen).to(torch.bfloat16)
    q = torch.randn((3, Hq, d), generator=gen).to(torch.bfloat16)
    pt = torch.tensor([gold["page_tables"][x] for x in ("x0", "x1", "x2")], dtype=torch.int32)
    lens = torch.tensor([48, 40, 47], dtype=torch.int32)
    kd, vd = k.cuda(), v.cuda()          # keep the device copies alive while the descriptor is used
    cache = L.make_cache(kd, vd)
    summ = torch.zeros((P, H, d), dtype=torch.bfloat16, device="cuda")
    L.lsa_build_summaries(cache, pt.cuda(), lens.cuda(), summ)
    prm = L.make_params(3, Hq, 3, 1, 16, 16, 0.2)
    ws = torch.zeros(max(16, L.lsa_decode_step_workspace_size(cache, prm)), dtype=torch.uint8, device="cuda")
    out = torch.empty((3, Hq, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((3, H, 1), dtype=torch.int32, device="cuda")
    qd, ptd, ld = q.cuda(), pt.cuda(), lens.cuda()
    L.lsa_decode_step(qd, cache, summ, None, ptd, ld, prm, idx, out, None, ws)
    check_status_clean()
    ref = oracle.decode(q, oracle.Cache(k, v), pt, lens, num_q_heads=Hq, k_blocks=1, sink=16, recent=16, scale=0.2)
    assert np.array_equal(idx.cpu().numpy(), ref["sel"])
    assert_attention_close(out, ref["out"], "fig2")


def test_bad_page_id_is_flagged_not_faulted():
    w = small("tiny")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    bad = g["page_table"].clone()
    bad[0, 5] = 10 ** 6          # out of range: the kernels check and skip it
    bad[0, 9] = -3
    g2 = dict(g, page_table=bad)
    st.g = g2
    st.run()
    torch.cuda.synchronize()
    code, flags = L.lsa_get_device_status(clear=True)
    assert code == L.LSA_ERR_BOUNDS
    assert torch.isfinite(st.out.float()).all()


def test_latent_cache_aliased_and_copied_values_agree():
    w = small("mla_small")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    assert g["v_cache"].data_ptr() == g["k_cache"].data_ptr()
    a = GpuStep(w, g)
    a.run()
    g2 = dict(g, v_cache=g["k_cache"][..., : w.dv].contiguous())
    b = GpuStep(w, g2)
    b.run()
    check_status_clean()
    assert torch.equal(a.idx, b.idx)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    ref = oracle_decode(w, cpu)
    assert_attention_close(b.out, ref["out"], "copied V")


# ---------------------------------------------------------------- coarse-to-fine

@pytest.mark.parametrize("name", ["c2f_small", "c2f_wrelu_small"])
def test_fine_topk_matches_oracle(name):
    """The fine pass alone (lsa_fine_topk) over the oracle's candidates: the
    head-sum score, and the weighted-ReLU indexer score on tensor cores."""
    w = small(name)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    ref = oracle_decode(w, cpu)
    ic = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
    prm = L.make_params(w.batch, w.num_q_heads, cpu["max_blocks"], 0, w.sink, w.recent, w.softmax_scale,
                        w.c2f_candidates, w.c2f_tokens, fine_head_weights=g.get("fine_weights"))
    cand = torch.from_numpy(ref["cand"]).cuda()
    tok = torch.empty((w.batch, 1, w.c2f_tokens), dtype=torch.int32, device="cuda")
    ws = torch.empty(w.batch * w.c2f_candidates * w.block_size * 4 + 256, dtype=torch.uint8, device="cuda")
    L.lsa_fine_topk(g["q"], ic, g["page_table"], g["seq_lens"], cand, prm, tok, ws)
    check_status_clean()
    assert np.array_equal(tok.cpu().numpy(), ref["sel"])
    # fine tokens lie inside the coarse candidates
    for r in range(w.batch):
        cs = set(ref["cand"][r, 0].tolist())
        assert all(t // w.block_size in cs for t in tok[r, 0].cpu().tolist() if t >= 0)


# ---------------------------------------------------------------- full-size workloads

FULL_CHUNK = {"b16_32k": 16, "b16_32k_quest": 16, "ragged": 8, "c2f": 4, "c2f_wrelu": 4, "mla": 2}


@pytest.mark.parametrize("name", ["b16_32k", "b16_32k_quest", "ragged", "c2f", "c2f_wrelu", "mla"])
def test_full_size_every_request(name):
    """Every request of the full-size workloads, from one call over the whole
    batch, checked against the oracle: the oracle runs on groups of requests
    (their pages gathered into a compact cache) so that its host copy stays
    small."""
    w = WORKLOADS[name]
    inp = make_inputs(w, "cuda")
    st = GpuStep(w, inp)
    st.run()
    check_status_clean()
    step = FULL_CHUNK[name]
    for r0 in range(0, w.batch, step):
        compare_step_rows(st, w, inp, list(range(r0, min(w.batch, r0 + step))))
