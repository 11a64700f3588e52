"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

  * number formats: torch's IEEE conversions and hand-worked closed forms;
  * the pages' worked examples (golden fixtures with citations);
  * brute force on tiny inputs with numpy (dense softmax attention, full
    argsort selection, einsum scores);
  * invariants: top-k covering every block equals dense attention; the
    selected set equals the first k of the stable argsort of the scores;
    log-sum-exp merge over any partition equals one pass; page permutation
    and page sharing do not change results; a constant V gives that V; the
    coarse block score is the mean of the fine token scores (linearity).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_inputs, small_workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- formats

def test_bf16_round_matches_torch_on_float_values():
    g = torch.Generator().manual_seed(5)
    x = torch.cat([
        torch.randn(20000, generator=g),
        torch.randn(2000, generator=g) * 1e-39,      # subnormal range
        torch.randn(2000, generator=g) * 1e37,
        torch.tensor([0.0, -0.0, 3.3895313892515355e38, -3.3895313892515355e38]),
    ]).to(torch.float32)
    want = bf16_bits(x.to(torch.bfloat16))
    got = np.array([oracle.bf16_round(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("x,bits", [
    (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # above the tie: single rounding
    (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    (2.0 ** -133, 0x0001),                     # smallest subnormal
    (2.0 ** -134, 0x0000),                     # tie between 0 and 2^-133 -> even
    (1.5 * 2.0 ** -133, 0x0002),               # tie -> even (up)
    ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),  # tie above the largest finite -> inf
    ((2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),  # largest finite
    (float("inf"), 0x7F80),
    (-float("inf"), 0xFF80),
])
def test_bf16_round_closed_forms(x, bits):
    assert oracle.bf16_round(x) == bits


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    # OCP E4M3: max normal 448, min normal 2^-6, min subnormal 2^-9, one = 0x38
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_decode(0x7F))


# ---------------------------------------------------------------- helpers

def tiny_inputs(**kw):
    w = WORKLOADS["tiny"].replace(**kw) if kw else WORKLOADS["tiny"]
    return w, make_inputs(w, "cpu")


def cache_of(inp, w):
    return oracle.Cache(inp["k_cache"], inp["v_cache"],
                        k8=inp.get("idx_keys"), k8_scale=inp.get("idx_scale"))


def np_dense(inp, w, r, hq, tokens=None):
    """Brute-force softmax attention (numpy fp64) of query head hq of
    request r over `tokens` (default: every token)."""
    b = w.block_size
    L = int(inp["lens"][r])
    toks = np.arange(L) if tokens is None else np.asarray(tokens)
    h = hq // w.group
    pt = inp["page_table"][r].numpy()
    K = f64(bf16_bits(inp["k_cache"][:, h]))      # [P, b, dk]
    V = f64(bf16_bits(inp["v_cache"][:, h].contiguous()))
    pages = pt[toks // b]
    Kt = K[pages, toks % b]                        # [n, dk]
    Vt = V[pages, toks % b]
    q = f64(bf16_bits(inp["q"][r, hq]))
    z = w.softmax_scale * (Kt @ q)
    m = z.max()
    p = np.exp(z - m)
    return (p @ Vt) / p.sum(), m + math.log(p.sum())


def assert_correctly_rounded(out_bits, exact):
    """Every bf16 output is a correct rounding of the fp64 value: within
    half a bf16 ulp (plus fp64 noise)."""
    got = f64(out_bits)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -126))) - 7)
    assert np.all(np.abs(got - exact) <= 0.5 * ulp * (1 + 1e-9) + 1e-300)


# ---------------------------------------------------------------- summaries

def test_summary_closed_forms():
    # keys of one block: x + d_t with sum_t d_t = 0  ->  mean = x exactly
    b, dk = 16, 8
    x = torch.tensor([1.5, -2.25, 0.0078125, 3.0, -0.5, 7.0, 1.0, -1.0])
    d = torch.linspace(-1, 1, b // 2).repeat_interleave(1)
    d = torch.cat([d, -d])
    k = (x[None, :] + d[:, None] * 0.25).to(torch.bfloat16).view(1, 1, b, dk)
    # the perturbations are symmetric and exactly representable
    assert torch.equal(k.float().mean(dim=2)[0, 0].to(torch.bfloat16).float(), x)
    c = oracle.Cache(k, k)
    s, valid = oracle.summaries(c, np.array([[0]], np.int32), np.array([16], np.int32))
    assert valid[0]
    assert np.array_equal(f64(s[0, 0]), x.numpy().astype(np.float64))


def test_summaries_vs_torch_when_mean_is_float_exact():
    # bf16 keys with one exponent (|x| in [1, 2)): the sum of 16 needs at
    # most 12 significant bits, so torch's fp32 mean is exact and its bf16
    # cast is a single correct rounding.
    g = torch.Generator().manual_seed(3)
    P, H, b, dk = 5, 2, 16, 32
    mag = 1.0 + torch.rand((P, H, b, dk), generator=g)
    sign = torch.where(torch.rand((P, H, b, dk), generator=g) < 0.5, -1.0, 1.0)
    k = (mag * sign).to(torch.bfloat16)
    c = oracle.Cache(k, k)
    pt = np.array([[0, 1, 2], [3, 4, -1]], np.int32)
    lens = np.array([48, 33], np.int32)
    s, valid = oracle.summaries(c, pt, lens)
    want = bf16_bits(k.float().mean(dim=2).to(torch.bfloat16))
    assert valid.tolist() == [True, True, True, True, True]  # page 4 has a full block (33 >= 32)
    assert np.array_equal(s, want)


def test_summaries_correctly_rounded_random():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    s, valid = oracle.summaries(c, inp["page_table"], inp["seq_lens"])
    K = f64(bf16_bits(inp["k_cache"]))                # [P, H, b, dk]
    exact = K.mean(axis=2)                              # fp64, exact for 16 addends here
    assert valid.all()
    assert_correctly_rounded(s, exact)


def test_summaries_only_full_blocks():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    lens = np.array([1000], np.int32)                   # 62 full blocks, tail of 8
    s, valid = oracle.summaries(c, inp["page_table"], lens)
    assert valid[:62].all() and not valid[62:].any()


# ---------------------------------------------------------------- scores + top-k

def test_topk_vortex_figure1_golden():
    gold = json.load(open(os.path.join(GOLD, "vortex_fig1_block_topk.json")))
    got = oracle.topk(np.array([gold["scores"]]), gold["k"])[0]
    assert got.tolist() == gold["selected_ascending"]


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(7)
    for n, k in [(1, 1), (5, 3), (64, 8), (300, 62), (1000, 1), (10, 20)]:
        s = rng.integers(-5, 5, size=n).astype(np.float64)     # many exact ties
        s[rng.random(n) < 0.1] = -np.inf                       # non-candidates
        order = np.lexsort((np.arange(n), -s))                 # score desc, index asc
        fin = [j for j in order if np.isfinite(s[j])][:k]
        want = sorted(fin) + [-1] * (k - len(fin))
        assert oracle.topk(s[None], k)[0].tolist() == want


def test_topk_negative_zero_ties_lower_index():
    s = np.array([[-0.0, 0.0, -0.0, -1.0]])
    assert oracle.topk(s, 2)[0].tolist() == [0, 1]


def test_block_scores_bruteforce_and_candidates():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    summ, _ = oracle.summaries(c, inp["page_table"], inp["seq_lens"])
    sc = oracle.block_scores(inp["q"], c, summ, inp["page_table"], inp["seq_lens"],
                             w.num_q_heads, w.sink, w.recent)
    S = f64(summ)[:, 0]                                  # [P, dk] (Hkv = 1)
    qs = f64(bf16_bits(inp["q"][0])).sum(axis=0)        # sum over the 4-head group
    want = S[inp["page_table"][0].numpy()] @ qs
    # sink 16 + recent 16 tokens, block 16: blocks 0 and 63 are forced
    assert np.isneginf(sc[0, 0, 0]) and np.isneginf(sc[0, 0, 63])
    assert np.allclose(sc[0, 0, 1:63], want[1:63], rtol=1e-12, atol=1e-12)
    # summaries computed from the keys on the fly give the same scores
    sc2 = oracle.block_scores(inp["q"], c, None, inp["page_table"], inp["seq_lens"],
                              w.num_q_heads, w.sink, w.recent)
    assert np.array_equal(sc, sc2)


def test_candidate_rule_ragged_forced_ranges():
    # block 64, sink 4, recent 512 and L = 1000: blocks touching [0,4) or
    # [488,1000) are forced; full blocks 1..6 are candidates (block 7 = 448..511
    # touches the recent range, block 15 is the partial tail).
    w = WORKLOADS["ragged"].replace(batch=1, seq_len_range=None, seq_lens=(1000,), name="x")
    inp = make_inputs(w, "cpu")
    c = cache_of(inp, w)
    sc = oracle.block_scores(inp["q"], c, None, inp["page_table"], inp["seq_lens"],
                             w.num_q_heads, w.sink, w.recent)
    finite = np.isfinite(sc[0, 0])
    assert np.flatnonzero(finite).tolist() == [1, 2, 3, 4, 5, 6]


# ---------------------------------------------------------------- attention

def test_decode_tiny_bruteforce_numpy():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"],
                        num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink,
                        recent=w.recent, scale=w.softmax_scale)
    # selection = first k of the stable argsort of the scores
    sc = oracle.block_scores(inp["q"], c, None, inp["page_table"], inp["seq_lens"],
                             w.num_q_heads, w.sink, w.recent)[0, 0]
    cand = np.flatnonzero(np.isfinite(sc))
    order = cand[np.lexsort((cand, -sc[cand]))]
    sel = sorted(order[: w.k_blocks].tolist())
    assert res["sel"][0, 0].tolist() == sel
    toks = list(range(16)) + [t for j in sel for t in range(j * 16, j * 16 + 16)] + \
        list(range(1024 - 16, 1024))
    for hq in range(w.num_q_heads):
        o, lse = np_dense(inp, w, 0, hq, toks)
        assert_correctly_rounded(res["out"][0, hq], o)
        assert abs(res["lse"][0, hq] - lse) < 1e-10


def test_dense_bruteforce_numpy():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    d = oracle.dense(inp["q"], c, inp["page_table"], inp["seq_lens"],
                     num_q_heads=w.num_q_heads, scale=w.softmax_scale)
    for hq in range(w.num_q_heads):
        o, lse = np_dense(inp, w, 0, hq)
        assert_correctly_rounded(d["out"][0, hq], o)
        assert abs(d["lse"][0, hq] - lse) < 1e-10


@pytest.mark.parametrize("name,lens", [
    ("tiny", (1024,)), ("b16_small", (4105, 3001, 777)), ("ragged_small", (4100, 900, 68, 4996, 2500)),
    ("mla_small", (3000, 1080))])
def test_topk_covering_all_blocks_equals_dense(name, lens):
    """With block-aligned forced ranges and k at least the number of
    candidates, the token set is every token: sparse equals dense."""
    w = small_workloads()[name]
    b = w.block_size
    resid = {L % b for L in lens}
    assert len(resid) == 1
    recent = resid.pop() + b          # L - recent is a block boundary for every request
    w = w.replace(k_blocks=100000, seq_lens=lens, seq_len_range=None, batch=len(lens),
                  sink=b, recent=recent)
    inp = make_inputs(w, "cpu")
    c = cache_of(inp, w)
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"],
                        num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink,
                        recent=w.recent, scale=w.softmax_scale)
    d = oracle.dense(inp["q"], c, inp["page_table"], inp["seq_lens"],
                     num_q_heads=w.num_q_heads, scale=w.softmax_scale)
    # same token set, different summation order: fp64 results agree to
    # ~1e-15, so the bf16 outputs are equal except at a rounding tie
    diff = np.abs(f64(res["out"]) - f64(d["out"]))
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(f64(d["out"])), 2.0 ** -126))) - 7)
    assert np.all(diff <= ulp)
    assert np.mean(res["out"] == d["out"]) > 0.999
    assert np.allclose(res["lse"], d["lse"], atol=1e-9)


def test_constant_v_gives_v_and_single_token():
    w, inp = tiny_inputs()
    v = torch.zeros_like(inp["v_cache"])
    vec = torch.randn(w.dv, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    v[:] = vec
    c = oracle.Cache(inp["k_cache"], v)
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"],
                        num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink,
                        recent=w.recent, scale=w.softmax_scale)
    assert np.array_equal(res["out"][0], np.tile(bf16_bits(vec), (w.num_q_heads, 1)))
    # a single-token cache attends V_0 with lse = scale * q.K_0
    c1 = cache_of(inp, w)
    one = oracle.decode(inp["q"], c1, inp["page_table"], np.array([1], np.int32),
                        num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink,
                        recent=w.recent, scale=w.softmax_scale)
    v0 = bf16_bits(inp["v_cache"][0, 0, 0])
    assert np.array_equal(one["out"][0], np.tile(v0, (w.num_q_heads, 1)))
    q = f64(bf16_bits(inp["q"][0]))
    k0 = f64(bf16_bits(inp["k_cache"][0, 0, 0]))
    assert np.allclose(one["lse"][0], w.softmax_scale * (q @ k0), atol=1e-12)


def test_empty_request():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    res = oracle.decode(inp["q"], c, inp["page_table"], np.array([0], np.int32),
                        num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink,
                        recent=w.recent, scale=w.softmax_scale)
    assert np.all(res["out"] == 0) and np.all(np.isneginf(res["lse"]))
    assert np.all(res["sel"] == -1)


def test_short_request_all_forced_equals_dense():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    lens = np.array([25], np.int32)      # L < sink + recent: every token forced
    res = oracle.decode(inp["q"], c, inp["page_table"], lens, num_q_heads=w.num_q_heads,
                        k_blocks=w.k_blocks, sink=w.sink, recent=w.recent, scale=w.softmax_scale)
    d = oracle.dense(inp["q"], c, inp["page_table"], lens, num_q_heads=w.num_q_heads,
                     scale=w.softmax_scale)
    assert np.array_equal(res["out"], d["out"])
    assert np.all(res["sel"] == -1)


def test_lse_merge_any_partition_equals_one_pass():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    rng = np.random.default_rng(0)
    q = f64(bf16_bits(inp["q"][0, 2]))
    toks = np.sort(rng.choice(1024, size=300, replace=False))
    ptr = inp["page_table"][0]
    o_all, l_all = oracle.attend_tokens(q, c, ptr, toks, 0, w.softmax_scale)
    for nparts in (1, 2, 5, 17):
        cuts = np.sort(rng.choice(np.arange(1, 300), size=nparts - 1, replace=False))
        parts = np.split(toks, cuts)
        os_, ls_ = zip(*[oracle.attend_tokens(q, c, ptr, p, 0, w.softmax_scale) for p in parts])
        o, l = oracle.lse_merge(np.stack(os_), np.array(ls_))
        assert np.allclose(o, o_all, rtol=1e-12, atol=1e-14)
        assert abs(l - l_all) < 1e-12
    # an empty part changes nothing
    o, l = oracle.lse_merge(np.stack([o_all, np.zeros_like(o_all)]), np.array([l_all, -np.inf]))
    assert np.allclose(o, o_all) and abs(l - l_all) < 1e-14


# ---------------------------------------------------------------- paging

def test_page_permutation_invariance():
    w = small_workloads()["b16_small"]
    inp = make_inputs(w, "cpu")
    c = cache_of(inp, w)
    args = dict(num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink, recent=w.recent,
                scale=w.softmax_scale)
    a = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], **args)
    P = inp["num_pages"]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    k2 = inp["k_cache"][perm]               # new page i holds old page perm[i]
    v2 = inp["v_cache"][perm]
    pt2 = inp["page_table"].clone()
    m = pt2 >= 0
    pt2[m] = inv[pt2[m].long()].to(torch.int32)
    b = oracle.decode(inp["q"], oracle.Cache(k2, v2), pt2, inp["seq_lens"], **args)
    for key in ("out", "lse", "sel"):
        assert np.array_equal(a[key], b[key])


def test_vortex_figure2_shared_pages():
    gold = json.load(open(os.path.join(GOLD, "vortex_fig2_paged_layout.json")))
    P, H, b, d, Hq = gold["num_pages"], 2, 16, 32, 4
    g = torch.Generator().manual_seed(21)
    k = torch.randn((P, H, b, d), generator=g).to(torch.bfloat16)
    v = torch.randn((P, H, b, d), generator=g).to(torch.bfloat16)
    q = torch.randn((3, Hq, d), generator=g).to(torch.bfloat16)
    pt = np.array([gold["page_tables"][x] for x in ("x0", "x1", "x2")], np.int32)
    lens = np.array([48, 40, 47], np.int32)
    args = dict(num_q_heads=Hq, k_blocks=1, sink=1, recent=9, scale=0.2)
    shared = oracle.decode(q, oracle.Cache(k, v), pt, lens, **args)
    s_shared, _ = oracle.summaries(oracle.Cache(k, v), pt, lens)
    for r in range(3):
        # private copy of request r's pages
        kp, vp = k[pt[r].tolist()], v[pt[r].tolist()]
        one = oracle.decode(q[r:r + 1], oracle.Cache(kp, vp), np.arange(3, dtype=np.int32)[None],
                            lens[r:r + 1], **args)
        assert np.array_equal(shared["out"][r], one["out"][0])
        assert np.array_equal(shared["sel"][r], one["sel"][0])
    # a shared page's summary is one value whoever references it
    s_priv, _ = oracle.summaries(oracle.Cache(k[[0, 3, 5]], v[[0, 3, 5]]),
                                 np.array([[0, 1, 2]], np.int32), np.array([48], np.int32))
    assert np.array_equal(s_shared[[0, 3, 5]], s_priv)


# ---------------------------------------------------------------- coarse-to-fine

def c2f_setup(**kw):
    w = small_workloads()["c2f_small"].replace(**kw)
    inp = make_inputs(w, "cpu")
    ic = oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])
    return w, inp, cache_of(inp, w), ic


def test_c2f_coarse_score_is_mean_of_fine_scores():
    w, inp, c, ic = c2f_setup()
    isumm, _ = oracle.summaries(ic, inp["page_table"], inp["seq_lens"], use_index_keys=True)
    sc = oracle.block_scores(inp["q"], ic, isumm, inp["page_table"], inp["seq_lens"],
                             w.num_q_heads, w.sink, w.recent, use_index_keys=True)
    qsum = f64(bf16_bits(inp["q"][0])).sum(axis=0)
    blocks = np.flatnonzero(np.isfinite(sc[0, 0]))[:40]
    f, t = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, 0, 0, blocks)
    fm = f.reshape(len(blocks), w.block_size).mean(axis=1)
    # difference only from rounding the mean key to bf16 (half an ulp per element)
    S = f64(isumm[inp["page_table"][0].numpy()[blocks], 0])
    bound = (np.abs(qsum)[None, :] * np.abs(S) * 2.0 ** -8).sum(axis=1) + 1e-9
    assert np.all(np.abs(sc[0, 0, blocks] - fm) <= bound)
    # and the fine scores are the dequantised dot products
    k8 = inp["idx_keys"].view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    sca = inp["idx_scale"].numpy().astype(np.float64)
    pg = inp["page_table"][0].numpy()[blocks]
    want = (k8[pg, 0] * sca[pg, 0][..., None]) @ qsum
    assert np.allclose(f, want.reshape(-1), rtol=1e-12, atol=1e-12)


def test_c2f_fine_tokens_inside_coarse_candidates():
    w, inp, c, ic = c2f_setup()
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"],
                        num_q_heads=w.num_q_heads, k_blocks=0, sink=w.sink, recent=w.recent,
                        scale=w.softmax_scale, index_cache=ic, c2f_candidates=w.c2f_candidates,
                        c2f_tokens=w.c2f_tokens)
    for r in range(w.batch):
        cand = set(res["cand"][r, 0][res["cand"][r, 0] >= 0].tolist())
        toks = res["sel"][r, 0][res["sel"][r, 0] >= 0]
        assert len(toks) == min(w.c2f_tokens, len(cand) * w.block_size)
        assert all((t // w.block_size) in cand for t in toks.tolist())
        assert np.all(np.diff(toks) > 0)


def test_c2f_all_blocks_is_exact_token_topk():
    w, inp, c, ic = c2f_setup(seq_lens=(2000, 1500), recent=0, c2f_candidates=1000,
                              c2f_tokens=300)
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"],
                        num_q_heads=w.num_q_heads, k_blocks=0, sink=0, recent=0,
                        scale=w.softmax_scale, index_cache=ic, c2f_candidates=w.c2f_candidates,
                        c2f_tokens=w.c2f_tokens)
    k8 = inp["idx_keys"].view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    sca = inp["idx_scale"].numpy().astype(np.float64)
    b = w.block_size
    for r in range(w.batch):
        L = inp["lens"][r]
        nfull = L // b
        toks = np.arange(nfull * b)
        pg = inp["page_table"][r].numpy()[toks // b]
        qsum = f64(bf16_bits(inp["q"][r])).sum(axis=0)
        f = (k8[pg, 0, toks % b] * sca[pg, 0, toks % b][:, None]) @ qsum
        order = np.lexsort((toks, -f))
        want = np.sort(toks[order[: w.c2f_tokens]])
        assert np.array_equal(res["sel"][r, 0], want)
        for hq in (0, 63):
            o, lse = np_dense(inp, w, r, hq, want)
            assert_correctly_rounded(res["out"][r, hq], o)


# ---------------------------------------------------------------- latent cache

def test_mla_aliased_v_equals_copied_v():
    w = small_workloads()["mla_small"].replace(seq_lens=(3000, 1100))
    inp = make_inputs(w, "cpu")
    assert inp["v_cache"].data_ptr() == inp["k_cache"].data_ptr()
    c_alias = oracle.Cache(inp["k_cache"], None, dv=w.dv)
    c_copy = oracle.Cache(inp["k_cache"], inp["k_cache"][..., : w.dv].clone())
    args = dict(num_q_heads=w.num_q_heads, k_blocks=w.k_blocks, sink=w.sink, recent=w.recent,
                scale=w.softmax_scale)
    a = oracle.decode(inp["q"], c_alias, inp["page_table"], inp["seq_lens"], **args)
    b = oracle.decode(inp["q"], c_copy, inp["page_table"], inp["seq_lens"], **args)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["sel"], b["sel"])


def test_mla_decode_bruteforce_numpy():
    """The latent cache with dk = 576 keys and dv = 512 values (the first 512
    key dims): the selection is the top-k of numpy scores over the candidate
    blocks, and every output head is the correctly rounded brute-force
    softmax over the forced tokens plus the selected blocks, with values read
    from the first dv dims (a value read with the key's width, or at the
    wrong offset, fails here)."""
    w = small_workloads()["mla_small"].replace(seq_lens=(3000, 1100))
    inp = make_inputs(w, "cpu")
    c = oracle.Cache(inp["k_cache"], None, dv=w.dv)
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], num_q_heads=w.num_q_heads,
                        k_blocks=w.k_blocks, sink=w.sink, recent=w.recent, scale=w.softmax_scale)
    assert res["out"].shape == (w.batch, w.num_q_heads, w.dv)
    summ, _ = oracle.summaries(c, inp["page_table"], inp["seq_lens"])
    S = f64(summ)[:, 0]                                   # [P, 576] (one latent head)
    b = w.block_size
    for r in range(w.batch):
        L = int(inp["lens"][r])
        se = min(w.sink, L)
        rs = max(L - w.recent, se)
        pt = inp["page_table"][r].numpy()
        qs = f64(bf16_bits(inp["q"][r])).sum(axis=0)     # the 64 heads share one latent head
        cand = np.array([j for j in range(L // b) if j * b >= se and (j + 1) * b <= rs])
        sc = S[pt[cand]] @ qs
        order = np.lexsort((cand, -sc))
        want = np.sort(cand[order[: w.k_blocks]])
        got = res["sel"][r, 0]
        assert np.array_equal(got[got >= 0], want)
        toks = sorted(set(range(se)) | set(range(rs, L)) |
                      {t for j in want.tolist() for t in range(j * b, (j + 1) * b)})
        for hq in (0, 17, 40, 63):
            o, lse = np_dense(inp, w, r, hq, toks)
            assert o.shape == (w.dv,)
            assert_correctly_rounded(res["out"][r, hq], o)
            assert abs(res["lse"][r, hq] - lse) <= 1e-10 * max(1.0, abs(lse))


def test_attend_selection_reproduces_decode_and_dense():
    w, inp = tiny_inputs()
    c = cache_of(inp, w)
    args = dict(num_q_heads=w.num_q_heads, sink=w.sink, recent=w.recent, scale=w.softmax_scale)
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], k_blocks=w.k_blocks, **args)
    a = oracle.attend_selection(inp["q"], c, inp["page_table"], inp["seq_lens"], res["sel"], **args)
    assert np.array_equal(a["out"], res["out"]) and np.array_equal(a["lse"], res["lse"])
    # every candidate block selected (block-aligned forced ranges) = dense
    allc = np.arange(1, 63, dtype=np.int32)[None, None]
    a = oracle.attend_selection(inp["q"], c, inp["page_table"], inp["seq_lens"], allc, **args)
    d = oracle.dense(inp["q"], c, inp["page_table"], inp["seq_lens"], num_q_heads=w.num_q_heads,
                     scale=w.softmax_scale)
    assert np.allclose(a["lse"], d["lse"], atol=1e-12)
    # invalid entries (forced block, out of range, repeated) are skipped
    junk = np.array([[[0, 5, 5, 63, 200, -1]]], dtype=np.int32)
    one = np.array([[[5]]], dtype=np.int32)
    x = oracle.attend_selection(inp["q"], c, inp["page_table"], inp["seq_lens"], junk, **args)
    y = oracle.attend_selection(inp["q"], c, inp["page_table"], inp["seq_lens"], one, **args)
    assert np.array_equal(x["out"], y["out"])


# ---------------------------------------------------------------- Quest min/max summaries

def quest_setup(lens=(1000, 333)):
    w = small_workloads()["b16_small"].replace(batch=len(lens), seq_lens=tuple(lens), name="quest")
    inp = make_inputs(w, "cpu")
    return w, inp, cache_of(inp, w)


def test_quest_summaries_are_the_blocks_max_and_min():
    """Quest keeps each block's element-wise maximum and minimum keys
    (Vortex blog post, end of "Why Long Generations Are Expensive"): numpy's
    max / min over the block's tokens, exactly, for full blocks only."""
    w, inp, c = quest_setup()
    qs, valid = oracle.quest_summaries(c, inp["page_table"], inp["seq_lens"])
    K = f64(bf16_bits(inp["k_cache"]))                       # [P, H, b, dk]
    full = set()
    for r, L in enumerate(inp["lens"]):
        full |= set(inp["page_table"][r, : L // w.block_size].tolist())
    assert set(np.flatnonzero(valid).tolist()) == full
    for p in sorted(full):
        assert np.array_equal(f64(qs[p, :, 0]), K[p].max(axis=1))
        assert np.array_equal(f64(qs[p, :, 1]), K[p].min(axis=1))
    assert np.all(qs[~valid] == 0)


def test_quest_score_bounds_every_token_of_the_block():
    """The Quest score of a block is an upper bound on q_g . k_t for every
    query head g of the group and every token t of the block (brute force),
    and the maximum over heads is taken: lowering one head's bound below the
    true maximum would fail here."""
    w, inp, c = quest_setup()
    qs, _ = oracle.quest_summaries(c, inp["page_table"], inp["seq_lens"])
    sc = oracle.block_scores(inp["q"], c, qs, inp["page_table"], inp["seq_lens"], w.num_q_heads, w.sink,
                             w.recent, summary_kind=1)
    K = f64(bf16_bits(inp["k_cache"]))
    G, b = w.group, w.block_size
    checked = 0
    for r in range(w.batch):
        pt = inp["page_table"][r].numpy()
        for h in range(w.num_kv_heads):
            Q = f64(bf16_bits(inp["q"][r, h * G:(h + 1) * G]))   # [G, dk]
            for j in np.flatnonzero(np.isfinite(sc[r, h])):
                true_max = (Q @ K[pt[j], h].T).max()                 # over heads and tokens
                assert sc[r, h, j] >= true_max - 1e-9 * abs(true_max)
                checked += 1
            # forced and tail blocks are not candidates
            L = inp["lens"][r]
            assert np.isneginf(sc[r, h, 0]) and np.isneginf(sc[r, h, (L - 1) // b])
    assert checked > 100


def test_quest_score_is_tight_on_a_block_of_equal_keys():
    """A block whose tokens all hold the same key x has max = min = x, so its
    bound is max_g q_g . x exactly; with a query whose coordinates are all
    positive the bound is q . max (and q . min for all negative)."""
    w, inp, _ = quest_setup(lens=(800,))
    b = w.block_size
    pt = inp["page_table"][0]
    k = inp["k_cache"].clone()
    k[pt[5], :, :] = k[pt[5], :, :1].expand(-1, b, -1)          # block 5: one key repeated
    inp2 = dict(inp, k_cache=k)
    c = cache_of(inp2, w)
    sc = oracle.block_scores(inp["q"], c, None, inp["page_table"], inp["seq_lens"], w.num_q_heads, w.sink,
                             w.recent, summary_kind=1)
    G = w.group
    K = f64(bf16_bits(k))
    for h in range(w.num_kv_heads):
        Q = f64(bf16_bits(inp["q"][0, h * G:(h + 1) * G]))
        assert sc[0, h, 5] == pytest.approx((Q @ K[pt[5], h, 0]).max(), rel=1e-12, abs=1e-12)
    # a positive query scores q . max; a negative one q . min
    q = torch.full_like(inp["q"], 0.5)
    qs, _ = oracle.quest_summaries(c, inp["page_table"], inp["seq_lens"])
    sp = oracle.block_scores(q, c, qs, inp["page_table"], inp["seq_lens"], w.num_q_heads, w.sink, w.recent,
                             summary_kind=1)
    sn = oracle.block_scores(-q, c, qs, inp["page_table"], inp["seq_lens"], w.num_q_heads, w.sink, w.recent,
                             summary_kind=1)
    S = f64(qs)
    for j in (2, 7, 30):
        for h in range(w.num_kv_heads):
            assert sp[0, h, j] == pytest.approx(0.5 * S[pt[j], h, 0].sum(), rel=1e-12)
            assert sn[0, h, j] == pytest.approx(-0.5 * S[pt[j], h, 1].sum(), rel=1e-12)


def test_quest_decode_selects_the_top_bounds_and_attends_them():
    w, inp, c = quest_setup(lens=(4096, 3001))
    qs, _ = oracle.quest_summaries(c, inp["page_table"], inp["seq_lens"])
    args = dict(num_q_heads=w.num_q_heads, sink=w.sink, recent=w.recent, scale=w.softmax_scale)
    res = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], k_blocks=w.k_blocks, summ=qs,
                        summary_kind=1, **args)
    sc = oracle.block_scores(inp["q"], c, qs, inp["page_table"], inp["seq_lens"], w.num_q_heads, w.sink,
                             w.recent, summary_kind=1)
    for r in range(w.batch):
        for h in range(w.num_kv_heads):
            cand = np.flatnonzero(np.isfinite(sc[r, h]))
            order = np.lexsort((cand, -sc[r, h, cand]))
            want = np.sort(cand[order[: w.k_blocks]])
            got = res["sel"][r, h]
            assert np.array_equal(got[got >= 0], want)
    a = oracle.attend_selection(inp["q"], c, inp["page_table"], inp["seq_lens"], res["sel"], **args)
    assert np.array_equal(a["out"], res["out"])
    # the mean-key selection differs on these inputs (the two scores rank differently)
    m = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], k_blocks=w.k_blocks, **args)
    assert not np.array_equal(m["sel"], res["sel"])


# ---------------------------------------------------------------- weighted-ReLU fine score

def wrelu_setup(positive_q=False, positive_k=False):
    w, inp, c, ic = c2f_setup(seq_lens=(2000, 1500), recent=0, c2f_candidates=6, c2f_tokens=100)
    if positive_q:
        inp["q"] = inp["q"].abs()
    if positive_k:
        k8 = inp["idx_keys"].view(torch.float8_e4m3fn).float().abs().to(torch.float8_e4m3fn)
        inp["idx_keys"] = k8.view(torch.uint8)
        ic = oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])
    return w, inp, ic


def test_weighted_relu_reduces_to_the_head_sum_when_every_dot_is_positive():
    """LeanSparse Eq. 6's aggregation on exact keys, sum_g w_g ReLU(q_g . k_t):
    with all-positive queries and keys every dot is positive, so with unit
    weights it equals the plain head-sum fine score (scale_t sum_g q_g .
    e4m3(k8_t)), which the coarse-score pin ties to the summaries."""
    w, inp, ic = wrelu_setup(positive_q=True, positive_k=True)
    ones = np.ones((w.batch, w.num_q_heads), dtype=np.float32)
    blocks = np.array([3, 7, 11], dtype=np.int64)
    for r in range(w.batch):
        f1, t1 = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, r, 0, blocks, fine_weights=ones)
        f0, t0 = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, r, 0, blocks)
        assert np.array_equal(t1, t0)
        assert np.all(f0 > 0)
        assert np.allclose(f1, f0, rtol=1e-12, atol=0)


def test_weighted_relu_negative_dots_contribute_nothing():
    """All-negative queries against all-positive keys: every dot is below
    zero, every head's ReLU is 0, so every fine score is 0 and the token
    top-k (ties to the lower token) takes the first candidate tokens."""
    w, inp, ic = wrelu_setup(positive_k=True)
    inp["q"] = -inp["q"].abs()
    wts = np.random.default_rng(3).uniform(0.1, 1.0, (w.batch, w.num_q_heads)).astype(np.float32)
    f, t = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, 0, 0, np.array([2, 9], np.int64),
                              fine_weights=wts)
    assert np.all(f == 0.0)
    res = oracle.decode(inp["q"], oracle.Cache(inp["k_cache"], inp["v_cache"]), inp["page_table"], inp["seq_lens"],
                        num_q_heads=w.num_q_heads, k_blocks=0, sink=0, recent=0, scale=w.softmax_scale,
                        index_cache=ic, c2f_candidates=w.c2f_candidates, c2f_tokens=w.c2f_tokens,
                        fine_weights=wts)
    for r in range(w.batch):
        cand = np.sort(res["cand"][r, 0][res["cand"][r, 0] >= 0])
        toks = np.concatenate([np.arange(j * w.block_size, (j + 1) * w.block_size) for j in cand])
        assert np.array_equal(res["sel"][r, 0], np.sort(toks)[: w.c2f_tokens])


def test_weighted_relu_is_linear_in_the_weights_and_each_weight_picks_its_head():
    """f(a w1 + b w2) = a f(w1) + b f(w2); a weight on head g alone gives
    w_g ReLU(q_g . k_t) (numpy over the decoded keys), so a weight applied
    to the wrong head, or a ReLU taken after the sum, fails here."""
    w, inp, ic = wrelu_setup()
    rng = np.random.default_rng(5)
    # weights on a 1/256 grid: 2 w1 + 3 w2 is then exact in float32
    w1 = (rng.integers(0, 256, (w.batch, w.num_q_heads)) / 256.0).astype(np.float32)
    w2 = (rng.integers(0, 256, (w.batch, w.num_q_heads)) / 256.0).astype(np.float32)
    blocks = np.array([1, 4], dtype=np.int64)
    args = (inp["q"], ic, inp["page_table"], w.num_q_heads, 1, 0, blocks)
    fa, _ = oracle.fine_scores(*args, fine_weights=w1)
    fb, _ = oracle.fine_scores(*args, fine_weights=w2)
    fab, _ = oracle.fine_scores(*args, fine_weights=(2 * w1 + 3 * w2).astype(np.float32))
    assert np.allclose(fab, 2 * fa + 3 * fb, rtol=1e-10, atol=1e-9)
    K8 = inp["idx_keys"].view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    S = inp["idx_scale"].numpy().astype(np.float64)
    b = w.block_size
    pt = inp["page_table"][1].numpy()
    toks = np.concatenate([np.arange(j * b, (j + 1) * b) for j in blocks])
    kt = K8[pt[toks // b], 0, toks % b] * S[pt[toks // b], 0, toks % b][:, None]
    for g in (0, 17, 63):
        one = np.zeros((w.batch, w.num_q_heads), dtype=np.float32)
        one[1, g] = 2.5
        fg, _ = oracle.fine_scores(*args, fine_weights=one)
        qg = f64(bf16_bits(inp["q"][1, g]))
        assert np.allclose(fg, 2.5 * np.maximum(kt @ qg, 0.0), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- approximate top-k (stochastic early exit)

def test_splitmix64_published_vectors():
    gold = json.load(open(os.path.join(GOLD, "splitmix64_vectors.json")))
    for v in gold["vectors"]:
        for n, want in enumerate(v["outputs"], start=1):
            assert oracle.splitmix64(v["seed"], n) == int(want, 0)


def _approx_invariants(s, k, sel):
    """What any approximate selection of this kind must satisfy: keff
    entries, ascending, candidates only, and no unselected candidate above a
    selected one by more than one bucket width (plus the remap's rounding)."""
    cand = ~np.isnan(s) & (s != -np.inf)
    m = int(cand.sum())
    keff = min(k, m)
    chosen = sel[sel >= 0]
    assert len(chosen) == keff and np.all(sel[keff:] == -1)
    assert np.all(np.diff(chosen) > 0) and np.all(cand[chosen])
    if 0 < keff < m:
        vals = s[cand].astype(np.float64)
        width = (vals.max() - vals.min()) / 2048
        rest = np.setdiff1d(np.flatnonzero(cand), chosen)
        assert s[rest].max() <= s[chosen].min() + width * (1 + 1e-4) + 1e-30


@pytest.mark.parametrize("seed", [0, 1, 99, 2**63 + 5])
def test_topk_approx_equals_exact_when_every_bucket_holds_one_key(seed):
    """Distinct values spread one per bucket: the boundary bucket holds one
    key, which the sample must take, so the result is the exact top-k."""
    n = 2048
    gen = np.random.default_rng(3)
    s = gen.permutation(n).astype(np.float32)
    for k in (1, 62, 300, 2047):
        got = oracle.topk_approx(s[None], k, seed)[0]
        assert np.array_equal(got, oracle.topk(s[None], k)[0])


def test_topk_approx_invariants_random_and_clustered_rows():
    gen = np.random.default_rng(11)
    rows = [gen.standard_normal(5000).astype(np.float32),
            (gen.integers(-30, 30, 4096) / 4).astype(np.float32),                   # heavy ties
            np.concatenate([gen.standard_normal(3000), 50 + gen.standard_normal(40)]).astype(np.float32),
            np.where(gen.random(3000) < 0.4, -np.inf, gen.standard_normal(3000)).astype(np.float32)]
    for s in rows:
        for k in (1, 30, 256, 2000):
            for seed in (0, 7):
                _approx_invariants(s, k, oracle.topk_approx(s[None], k, seed)[0])


def test_topk_approx_all_candidates_empty_and_nan():
    s = np.array([[1.0, np.nan, -np.inf, 3.0, 2.0]], dtype=np.float32)
    assert oracle.topk_approx(s, 5, 1).tolist() == [[0, 3, 4, -1, -1]]
    assert oracle.topk_approx(s, 3, 1).tolist() == [[0, 3, 4]]
    assert oracle.topk_approx(s, 0, 1).shape == (1, 0)
    assert oracle.topk_approx(np.full((1, 4), -np.inf, np.float32), 2, 1).tolist() == [[-1, -1]]


def test_topk_approx_confident_winners_are_kept_and_the_rest_is_a_circular_window():
    """h well-separated high values above a run of equal values: the high
    ones are always taken, and the k - h others form a circular run of the
    equal ones in column order, whose start moves with the seed."""
    n, h, k = 1000, 7, 50
    s = np.zeros(n, np.float32)
    hi = np.array([13, 200, 201, 555, 700, 901, 999])
    s[hi] = 1000 + np.arange(h) * 100
    starts = set()
    low = np.setdiff1d(np.arange(n), hi)
    for seed in range(40):
        got = oracle.topk_approx(s[None], k, seed)[0]
        assert set(hi) <= set(got.tolist())
        rest = np.setdiff1d(got, hi)
        pos = np.searchsorted(low, rest)          # numbers 0 .. len(low)-1 in column order
        assert len(pos) == k - h
        gaps = np.diff(np.concatenate([pos, [pos[0] + len(low)]]))
        assert np.sum(gaps != 1) == 1             # one circular run
        starts.add(int(pos[(int(np.argmax(gaps != 1)) + 1) % len(pos)]))
    assert len(starts) > 30


def test_topk_approx_samples_the_boundary_bucket_uniformly():
    """Over many seeds every key of the crowded boundary bucket is taken
    with probability take / cnt (a binomial bound), and nothing below it."""
    n, k = 400, 100
    s = np.zeros(n, np.float32)
    s[:60] = 10 + np.arange(60, dtype=np.float32)      # 60 confident winners
    s[60:160] = 5.0                                    # boundary bucket: 100 equal keys, 40 taken
    s[160:] = -5.0 - np.arange(n - 160, dtype=np.float32) / 1000
    trials = 2000
    freq = np.zeros(n)
    for seed in range(trials):
        got = oracle.topk_approx(s[None], k, seed * 7919 + 1)[0]
        freq[got] += 1
    assert np.all(freq[:60] == trials) and np.all(freq[160:] == 0)
    p = 40 / 100
    sd = math.sqrt(trials * p * (1 - p))
    assert np.all(np.abs(freq[60:160] - trials * p) < 5 * sd)


# ---------------------------------------------------------------- PQ32 coarse scores and the miss filter

def pq_setup(**kw):
    w = small_workloads()["c2f_pq_small"].replace(**kw)
    inp = make_inputs(w, "cpu")
    ic = oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])
    return w, inp, ic


def lossless_pq(inp, seed=0):
    """Rewrites the index keys as their codes' centroids exactly: centroids
    drawn from values exact in e4m3 and bf16, keys = e4m3(centroid), scale 1."""
    rng = np.random.default_rng(seed)
    vals = np.array([-4, -3, -2, -1.5, -1, -0.5, 0, 0.5, 1, 1.5, 2, 3, 4], dtype=np.float32)
    cb = torch.from_numpy(rng.choice(vals, (32, 256, 4))).to(torch.bfloat16)
    codes = inp["pq_codes"].long()
    P, H, b, _ = codes.shape
    keys = cb.float()[torch.arange(32), codes].reshape(P, H, b, 128)
    inp["pq_codebook"] = cb
    inp["idx_keys"] = keys.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    inp["idx_scale"] = torch.ones((P, H, b), dtype=torch.float32)
    return oracle.Cache(None, None, k8=inp["idx_keys"], k8_scale=inp["idx_scale"])


def test_pq_score_with_lossless_codes_is_the_exact_indexer_score():
    """When every key's subvectors are exactly its codes' centroids, Eq. 6's
    PQ score equals the exact weighted-ReLU score of the FP8 key (the fine
    score, a separate function pinned above): a wrong subspace offset,
    centroid index, weight or a ReLU outside the head sum fails here."""
    w, inp, ic = pq_setup(seq_lens=(640, 300))
    ic = lossless_pq(inp)
    b = w.block_size
    for r in (0, 1):
        for blk in (0, 3):
            f, _ = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, r, 0,
                                      np.array([blk]), fine_weights=inp["fine_weights"])
            s = oracle.pq_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, inp["fine_weights"],
                                 inp["pq_codes"], inp["pq_codebook"], r, 0, blk * b, b)
            assert np.allclose(s, f, rtol=1e-12, atol=1e-9)


def test_pq_score_relu_and_weights():
    """All-positive queries against all-negative centroids: every head's dot
    is negative, so the score is 0; flipping the centroids' sign gives the
    weighted sum of the heads' dots (linear in the weights)."""
    w, inp, ic = pq_setup(seq_lens=(640, 300))
    inp["q"] = inp["q"].abs()
    cb = inp["pq_codebook"].float().abs().to(torch.bfloat16)
    b = w.block_size
    args = (inp["q"], ic, inp["page_table"], w.num_q_heads)
    neg = oracle.pq_scores(*args, inp["fine_weights"], inp["pq_codes"], (-cb.float()).to(torch.bfloat16), 0, 0, 0, b)
    assert np.all(neg == 0.0)
    pos = oracle.pq_scores(*args, inp["fine_weights"], inp["pq_codes"], cb, 0, 0, 0, b)
    w2 = (inp["fine_weights"] * 2.0).contiguous()
    pos2 = oracle.pq_scores(*args, w2, inp["pq_codes"], cb, 0, 0, 0, b)
    assert np.all(pos > 0) and np.allclose(pos2, 2 * pos, rtol=1e-12)


def test_pq_encode_picks_the_nearest_centroid():
    """Keys equal to a centroid get it back (the lowest index among equal
    centroids); random keys get a centroid at the smallest fp64 distance up
    to fp32 rounding."""
    w, inp, ic = pq_setup(seq_lens=(640, 300))
    b = w.block_size
    slots = np.arange(0, 40, dtype=np.int64)     # tokens of page 0 (one KV head)
    got = oracle.pq_encode(ic, inp["pq_codebook"], slots)
    K8 = inp["idx_keys"].view(torch.float8_e4m3fn).float().numpy().astype(np.float64).reshape(-1, 128)
    S = inp["idx_scale"].numpy().astype(np.float64).reshape(-1)
    cb = inp["pq_codebook"].float().numpy().astype(np.float64)
    for i, s in enumerate(slots):
        k = (K8[s] * S[s]).reshape(32, 4)
        d = ((cb - k[:, None, :]) ** 2).sum(-1)          # [32, 256]
        dmin = d.min(axis=1)
        chosen = d[np.arange(32), got[i]]
        assert np.all(chosen <= dmin * (1 + 1e-5) + 1e-6)
    ic2 = lossless_pq(inp, seed=3)
    cbl = inp["pq_codebook"].float().numpy()
    got2 = oracle.pq_encode(ic2, inp["pq_codebook"], slots)
    codes = inp["pq_codes"].numpy().reshape(-1, 32)
    for i, s in enumerate(slots):
        for j in range(32):
            same = np.flatnonzero((cbl[j] == cbl[j, codes[s, j]]).all(axis=1))
            assert got2[i, j] == same[0]


def test_miss_filter_closed_form():
    """Hits stay; a miss stays only at or above the k-th largest coarse score
    minus one sample standard deviation (numpy's, ddof=1)."""
    s = np.array([10.0, 9.0, 8.0, 1.0, 0.0, 4.0])
    hit = np.array([0, 0, 0, 0, 1, 0])
    keep, tau = oracle.miss_filter(s, hit, 2)
    assert tau == pytest.approx(9.0 - np.std(s, ddof=1), rel=1e-14)
    assert keep.tolist() == [True, True, True, False, True, False]
    keep, tau = oracle.miss_filter(s, np.zeros(6), 6)      # no k-th largest: everything kept
    assert keep.all() and tau == -math.inf
    keep, _ = oracle.miss_filter(s, np.ones(6), 1)         # all hits
    assert keep.all()


def _pq_args(w, inp, ic, **kw):
    a = dict(num_q_heads=w.num_q_heads, sink=w.sink, recent=w.recent, fine_weights=inp["fine_weights"],
             pq_codes=inp["pq_codes"], pq_codebook=inp["pq_codebook"], pq_hit=inp["pq_hit"],
             pq_candidates=w.pq_candidates, tokens=w.c2f_tokens)
    a.update(kw)
    return a


def _exact_topk_all_tokens(w, inp, ic, r, k):
    """Brute force: the exact weighted-ReLU top-k over every full block's
    tokens and the partial last block's tokens (no forced ranges)."""
    b = w.block_size
    L = int(inp["seq_lens"][r])
    nblk = (L + b - 1) // b
    f, t = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, r, 0,
                              np.arange(nblk), fine_weights=inp["fine_weights"])
    f = np.where(t < L, f, -np.inf)
    return oracle.topk(f[None], k)[0]


def test_pq_select_every_token_a_cached_candidate_is_the_exact_topk():
    """With C at least every encoded token and every key cached, the coarse
    pass keeps everything and the selection is the exact top-k over all
    tokens (the coarse-to-fine claim with no approximation left)."""
    w, inp, ic = pq_setup(seq_lens=(640 + 21, 300), recent=0)
    for r in (0, 1):
        got = oracle.pq_select(inp["q"], ic, inp["page_table"], inp["seq_lens"],
                               **_pq_args(w, inp, ic, pq_hit=None, pq_candidates=700, tokens=50), r=r, h=0)
        assert np.array_equal(got["sel"], _exact_topk_all_tokens(w, inp, ic, r, 50))
        assert got["kept"][got["cand"] >= 0].all()


def test_pq_select_lossless_codes_coarse_is_exact():
    """Lossless codes make the coarse score exact: the C candidates are the
    exact top-C of the encoded tokens, and with C = k and every key cached
    the selection is the exact top-k over the candidates and the tail."""
    w, inp, ic = pq_setup(seq_lens=(640 + 21, 300), recent=0)
    ic = lossless_pq(inp, seed=1)
    b = w.block_size
    for r in (0, 1):
        L = int(inp["seq_lens"][r])
        nfull = L // b
        f, t = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, r, 0, np.arange(nfull),
                                  fine_weights=inp["fine_weights"])
        got = oracle.pq_select(inp["q"], ic, inp["page_table"], inp["seq_lens"],
                               **_pq_args(w, inp, ic, pq_hit=None, pq_candidates=60, tokens=60), r=r, h=0)
        assert np.array_equal(got["cand"], oracle.topk(f[None], 60)[0])
        tail = np.arange(nfull * b, L)
        ft, tt = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, r, 0,
                                    np.array([nfull]) if L % b else np.zeros(0, np.int64),
                                    fine_weights=inp["fine_weights"])
        pool = np.concatenate([got["cand"], tail])
        fpool = np.concatenate([f[got["cand"]], ft[: len(tail)]])
        order = sorted(range(len(pool)), key=lambda i: (-fpool[i], pool[i]))[:60]
        assert np.array_equal(got["sel"], np.sort(pool[order]))


def test_pq_select_filter_and_final_tokens():
    """The kept candidates are exactly the hits and the misses at or above
    the threshold; the final tokens are kept candidates or tail tokens."""
    w, inp, ic = pq_setup()
    b = w.block_size
    for r in (0, 1):
        L = int(inp["seq_lens"][r])
        got = oracle.pq_select(inp["q"], ic, inp["page_table"], inp["seq_lens"], **_pq_args(w, inp, ic), r=r, h=0)
        cand = got["cand"][got["cand"] >= 0]
        pt = inp["page_table"][r].numpy()
        hit = inp["pq_hit"].numpy()[pt[cand // b], 0, cand % b].astype(bool)
        s = np.concatenate([oracle.pq_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, inp["fine_weights"],
                                             inp["pq_codes"], inp["pq_codebook"], r, 0, int(t), 1) for t in cand])
        keep, tau = oracle.miss_filter(s, hit, w.c2f_tokens)
        assert got["tau"] == pytest.approx(tau, rel=1e-12)
        assert np.array_equal(got["kept"][: len(cand)], keep)
        assert 0 < keep.sum() < len(cand)
        sel = got["sel"][got["sel"] >= 0]
        tail = set(range((L // b) * b, L))
        allowed = set(cand[keep].tolist()) | tail
        assert set(sel.tolist()) <= allowed


def test_pq_decode_attends_its_selection():
    w, inp, ic = pq_setup()
    c = oracle.Cache(inp["k_cache"], inp["v_cache"])
    d = oracle.decode(inp["q"], c, inp["page_table"], inp["seq_lens"], num_q_heads=w.num_q_heads, k_blocks=0,
                      sink=w.sink, recent=w.recent, scale=w.softmax_scale, index_cache=ic,
                      c2f_tokens=w.c2f_tokens, fine_weights=inp["fine_weights"], pq_candidates=w.pq_candidates,
                      pq_codes=inp["pq_codes"], pq_codebook=inp["pq_codebook"], pq_hit=inp["pq_hit"])
    for r in (0, 1):
        got = oracle.pq_select(inp["q"], ic, inp["page_table"], inp["seq_lens"], **_pq_args(w, inp, ic), r=r, h=0)
        assert np.array_equal(d["sel"][r, 0], got["sel"])
        assert np.array_equal(d["cand"][r, 0], got["cand"])
    a = oracle.attend_selection(inp["q"], c, inp["page_table"], inp["seq_lens"], d["sel"],
                                num_q_heads=w.num_q_heads, sink=w.sink, recent=w.recent, scale=w.softmax_scale,
                                token_mode=True)
    assert np.array_equal(a["out"], d["out"])


def test_token_scores_wrelu_equal_the_block_fine_scores():
    w, inp, ic = pq_setup()
    blocks = np.array([2, 7])
    f, t = oracle.fine_scores(inp["q"], ic, inp["page_table"], w.num_q_heads, 1, 0, blocks,
                              fine_weights=inp["fine_weights"])
    g = oracle.token_scores_wrelu(inp["q"], ic, inp["page_table"], w.num_q_heads, inp["fine_weights"], 1, 0, t[::-1])
    assert np.array_equal(g, f[::-1])


def test_attend_selection_token_rule():
    """A token selection attends any token outside the forced ranges, the
    partial last block's included (the PQ32 selection may keep that tail),
    and skips a token inside a forced range (it is attended as forced)."""
    w, inp, ic = pq_setup(seq_lens=(64 * 5 + 20, 64 * 3), recent=8)
    c = oracle.Cache(inp["k_cache"], inp["v_cache"])
    L0 = 64 * 5 + 20
    rs = L0 - 8
    sel = np.full((2, 1, 4), -1, dtype=np.int32)
    sel[0, 0, :3] = [7, 64 * 5 + 3, rs + 1]        # a full-block token, a tail token, a forced one
    a = oracle.attend_selection(inp["q"], c, inp["page_table"], inp["seq_lens"], sel, num_q_heads=w.num_q_heads,
                                sink=0, recent=8, scale=w.softmax_scale, token_mode=True)
    toks = [7, 64 * 5 + 3] + list(range(rs, L0))
    qd = f64(bf16_bits(inp["q"][0, 5]))
    o, lse = oracle.attend_tokens(qd, c, inp["page_table"][0], toks, 0, w.softmax_scale)
    assert a["lse"][0, 5] == pytest.approx(lse, rel=1e-14)
    assert np.array_equal(a["out"][0, 5], np.array([oracle.bf16_round(x) for x in o], dtype=np.uint16))
