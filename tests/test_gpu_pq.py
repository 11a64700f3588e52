"""PQ32 coarse-to-fine selection on the GPU against the oracle, stage by stage.

The coarse scores come from tensor-core products in fp32, the oracle's in
fp64, so the three decisions the method makes (the top-C coarse candidates,
the miss filter's threshold, the top-k fine tokens) are checked in the order
the method takes them, each against the oracle applied to the GPU's own
inputs of that stage:
  - the PQ32 codes: bit-exact (the encoder's distance order is fixed);
  - the coarse scores: within the fp32 rounding bound of the products;
  - the candidates: the exact top-C of the GPU's coarse scores, bit for bit;
  - the miss filter and the fine top-k: the oracle's filter and exact fine
    scores on those candidates, the final tokens equal up to fine-score
    ties within the fp32 rounding of the fine scores;
  - attention: the oracle's attention over the GPU's tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_decode_block_gb300 as L
from helpers import (GpuStep, assert_attention_close, assert_lse_close, check_status_clean, oracle_cache,
                     oracle_index, to_dev)
from workloads import WORKLOADS, make_inputs, small_workloads

pytestmark = pytest.mark.gpu


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


def gpu_coarse(st, w, g):
    """The coarse scores of every token position ([B, max_blocks * b]),
    from lsa_pq_scores (the same kernel as the step's)."""
    T = g["max_blocks"] * w.block_size
    out = torch.empty((w.batch, T), dtype=torch.float32, device="cuda")
    L.lsa_pq_scores(g["q"], st.icache, g["page_table"], g["seq_lens"], st.params, out)
    check_status_clean()
    return out.cpu().numpy()


def step_candidates(st, w, g):
    """The coarse candidates the step wrote to its workspace."""
    T = g["max_blocks"] * w.block_size
    ru = lambda x: (x + 255) // 256 * 256
    off = ru(w.batch * T * 4) + ru(w.batch * w.c2f_tokens * 4)
    raw = st.ws[off: off + w.batch * w.pq_candidates * 4].view(torch.int32)
    return raw.view(w.batch, w.pq_candidates).cpu().numpy()


def coarse_bound(w, cpu, r, toks):
    """|fp32 - exact| bound of the coarse scores of tokens `toks`: each head's
    dot sums 128 products (each exact), rounded 128 times at most, then the
    weighted ReLUs are summed in fp32: 4 * 192 * 2^-24 * sum_g w_g sum_i
    |q_gi c_i|, with margin."""
    b = w.block_size
    q = np.abs(cpu["q"][r].float().numpy().astype(np.float64))              # [64, 128]
    cb = cpu["pq_codebook"].float().numpy().astype(np.float64)              # [32, 256, 4]
    pt = cpu["page_table"][r].numpy()
    codes = cpu["pq_codes"].numpy()[pt[toks // b], 0, toks % b].astype(np.int64)   # [n, 32]
    cent = np.abs(cb[np.arange(32)[None, :], codes]).reshape(len(toks), 128)       # [n, 128]
    wt = cpu["fine_weights"][r].numpy().astype(np.float64)
    return 4 * 192 * 2.0 ** -24 * (cent @ q.T @ wt) + 1e-30


def check_coarse(w, cpu, coarse, r, toks):
    ic = oracle_index(cpu)
    ref = np.concatenate([oracle.pq_scores(cpu["q"], ic, cpu["page_table"], w.num_q_heads, cpu["fine_weights"],
                                           cpu["pq_codes"], cpu["pq_codebook"], r, 0, int(t), 1) for t in toks])
    got = coarse[r, toks].astype(np.float64)
    err = np.abs(got - ref)
    bound = coarse_bound(w, cpu, r, toks)
    assert np.all(err <= bound), f"coarse: worst {np.max(err / bound):.3g} of the bound"


def reference_selection(w, cpu, coarse, r, hit_none=False):
    """Steps 2-4 on the GPU's coarse scores: the exact top-C of them, the
    oracle's miss filter, the oracle's exact fine scores of the kept
    candidates and of the tail, and their top-k."""
    b = w.block_size
    Lr = int(cpu["seq_lens"][r])
    s = coarse[r].astype(np.float64)
    cand = oracle.topk(s[None], w.pq_candidates)[0]
    cv = cand[cand >= 0]
    pt = cpu["page_table"][r].numpy()
    hit = (np.ones(len(cv), np.uint8) if hit_none
           else cpu["pq_hit"].numpy()[pt[cv // b], 0, cv % b].astype(np.uint8))
    keep, tau = oracle.miss_filter(s[cv], hit, w.c2f_tokens)
    se = min(w.sink, Lr)
    rs = max(Lr - w.recent, se)
    tail = np.array([t for t in range((Lr // b) * b, Lr) if se <= t < rs], dtype=np.int64)
    pool = np.concatenate([cv[keep], tail]).astype(np.int64)
    ic = oracle_index(cpu)
    fpool = oracle.token_scores_wrelu(cpu["q"], ic, cpu["page_table"], w.num_q_heads, cpu["fine_weights"], r, 0,
                                      pool)
    order = sorted(range(len(pool)), key=lambda i: (-fpool[i], pool[i]))[: w.c2f_tokens]
    sel = np.sort(pool[order])
    return dict(cand=cand, cv=cv, s_cand=s[cv], keep=keep, tau=tau, pool=pool, fpool=fpool, sel=sel)


def check_selection(w, ref, sel_gpu):
    """The GPU's final tokens equal the reference's up to ties of the fine
    scores at the k-th (within their fp32 rounding) and candidates whose
    coarse score sits on the threshold."""
    got = sel_gpu[sel_gpu >= 0]
    want = ref["sel"]
    if np.array_equal(got, want):
        return 0
    assert len(got) == len(want), "selection sizes differ"
    diff = np.setxor1d(got, want)
    fk = ref["fpool"][np.isin(ref["pool"], want)].min()
    eps = 5e-5 * (1.0 + abs(fk))
    near_tau = set(ref["cv"][np.abs(ref["s_cand"] - ref["tau"]) <= 1e-9 * (1.0 + abs(ref["tau"]))].tolist())
    fmap = dict(zip(ref["pool"].tolist(), ref["fpool"].tolist()))
    for t in diff.tolist():
        ok = t in near_tau or (t in fmap and abs(fmap[t] - fk) <= eps)
        assert ok, f"token {t} differs and is no tie (f={fmap.get(t)}, k-th {fk})"
    return len(diff)


def check_step(w, cpu, g, st, reqs, coarse, hit_none=False):
    cand_gpu = step_candidates(st, w, g)
    sel_gpu = st.idx.cpu().numpy()[:, 0]
    for r in reqs:
        ref = reference_selection(w, cpu, coarse, r, hit_none)
        assert np.array_equal(cand_gpu[r], ref["cand"]), f"request {r}: coarse candidates differ"
        check_selection(w, ref, sel_gpu[r])
    a = oracle.attend_selection(cpu["q"], oracle_cache(cpu), cpu["page_table"], cpu["seq_lens"],
                                st.idx.cpu().numpy(), num_q_heads=w.num_q_heads, sink=w.sink, recent=w.recent,
                                scale=w.softmax_scale, token_mode=True)
    idx = list(reqs)
    assert_attention_close(st.out[idx], a["out"][idx], w.name)
    assert_lse_close(st.lse[idx], a["lse"][idx], w.name)


def test_pq_encode_bit_exact():
    w = small("c2f_pq_small")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    icache = L.make_cache(g["idx_keys"], None, k_scale=g["idx_scale"])
    codes = torch.full_like(g["pq_codes"], 0xAB)
    L.lsa_pq_encode(icache, g["pq_codebook"], g["page_table"], g["seq_lens"], codes)
    check_status_clean()
    b = w.block_size
    ic = oracle_index(cpu)
    got = codes.cpu().numpy()
    for r in range(w.batch):
        nfull = int(cpu["seq_lens"][r]) // b
        pages = cpu["page_table"][r, :nfull].numpy().astype(np.int64)
        slots = (pages[:, None] * b + np.arange(b)[None, :]).reshape(-1)
        want = oracle.pq_encode(ic, cpu["pq_codebook"], slots)
        assert np.array_equal(got.reshape(-1, 32)[slots], want)
        # the partial last block is not encoded
        if int(cpu["seq_lens"][r]) % b:
            last = int(cpu["page_table"][r, nfull])
            assert np.all(got[last] == 0xAB)


def test_pq_scores_within_rounding():
    w = small("c2f_pq_small")
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    coarse = gpu_coarse(st, w, g)
    b = w.block_size
    T = g["max_blocks"] * b
    for r in range(w.batch):
        Lr = int(cpu["seq_lens"][r])
        nfull = Lr // b
        se = min(w.sink, Lr)
        rs = max(Lr - w.recent, se)
        cand_tok = np.array([t for t in range(nfull * b) if (t // b) * b >= se and (t // b + 1) * b <= rs])
        check_coarse(w, cpu, coarse, r, cand_tok)
        rest = np.setdiff1d(np.arange(T), cand_tok)
        assert np.all(np.isneginf(coarse[r, rest]))


def test_pq_scores_request_changes_every_tile():
    """Requests of about 150 tiles of 128 tokens each, ragged, so that the
    scorer's persistent CTAs (tiles strided by the grid) change request at
    nearly every tile: each change flips the query slot and reloads the head
    weights, while the prefetch rings run ahead across requests."""
    w = small("c2f_pq_small", batch=6, seq_lens=(19203, 4100, 17000, 64 * 100 + 3, 12345, 960))
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    coarse = gpu_coarse(st, w, g)
    b = w.block_size
    rng = np.random.default_rng(3)
    for r in range(w.batch):
        Lr = int(cpu["seq_lens"][r])
        nfull = Lr // b
        se = min(w.sink, Lr)
        rs = max(Lr - w.recent, se)
        cand_tok = np.array([t for t in range(nfull * b) if (t // b) * b >= se and (t // b + 1) * b <= rs])
        if len(cand_tok):
            check_coarse(w, cpu, coarse, r, np.sort(rng.choice(cand_tok, size=min(400, len(cand_tok)), replace=False)))
        rest = np.setdiff1d(np.arange(coarse.shape[1]), cand_tok)
        assert np.all(np.isneginf(coarse[r, rest]))
    st.run()
    check_status_clean()
    check_step(w, cpu, g, st, range(w.batch), coarse)


@pytest.mark.parametrize("variant", ["base", "short", "all_hits", "no_hits", "few_candidates"])
def test_pq_step_stagewise(variant):
    kw = {}
    if variant == "short":
        kw = dict(seq_lens=(64 * 30 + 5, 64 * 3, 40), batch=3, pq_candidates=1024, c2f_tokens=256)
    elif variant == "few_candidates":
        kw = dict(pq_candidates=300, c2f_tokens=200)
    w = small("c2f_pq_small", **kw)
    cpu = make_inputs(w, "cpu")
    if variant == "no_hits":
        cpu["pq_hit"] = torch.zeros_like(cpu["pq_hit"])
    g = to_dev(cpu)
    if variant == "all_hits":
        g["pq_hit"] = None
    st = GpuStep(w, g)
    st.run()
    check_status_clean()
    coarse = gpu_coarse(st, w, g)
    check_step(w, cpu, g, st, range(w.batch), coarse, hit_none=variant == "all_hits")


def test_pq_step_repeats_bit_identical():
    """The step resets the rows' counts and extremes it accumulates, so a
    second call on the same workspace gives the same bits."""
    w = small("c2f_pq_small")
    g = to_dev(make_inputs(w, "cpu"))
    st = GpuStep(w, g)
    st.run()
    a = (st.idx.clone(), st.out.clone())
    st.run()
    check_status_clean()
    assert torch.equal(st.idx, a[0])
    assert torch.equal(st.out.view(torch.int16), a[1].view(torch.int16))


def test_pq_full_size_every_request():
    """The full-size workload (B=4, 512K tokens each, C=8192, k=2048): coarse
    scores on a sample of tokens, then every request's candidates, filter,
    tokens and attention."""
    w = WORKLOADS["c2f_pq"]
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    st.run()
    check_status_clean()
    coarse = gpu_coarse(st, w, g)
    rng = np.random.default_rng(0)
    for r in range(w.batch):
        nfull = int(cpu["seq_lens"][r]) // w.block_size
        toks = rng.choice(nfull * w.block_size, size=2000, replace=False)
        check_coarse(w, cpu, coarse, r, np.sort(toks))
    check_step(w, cpu, g, st, range(w.batch), coarse)
