"""Host-side checks of the seeded generators and the byte account."""
import torch

from workloads import WORKLOADS, algorithmic_bytes, make_inputs, small_workloads


def test_byte_account_b16_32k():
    w = WORKLOADS["b16_32k"]
    acc = algorithmic_bytes(w, [32768] * 16)
    # KV bytes read for n tokens = 2 (K and V) * h_kv * d_h * n * 2 bytes
    # (ByteCross, Section 3.1, Eq. 4), with n = 1024 attended tokens per request
    assert acc["kv"] == 16 * (2 * 8 * 128 * 1024 * 2)
    # 2046 candidate blocks (block 0 = sink, block 2047 = recent window)
    assert acc["summaries"] == 16 * 8 * 2046 * 128 * 2
    assert acc["total"] == 134_545_408


def test_byte_account_latent_counts_k_once():
    w = WORKLOADS["mla"]
    acc = algorithmic_bytes(w, [1 << 20] * 4)
    assert acc["kv"] == 4 * 1988 * 576 * 2
    assert acc["summaries"] == 4 * 16381 * 576 * 2


def test_generator_is_seeded_and_structured():
    w = small_workloads()["b16_small"]
    a = make_inputs(w, "cpu")
    b = make_inputs(w, "cpu")
    for k in ("q", "k_cache", "v_cache", "page_table", "seq_lens"):
        assert torch.equal(a[k], b[k])
    pt = a["page_table"]
    used = pt[pt >= 0]
    assert used.unique().numel() == used.numel() == a["num_pages"]   # a permutation
    assert a["lens"] == [4096, 3001, 777]


def test_c2f_index_keys_quantised_per_token():
    w = small_workloads()["c2f_small"]
    a = make_inputs(w, "cpu")
    k8 = a["idx_keys"].view(torch.float8_e4m3fn).float()
    # per-token scale maps the largest magnitude to the e4m3 maximum 448
    assert torch.all(k8.abs().amax(dim=-1) == 448.0)
    assert a["idx_scale"].dtype == torch.float32
