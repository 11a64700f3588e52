"""The C-ABI library loads, exports every function include/lsa.h declares,
and validates arguments on the host (no GPU needed: these calls return
before any CUDA work)."""
import ctypes as C
import os
import re

import pytest

import __graft_entry__
from sparse_attention_decode_block_gb300 import lsa as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lsa.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return L.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_calls_of_the_path():
    names = declared_functions()
    for n in ("lsa_build_summaries", "lsa_append_block", "lsa_score", "lsa_topk", "lsa_sparse_decode",
              "lsa_decode_step"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in lsa.h but not exported"
    assert sorted(L.EXPORTED) == names


def test_struct_layouts_match_header():
    # lsa_cache: 2 pointers, 6 int64 strides, 6 int32, 1 pointer, 2 int64
    assert C.sizeof(L.lsa_cache) == 8 * 2 + 8 * 6 + 4 * 6 + 8 + 8 * 2
    # 11 int32 / float fields, padding, a pointer, an int32, padding, 3 pointers
    assert C.sizeof(L.lsa_params) == 4 * 12 + 8 + 8 + 8 * 3


def test_status_strings(lib):
    assert L.lsa_status_string(0) == "ok"
    assert "workspace" in L.lsa_status_string(3)
    assert L.lsa_status_string(99) == "unknown status"


def _cache(**kw):
    c = L.lsa_cache()
    c.k = 4096
    c.v = 8192
    c.k_page_stride = c.v_page_stride = 8 * 16 * 128
    c.k_head_stride = c.v_head_stride = 16 * 128
    c.k_token_stride = c.v_token_stride = 128
    c.num_pages, c.block_size, c.num_kv_heads, c.dk, c.dv = 64, 16, 8, 128, 128
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_host_validation_rejects_bad_arguments(lib):
    prm = L.make_params(2, 32, 4, 2, 16, 16)
    fake = C.c_void_p(1 << 20)
    s = C.c_void_p(0)
    cases = [
        _cache(k=None),
        _cache(k=4100),              # misaligned pointer
        _cache(dk=100),              # dk*2 not a multiple of 16
        _cache(num_pages=0),
        _cache(k_token_stride=64),   # token stride shorter than a row
        _cache(k_head_stride=1000 + 3),
    ]
    for c in cases:
        rc = lib.lsa_score(fake, C.byref(c), fake, fake, fake, C.byref(prm), fake, s)
        assert rc == L.LSA_ERR_INVALID_ARG
    bad = L.make_params(2, 30, 4, 2, 16, 16)   # 30 query heads over 8 KV heads
    assert lib.lsa_score(fake, C.byref(_cache()), fake, fake, fake, C.byref(bad), fake, s) == L.LSA_ERR_INVALID_ARG
    neg = L.make_params(2, 32, 4, -1, 16, 16)
    assert lib.lsa_sparse_decode(fake, C.byref(_cache()), fake, fake, fake, C.byref(neg), fake, None, None, 0,
                                 s) == L.LSA_ERR_INVALID_ARG
    assert lib.lsa_topk(fake, None, -1, 4, 2, fake, s) == L.LSA_ERR_INVALID_ARG
    assert lib.lsa_topk(fake, None, 3, 4, 2, None, s) == L.LSA_ERR_INVALID_ARG
    assert lib.lsa_topk_approx(fake, None, 3, 4, -2, 1, fake, s) == L.LSA_ERR_INVALID_ARG
    assert lib.lsa_topk_approx(fake, None, 3, 4, 2, 1, None, s) == L.LSA_ERR_INVALID_ARG


def test_empty_work_is_ok_without_launching(lib):
    s = C.c_void_p(0)
    c = _cache()
    prm = L.make_params(0, 32, 4, 2, 16, 16)
    assert lib.lsa_score(None, C.byref(c), None, None, None, C.byref(prm), None, s) == L.LSA_OK
    assert lib.lsa_topk(None, None, 0, 10, 3, None, s) == L.LSA_OK
    assert lib.lsa_topk(None, None, 5, 10, 0, None, s) == L.LSA_OK
    assert lib.lsa_topk_approx(None, None, 0, 10, 3, 7, None, s) == L.LSA_OK
    assert lib.lsa_build_summaries(C.byref(c), None, None, 0, 4, None, s) == L.LSA_OK


def test_unsupported_shapes_are_reported(lib):
    c = _cache(dk=96, dv=96)
    prm = L.make_params(2, 32, 4, 2, 16, 16)
    assert lib.lsa_sparse_decode_workspace_size(C.byref(c), C.byref(prm)) == 0
    fake = C.c_void_p(1 << 20)
    rc = lib.lsa_sparse_decode(fake, C.byref(c), fake, fake, fake, C.byref(prm), fake, None, None, 0, C.c_void_p(0))
    assert rc == L.LSA_ERR_UNSUPPORTED


def test_workspace_too_small_is_reported(lib):
    c = _cache()
    prm = L.make_params(4, 32, 4, 2, 16, 16, num_splits=3)
    need = lib.lsa_sparse_decode_workspace_size(C.byref(c), C.byref(prm))
    assert need > 0
    fake = C.c_void_p(1 << 20)
    rc = lib.lsa_sparse_decode(fake, C.byref(c), fake, fake, fake, C.byref(prm), fake, None, fake, need - 1,
                               C.c_void_p(0))
    assert rc == L.LSA_ERR_WORKSPACE
    assert lib.lsa_decode_step_workspace_size(C.byref(c), C.byref(prm)) >= need


def test_binding_fails_loudly_without_library(tmp_path):
    import subprocess
    import sys
    env = dict(os.environ, LSA_LIBRARY=str(tmp_path / "missing.so"))
    code = ("import sparse_attention_decode_block_gb300 as L\n"
            "try:\n    L.lsa_status_string(0)\nexcept RuntimeError as e:\n"
            "    print('LOUD', e)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert "LOUD" in r.stdout and "missing" in r.stdout
