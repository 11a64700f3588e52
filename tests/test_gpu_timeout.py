"""Bounded device waits run out instead of hanging.

The tensor-core attention's tiles (the 64-head groups of the coarse-to-fine
and latent-cache steps) wait for the rest of their row before merging it.
The wait gives up after a budget of SM clock cycles, records LSA_ERR_TIMEOUT
in the device status word and lets the kernel finish.  Here every counter
the wait reads starts at a value it never reaches (the workspace is filled
with 0xff bytes instead of zeros) and the budget is cut to a few
microseconds: the call must return promptly with LSA_ERR_TIMEOUT, and the
same call on a zeroed workspace must then match the oracle.
"""
import time

import pytest
import torch

import sparse_attention_decode_block_gb300 as L
from helpers import GpuStep, check_status_clean, to_dev
from test_gpu_parity import compare_step_rows, small
from workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    L.lsa_get_device_status(clear=True)
    yield


@pytest.mark.parametrize("name", ["c2f_small", "mla_small"])
def test_wait_that_cannot_end_times_out_then_zeroed_workspace_recovers(name, monkeypatch):
    w = small(name)
    cpu = make_inputs(w, "cpu")
    g = to_dev(cpu)
    st = GpuStep(w, g)
    st.run()
    check_status_clean()
    # counters that never reach what their waits expect
    st.ws.fill_(0xFF)
    monkeypatch.setenv("LSA_SPIN_BUDGET", "20000")   # SM clock cycles: about 10 us
    t0 = time.time()
    st.run()
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    code, flags = L.lsa_get_device_status(clear=True)
    assert code == L.LSA_ERR_TIMEOUT, f"status {L.lsa_status_string(code)} flags {flags:#x}"
    assert elapsed < 10.0
    # the context is usable: a zeroed workspace gives the oracle's answer
    monkeypatch.delenv("LSA_SPIN_BUDGET")
    st.ws.zero_()
    st.run()
    check_status_clean()
    compare_step_rows(st, w, cpu, range(w.batch))
    # and the call leaves the workspace ready for the next one
    st.run()
    check_status_clean()
    compare_step_rows(st, w, cpu, range(w.batch))
