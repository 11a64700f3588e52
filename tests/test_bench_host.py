"""Host logic of bench.py's multi-rank (replica) mode, on CPU with gloo.

Each rank runs an independent replica; the only cross-rank steps are the
barrier around the timed region and the max over ranks of its length, and
the job's value counts every rank's calls.  Tested here with two gloo ranks.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], torch.device("cpu"), world)
        out[rank] = (ms, bench.job_calls_per_s(100, world, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    times = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        ms, calls = out[r]
        assert ms == 20.0                       # every rank sees the slowest rank's time
        assert calls == pytest.approx(2 * 100 / 0.020)   # both replicas' calls in that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, torch.device("cpu"), 1) == 3.0
    assert bench.job_calls_per_s(10, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_e2e_staging_buffer_layout():
    """The e2e leg's staging buffers: every tensor at a 16-byte aligned offset
    of one buffer, views that alias it, and the buffer's size the bytes a step
    copies (checked on CPU memory; the bench pins the host side)."""
    sys.path.insert(0, ROOT)
    import bench
    q = torch.randn(3, 5, 128).to(torch.bfloat16)
    pt = torch.randint(0, 1000, (3, 7), dtype=torch.int32)
    lens = torch.arange(3, dtype=torch.int32)
    buf, (vq, vpt, vl) = bench._packed([q, pt, lens], pinned=False, dev="cpu")
    offs = [v.data_ptr() - buf.data_ptr() for v in (vq, vpt, vl)]
    assert offs[0] == 0 and all(o % 16 == 0 for o in offs)
    assert offs[1] >= q.numel() * 2 and offs[2] >= offs[1] + pt.numel() * 4
    assert buf.numel() == offs[2] + 16   # 12 bytes of lengths, rounded up to 16
    vq.copy_(q)
    vpt.copy_(pt)
    vl.copy_(lens)
    assert torch.equal(vq, q) and torch.equal(vpt, pt) and torch.equal(vl, lens)
    assert vq.shape == q.shape and vpt.dtype == torch.int32
    # the views write through to the one buffer that a step copies
    raw = buf[offs[1]:offs[1] + 4].view(torch.int32)
    assert int(raw[0]) == int(pt[0, 0])
