"""Host logic of bench.py on the CPU: the multi-rank replicas path (barrier, max over ranks,
whole-job rate) on a world_size-2 gloo process group, and the code hash that keeps a
recorded DRAM-traffic capture attached to its kernel."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(('127.0.0.1', 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR='127.0.0.1', MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group('gloo', rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_setup()
        barrier, max_over_ranks = bench.make_ranks(dist, torch.device('cpu'))
        barrier()
        ms = max_over_ranks(1.0 + rank * 0.5)          # rank 1 is the slow one: 1.5 ms
        out.put((r, ws, local, ms, bench.whole_job_rate(4096, ws, ms)))
        barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    ctx = mp.get_context('spawn')
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    for r, (rank, ws, local, ms, rate) in enumerate(got):
        assert (rank, ws, local) == (r, 2, r)
        assert ms == 1.5                                  # every rank sees the slowest time
        assert rate == pytest.approx(2 * 4096 / 1.5e-3)   # tokens of both ranks over it


def test_one_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    barrier, max_over_ranks = bench.make_ranks(None, torch.device('cpu'))
    barrier()
    assert max_over_ranks(2.5) == 2.5
    assert bench.whole_job_rate(4096, 1, 2.0) == pytest.approx(4096 / 2e-3)


def test_code_hash_ignores_comments_only():
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) {\n  return x + 1;  // one\n}\n"
    b = "/* a note */\nint f(int x)   {\n  return x + 1;\n}  // trailing\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(c)


def test_clock_summary_takes_the_busy_samples():
    sys.path.insert(0, ROOT)
    import bench
    lines = [
        '0, 1200, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active, 0\n',     # idle
        '0, 2070, 2070, 240.0, 0x0, Not Active, Not Active, Not Active, Not Active, 97\n',
        '0, 2055, 2070, 260.0, 0x4, Not Active, Not Active, Not Active, Active, 100\n',
        '0, 2070, 2070, 230.0, 0x0, Not Active, Not Active, Not Active, Not Active, 64\n',
        'garbage line\n',
    ]
    r = bench.summarize_clocks(lines)
    assert r['samples'] == 4 and r['samples_under_load'] == 3
    assert r['sm_mhz'] == 2070.0 and r['sm_max_mhz'] == 2070.0
    assert r['reasons'] == ['sw_power_cap'] and r['power_w_max'] == 260.0
    # no utilization counter (or none busy): every sample counts
    r = bench.summarize_clocks([ln.rsplit(',', 1)[0] + ', [N/A]\n' for ln in lines[:2]])
    assert r['samples'] == 2 and r['samples_under_load'] == 2 and r['sm_mhz'] == (1200 + 2070) / 2
