"""bench.py's multi-rank host logic on CPU: two gloo ranks, each timing its
own replica; the reported time is the max over ranks and the throughput
counts every rank's work (weak scaling)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    local = 1.0 + rank                    # rank 1 is the slow one
    bench.barrier()
    m = bench.max_over_ranks(local)
    agg = bench.aggregate_throughput(bytes_per_step=1000, rows_per_step=10, steps=5,
                                     max_seconds=m, world=world)
    out[rank] = (m, agg["gbs"], agg["rows_per_s"], agg["ms_per_step"])
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        m, gbs, rows, ms = out[r]
        assert m == 2.0
        assert gbs == pytest.approx(2 * 1000 * 5 / 2.0 / 1e9)
        assert rows == pytest.approx(2 * 10 * 5 / 2.0)
        assert ms == pytest.approx(400.0)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    a = bench.aggregate_throughput(9344, 1, 100, 0.5, 1)
    assert a["gbs"] == pytest.approx(9344 * 100 / 0.5 / 1e9)


def test_traffic_record_key_ignores_comments_and_layout():
    """The ncu traffic record stays valid across comment and whitespace
    edits of the kernel sources, and not across code edits."""
    sys.path.insert(0, ROOT)
    import bench
    code = 'int f(int a) {  // first\n  /* two\n lines */ return a + 1; }\nconst char* s = "x // y";\n'
    same = 'int f(int a) { return a + 1; }   /* moved */\nconst char* s = "x // y";'
    assert bench.code_without_comments(code) == bench.code_without_comments(same)
    assert bench.code_without_comments(code) != bench.code_without_comments(code.replace("+ 1", "+ 2"))
    assert bench.code_without_comments(code) != bench.code_without_comments(code.replace("x // y", "x y"))
    assert "'/'" in bench.code_without_comments("char c = '/'; // slash")
    assert len(bench.kernel_source_hash()) == 16
