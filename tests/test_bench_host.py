"""bench.py's host logic on CPU: two gloo ranks, each timing its own
replica (the reported time is the max over ranks and the throughput counts
every rank's work: weak scaling); the traffic record's source key; the
reference arm's JSON line; no output line without a GPU."""
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


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores and
    prints one JSON line with the main arm's metric and unit, the `impl`
    key, its own cpu_baseline and an e2e entry with no device copies."""
    import json
    import subprocess
    sys.path.insert(0, ROOT)
    import bench
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_gpu_arm_fails_loudly_without_a_gpu():
    """With no GPU the bench exits non-zero instead of falling back."""
    import subprocess
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode != 0
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
