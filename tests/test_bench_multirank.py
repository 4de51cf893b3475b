"""The bench's N > 1 host logic on CPU: two gloo ranks (no GPU).

Each rank reports its own step times; the job time is the maximum over ranks, the job rate
counts every rank's units (weak scaling), and only rank 0 prints.  The reference arm's other
ranks exit without work.
"""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured total 10 + r ms over 4 steps and an e2e step of 3 - r ms
        total, e2e = bench.max_over_ranks([10.0 + rank, 3.0 - rank], world, "cpu")
        value, mean_ms = bench.job_rate(world, 1000.0, total, 4)
        args = type("A", (), dict(workload="softmax_1d", warmup=0, steps=1, gpus=world, ref_budget=0.05))()
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.reference_arm(args, world, rank) if rank == 1 else 0
        results[rank] = dict(total=total, e2e=e2e, value=value, mean_ms=mean_ms, rc=rc, out=buf.getvalue())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reduce_to_the_slowest():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    for r in range(world):
        assert res[r]["total"] == 11.0          # max over ranks of 10 + r
        assert res[r]["e2e"] == 3.0             # max over ranks of 3 - r
        assert res[r]["mean_ms"] == pytest.approx(11.0 / 4)
        # two ranks x 1000 units per 2.75 ms step
        assert res[r]["value"] == pytest.approx(2 * 1000.0 / (11.0 / 4 / 1e3))
    assert res[1]["rc"] == 0 and res[1]["out"] == ""   # non-zero ranks of the reference arm print nothing


def test_reference_arm_rank0_prints_one_line(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), dict(workload="softmax_1d", warmup=0, steps=1, gpus=1, ref_budget=0.05))()
    assert bench.reference_arm(args, 1, 0) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_compact_suite_entry_and_baseline_configs():
    """The bench line's suite entries are short objects carrying the roofline; every problem
    statement configuration is a workload of the bench, and one core of the oracle is a process
    pinned to one CPU."""
    sys.path.insert(0, ROOT)
    import bench
    e = {"value": 1.5, "unit": "GB/s", "ms_per_step": 0.2,
         "roofline": {"bound": "hbm", "peak": 6769.4, "frac": 0.5, "traffic": 1e6}}
    c = bench.compact(e, [0.1, 0.05])
    assert c == {"v": 1.5, "u": "GB/s", "ms": 0.2, "bound": "hbm", "peak": 6769.4, "frac": 0.5, "dram_mb": 1.0,
                 "oracle": [0.1, 0.05]}
    assert "oracle" not in bench.compact(e)
    assert bench.compact({**e, "value": 1234.5678, "roofline": {**e["roofline"], "traffic": None}})["v"] == 1235.0
    # the problem statement's configurations and the backward come last in the line
    names = ["softmax_rows", "gqa_causal_prefill_bshd", "gqa_causal_backward", "single_head_m64_n100", "x"]
    order = bench.suite_order(names)
    assert order[:2] == ["gqa_causal_prefill_bshd", "x"] and order[2] == "gqa_causal_backward"
    assert set(order[3:]) == {"softmax_rows", "single_head_m64_n100"}
    assert set(bench.BASELINE_CONFIGS) <= set(bench.WORKLOADS)
    one = bench.oracle_one_core("single_head_m64_n100", 0.2)
    assert one is not None and one["cores"] == 1 and one["value"] > 0 and one["unit"] == "TFLOP/s"
