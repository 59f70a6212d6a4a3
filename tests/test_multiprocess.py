"""The multi-process side of bench.py on CPU (gloo, world size 2): the
slowest rank defines the job's time, the reported value aggregates all ranks,
ranks run independent token streams, and the reference arm runs on rank 0
only. (The path itself has no exchange step: replicas only.)"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import json
    import sys

    import torch.distributed as dist

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    mine = [10.0 + rank, 20.0 - 5.0 * rank]  # rank 1 slower in the first, faster in the second
    got = bench.max_over_ranks(mine, dist)

    class Args:
        warmup, steps = 1, 1

    ref_out = bench.run_reference(Args, rank) if rank != 0 else "skipped on rank 0 (runs the oracle)"
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got, "seeds": bench.replica_seeds(rank), "ref": ref_out}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo(tmp_path):
    import json

    import torch.multiprocessing as mp

    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["max"] == r1["max"] == [11.0, 20.0]
    assert r0["seeds"] != r1["seeds"]  # independent replicas
    assert r1["ref"] is None  # the reference arm does no work off rank 0


def test_aggregate_counts_every_rank():
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    assert bench.aggregate_tokens_per_s(1, 0.025) == pytest.approx(40000.0)
    assert bench.aggregate_tokens_per_s(4, 0.025) == pytest.approx(160000.0)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_reference_arm_json_line():
    """`bench.py --impl reference` prints one JSON line with the contract's
    keys, its own metric, the oracle as cpu_baseline and an e2e object."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert "workload" in d["config"]
