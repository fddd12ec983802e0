"""The N > 1 host path of bench.py on CPU: two gloo ranks launched by
torch.distributed.run report the slowest rank's time and every rank's work,
and the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time_and_all_the_work(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import json, os, sys
        sys.path.insert(0, {ROOT!r})
        import torch.distributed as dist
        import bench
        rank, _, world = bench.dist_env()
        dist.init_process_group("gloo")
        ms = bench.slowest_rank_ms(10.0 + 5.0 * rank, world, "cpu")
        rate = bench.job_rate(2.0e9, world, 10, ms, False)
        dist.barrier()
        with open(os.path.join({str(tmp_path)!r}, f"rank{{rank}}.json"), "w") as f:
            json.dump({{"rank": rank, "world": world, "ms": ms, "rate": rate}}, f)
        dist.destroy_process_group()
    """))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", str(script)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=180, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / f"rank{k}.json").read_text()) for k in range(2)]
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["world"] == 2
        assert l["ms"] == 15.0  # rank 1 was slower
        # 2 ranks x 2 GB x 10 steps in 15 ms
        assert l["rate"] == pytest.approx(2 * 2.0e9 * 10 / 15e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        config, steps, warmup, gpus = "tiny_prefill_hd256", 1, 3, 2

    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
