"""The N > 1 launch of bench.py on CPU: ranks as gloo processes (world size 2).

Heads are independent, so the ranks share nothing on the data path; what the
multi-GPU run adds is host logic: the barrier around the timed region, the
maximum of the per-rank times, the whole-job rate, and the reference arm that
only rank 0 runs.  These run here without a GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        elapsed = 0.25 * (rank + 1)          # rank 1 is the slow one
        bench.barrier(world)
        slowest = bench.max_over_ranks(elapsed, world)
        tokens = 1000 * (rank + 1)           # per-rank work is fixed (weak scaling) ...
        rate = bench.aggregate(1000, world, slowest, steps=4)  # ... and equal on every rank
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"dist_env": [r, w, local], "slowest": slowest, "rate": rate,
                       "tokens": tokens}, f)
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_ranks_with_gloo(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert x["dist_env"] == [r, world, r]
        assert x["slowest"] == 0.5                     # the maximum over both ranks
        assert x["rate"] == pytest.approx(1000 * 2 * 4 / 0.5)  # all ranks' tokens / max time


def test_reference_arm_prints_once_under_two_ranks():
    """Under torchrun every rank starts bench.py; only rank 0 times the oracle and
    prints the JSON line, the others exit 0 without output."""
    outs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
        p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1",
                            "--steps", "1", "--warmup", "1"], cwd=ROOT, env=env,
                           capture_output=True, text=True, timeout=300)
        assert p.returncode == 0, p.stderr[-2000:]
        outs.append([ln for ln in p.stdout.splitlines() if ln.strip()])
    assert outs[1] == []
    assert len(outs[0]) == 1
    line = json.loads(outs[0][0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
