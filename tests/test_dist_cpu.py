"""The multi-rank host logic of bench.py on CPU with the gloo backend, world size 2: rank setup
from the launcher's environment, the max-over-ranks timing, the barrier, and the reference arm
under torch.distributed.run (rank 0 alone runs and prints; the other rank exits 0 without work).
The path itself has no data-path collective: N GPUs run N independent replicas."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    r, world, local = bench.dist_setup(2)
    got = bench.max_over_ranks(10.0 * (rank + 1), world)  # each rank's own time: 10, 20
    bench.barrier(world)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": world, "local": local, "max": got,
                   "backend": dist.get_backend()}, f)
    dist.destroy_process_group()


def test_two_ranks_setup_max_and_barrier(tmp_path):
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in (0, 1):
        res = json.load(open(tmp_path / f"rank{rank}.json"))
        assert res == {"rank": rank, "world": 2, "local": rank, "max": 20.0, "backend": "gloo"}


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--S", "64",
           "--Smax", "256"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1
    assert line["warmup"] == 3 and line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "us/layer", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
