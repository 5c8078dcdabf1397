"""Host logic of bench.py's multi-process path on CPU: two gloo ranks (replicas of the step,
no data-path collective), the max-over-ranks timing and the sum of the units all ranks
processed, and the reference arm printing on rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_init(world)
    assert (r, w, local) == (rank, world, rank)
    elapsed = bench.max_over_ranks(1.0 + rank, w)        # slowest rank decides
    units = bench.sum_over_ranks(100.0 * (rank + 1), w)   # all ranks' units
    bench.barrier(w)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"elapsed": elapsed, "units": units}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_summed_units(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for rank in range(world):
        d = json.loads((tmp_path / f"r{rank}.json").read_text())
        assert d["elapsed"] == 2.0
        assert d["units"] == 300.0


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("world", [1, 2])
def test_bench_config_names_replicas(world):
    sys.path.insert(0, ROOT)
    import bench
    cfg = bench.config_for(world)
    assert cfg["parallelism"] == ("single" if world == 1 else f"replicas{world}")
    assert "workload" in cfg and "model" not in cfg


def test_bench_sizes_and_rotation():
    """Algorithmic bytes of the headline (configuration 3) and the copy rotation that keeps a
    re-read buffer out of L2."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.chain_bytes(256, 8, 128256, 2) == (256 * 17 * 128256 * 2 + 4 * 256 * 8
                                                    + 4 * 256 * 9 + 4 * 256 + 4 * 256 * 9)
    assert abs(bench.chain_bytes(256, 8, 128256, 2) / 1e9 - 1.116) < 0.001
    for nbytes in (4.26e6, 36e6, 45.06e6, 131e6, 1.116e9):
        n = bench.copies_for(nbytes)
        assert (n - 1) * nbytes > 3 * bench.L2_BYTES or n == 1 or n == 128
        assert n == 1 or (n - 2) * nbytes <= 3 * bench.L2_BYTES
    assert set(bench.ROW_NAMES) >= {"cfg1_chain_tiny", "cfg2_chain_32k", "cfg3_sigma0.25",
                                    "cfg3_sigma1", "cfg3_sigma4", "cfg4_tree_32k",
                                    "cfg5_B1024_g3", "cfg5_B1024_g7"}
    a = bench.parse([])
    assert a.steps >= 1 and a.warmup >= 3 and a.rows == "all"
