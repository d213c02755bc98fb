"""The benchmark's multi-GPU logic on CPU ranks (gloo, world size 2): every rank gets
its own batch (weak scaling), the job time is the slowest rank's, and the value counts
all ranks' bytes.  Decode needs no exchange between ranks, so no collective touches the
data path; only the timing is reduced."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads

        seed = bench.replica_seed(1, rank)
        case = workloads.build_case("r", S=3, Hq=4, Hkv=2, D=64, bs=16, context_lens=[5, 40, 77],
                                    seed=seed, poison=False)
        mine = [10.0 + 5 * rank, 2.0 - rank]
        got = bench.slowest_rank(mine, torch.device("cpu"))
        digest = float(case.q.float().sum())
        out.put((rank, seed, got, digest))
    finally:
        dist.destroy_process_group()


def test_two_ranks_weak_scaling():
    import sys
    from pathlib import Path

    root = str(Path(__file__).resolve().parents[1])
    if root not in sys.path:
        sys.path.insert(0, root)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, g0, d0), (r1, s1, g1, d1) = res
    assert s0 != s1 and d0 != d1  # independent batches
    assert g0 == g1 == [15.0, 2.0]  # element-wise max over ranks
    import bench

    assert bench.whole_job_gbs(1_000_000_000, 2, 1.0) == pytest.approx(2000.0)


def test_bench_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` outside torchrun starts two local ranks itself (here on the
    reference arm, which needs no GPU): one JSON line, from rank 0, reporting 2 GPUs."""
    import json
    import subprocess
    import sys
    from pathlib import Path

    root = Path(__file__).resolve().parents[1]
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    proc = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                           "--config", "tiny", "--steps", "2", "--warmup", "3"],
                          cwd=root, capture_output=True, text=True, env=env, timeout=300)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [l for l in proc.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["n_gpus"] == 2 and res["impl"] == "reference"


def test_bench_gpus_flag_must_match_world_size():
    import subprocess
    import sys
    from pathlib import Path

    root = Path(__file__).resolve().parents[1]
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    proc = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "1",
                           "--config", "tiny", "--steps", "2", "--warmup", "3"],
                          cwd=root, capture_output=True, text=True, env=env, timeout=300)
    assert proc.returncode != 0 and "WORLD_SIZE" in proc.stderr
