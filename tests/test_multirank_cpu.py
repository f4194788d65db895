"""The N>1 host path of bench.py on CPU: two gloo ranks agree on the
max-over-ranks step time, the whole-job value counts every rank's bytes,
and the reference arm under torchrun prints one line from rank 0 only.

The path has no exchange step (sequences and kv heads are independent), so
N GPUs run N independent replicas; the only collectives are the barrier and
this max."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # rank r measured step 1+r ms and decode 5-r ms
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank], "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(got, f)


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    ws = 2
    mp.spawn(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, join=True)
    for r in range(ws):
        assert json.load(open(tmp_path / f"rank{r}.json")) == [2.0, 5.0]


def test_job_value_counts_all_ranks():
    import bench
    one = bench.job_gb_s(1, 300_000_000, 0.06)
    assert abs(bench.job_gb_s(2, 300_000_000, 0.06) - 2 * one) < 1e-9
    assert abs(one - 5000.0) < 1e-9
    assert bench.max_over_ranks([3.5, 1.0], "cpu") == [3.5, 1.0]  # world size 1


def test_reference_arm_under_torchrun_prints_from_rank0_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
