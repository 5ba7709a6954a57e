"""bench.py's host logic on the CPU: the multi-rank reductions over gloo with
two ranks (the job value is the bytes of all ranks over the slowest rank's
time), the reference arm under a two-rank torchrun launch (rank 0 alone
prints one JSON line), and the algorithmic byte count of a decode call."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    r, w, local = bench.dist_setup(world)
    ms = 10.0 + 5.0 * r             # rank 1 is the slower one
    nbytes = 1e9 * (r + 1)
    bench.barrier(w)
    ms_max = bench.max_over_ranks(ms, w, "cpu")
    total = bench.sum_over_ranks(nbytes, w, "cpu")
    value = total / (ms_max * 1e-3) / 1e9
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "ms_max": ms_max, "total": total, "value": value}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_reductions_over_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, rec in enumerate(res):
        assert rec["rank"] == r and rec["world"] == 2 and rec["local"] == r
        assert rec["ms_max"] == 15.0          # the slowest rank's time
        assert rec["total"] == 3e9            # all ranks' bytes
        assert rec["value"] == pytest.approx(3e9 / 15e-3 / 1e9)


def test_single_rank_reductions_are_identity():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.sum_over_ranks(2.0, 1, "cpu") == 2.0
    bench.barrier(1)


def test_reference_arm_under_two_rank_launch():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--batch", "8"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def test_call_bytes_counts_every_stream():
    lens = np.array([0, 5, 127, 128, 1000], np.int32)
    B = lens.size
    kv = int(lens.sum()) * 2 * bench.HKV * bench.D * 2           # cached K and V
    qo = 2 * B * bench.HQ * bench.D * 2                            # q in, out
    new = 2 * B * 2 * bench.HKV * bench.D * 2                      # new K/V read and appended
    table = 4 * int(sum((L + 1 + bench.P - 1) // bench.P for L in lens))
    assert bench.call_bytes(lens, B) == kv + qo + new + table + 4 * B


def test_timed_steps_span_the_whole_cycle():
    cap = bench.DECODE_CAPACITY
    assert bench.timed_decode_steps(cap) == list(range(cap))  # one full cycle: every step once
    for k in (1, 3, 5, 20, 100, 600):
        steps = bench.timed_decode_steps(k)
        assert len(steps) == k and all(0 <= s < cap for s in steps)
        if k <= cap:
            assert steps == sorted(set(steps))  # distinct, in cycle order
        # the mean decode step of the sample is the cycle's mean, within half a stride
        assert abs(np.mean(steps) - (cap - 1) / 2) <= cap / (2 * k) + 0.5
    assert bench.timed_decode_steps(20)[0] < 32 and bench.timed_decode_steps(20)[-1] > cap - 32
