"""The N > 1 path of bench.py on CPU: two ranks over gloo (127.0.0.1), as
torchrun launches them.  The product path does not shard across GPUs (each
rank is an independent replica), so what runs on more than one rank is the
host logic: rendezvous, barrier, the max of the ranks' times and the sum of
their work, and the reference arm printing on rank 0 alone.  One more test
runs the reference arm on one rank and checks its line's contract keys."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup()
assert world == 2 and rank in (0, 1)
bench.barrier(world)
mx = bench.max_over_ranks(1.5 + rank, world)        # per-rank times 1.5, 2.5
sm = bench.sum_over_ranks(10.0 * (rank + 1), world)  # per-rank work 10, 20
print(json.dumps({{"rank": rank, "max": mx, "sum": sm}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code_or_args, timeout=240):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        cmd = [sys.executable, "-c", code_or_args] if isinstance(code_or_args, str) else [sys.executable, *code_or_args]
        procs.append(subprocess.Popen(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        finally:
            if p.poll() is None:
                p.kill()
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_rank_reductions_over_gloo():
    outs = _launch(_CHILD.format(root=ROOT))
    got = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(g["rank"] for g in got) == [0, 1]
    for g in got:
        assert g["max"] == 2.5      # the slowest rank's time
        assert g["sum"] == 30.0     # every rank's work


def test_reference_arm_prints_on_rank_zero_only():
    outs = _launch(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"])
    lines = [[l for l in o.splitlines() if l.startswith("{")] for o in outs]
    assert len(lines[0]) == 1 and lines[1] == []
    d = json.loads(lines[0][0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["parallelism"] == "replicas x2"


def test_reference_arm_line_has_the_contract_keys():
    # one rank: the reference arm's JSON line carries the keys the bench
    # contract asks for, with the headline's metric and config
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    sys.path.insert(0, ROOT)
    import bench
    assert d["metric"] == bench.METRIC and d["config"] == bench.decode_config(80, 1)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
