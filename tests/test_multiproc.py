"""The N>1 path of bench.py on CPU with the gloo backend (world size 2).

The hot path shards by independent units (ciphertexts); every rank runs its
own shard with no data-path collective, and the job's time is the max over
ranks.  This checks the rank logic bench.py uses: distinct input shards per
rank, the max-over-ranks reduction, the whole-job rate, and that the CPU
reference arm prints only on rank 0.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
from ntt_arithmetic_gb300 import inputs
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
local_ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
m = bench.max_over_ranks(local_ms)
seed = bench.rank_seed(rank)
x = inputs.uniform_residues((1, 2, 64), [97, 193], seed)
import torch
digests = [None] * world
dist.all_gather_object(digests, inputs.digest(x))   # test-only check of the shards
rate = bench.whole_job_rate(1056, world, m)
if rank == 0:
    print(json.dumps({{"max_ms": m, "rate": rate, "distinct_shards": len(set(digests)) == world}}))
dist.barrier()
dist.destroy_process_group()
"""


def _launch(script: str, world: int, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(world), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-3000:]
    return [o for o, _ in outs]


def test_gloo_world2_max_over_ranks_and_shards():
    outs = _launch(WORKER.format(root=ROOT), 2)
    import json
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["max_ms"] == 15.0
    assert abs(line["rate"] - 1056 * 2 / 15e-3) < 1e-6
    assert line["distinct_shards"]
    # rank 1 prints nothing of its own (some gloo builds log their connections)
    assert not [ln for ln in outs[1].splitlines() if ln.strip() and not ln.startswith("[Gloo]")]


def test_reference_arm_prints_only_on_rank0():
    """bench.py --impl reference: rank 0 runs the oracle sample and prints one
    JSON line; other ranks exit 0 without work (checked without running the
    oracle on rank 1)."""
    code = ("import sys; sys.path.insert(0, %r); import bench, types;"
            "bench.reference(types.SimpleNamespace(steps=1, warmup=0))" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, RANK="1", WORLD_SIZE="2"),
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.slow
def test_reference_arm_line_on_rank0():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
