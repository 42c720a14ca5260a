"""The N > 1 launch path on the host: two gloo ranks under torchrun.

bench.py runs one replica per GPU with no data-path collective (the path
does not shard); what the ranks share is a barrier and the max over ranks of
the timed seconds, from which the whole-job value is computed.  The same
Dist logic runs here with the gloo backend on CPU tensors.
"""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DRIVER = r'''
import json, os, sys
sys.path.insert(0, {root!r})
os.chdir({root!r})
import bench
d = bench.Dist(backend="gloo")
d.barrier()
secs = 1.0 + 0.5 * d.rank          # this rank's timed seconds
t_max = d.max(secs)
units = 100.0                       # units one rank processed
value = units * d.world / t_max     # whole-job throughput, as bench reports it
with open(os.path.join({out!r}, f"rank{{d.rank}}.json"), "w") as f:
    json.dump({{"rank": d.rank, "world": d.world, "t_max": t_max, "value": value}}, f)
d.close()
'''


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_share_barrier_and_max(tmp_path):
    script = tmp_path / "driver.py"
    script.write_text(DRIVER.format(root=ROOT, out=str(tmp_path)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", str(script)]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    res = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert [x["rank"] for x in res] == [0, 1]
    for x in res:
        assert x["world"] == 2
        assert x["t_max"] == 1.5          # the slower rank's seconds, on every rank
        assert x["value"] == 100.0 * 2 / 1.5


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    """Under torchrun only rank 0 times the oracle; the others return without
    work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload, rel, kv, steps, warmup = "local_decode", "f32", "bf16", 1, 0

    assert bench.reference(Args()) is None
    assert capsys.readouterr().out == ""
