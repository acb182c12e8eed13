"""bench.py's N>1 path on the host: two gloo ranks launched the way the
benchmark driver launches N GPUs (torch.distributed.run on 127.0.0.1) check
the max/sum reductions over ranks, the barrier, the whole-job (weak-scaling)
throughput every rank agrees on, and that only rank 0 runs the reference arm.
No GPU and no data-path collective are involved: the decode path shards by
sequence."""
import os
import socket
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_job_throughput():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(HERE, "_multirank_worker.py")]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "MULTIRANK_OK world=2" in r.stdout
