"""bench.py's multi-rank host logic on two CPU processes (gloo, 127.0.0.1):
the step time is the slowest rank's, the value is the whole job's (weak
scaling: world_size x each rank's tokens), and the reference arm prints one
line from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.join(HERE, "gloo_worker.py")],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=300)
            assert p.returncode == 0, err[-2000:]
            outs.append([json.loads(l) for l in out.splitlines() if l.startswith("{")])
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    results = [o[-1] for o in outs]
    for rank, r in enumerate(results):
        assert r["rank"] == rank and r["world_size"] == 2 and r["local_rank"] == rank
        assert r["max_ms"] == 3.0                      # the slower rank's time
        assert r["value"] == pytest.approx(2 * 1000 / 3e-3)
    # the reference line: rank 0 only, one line, reporting the job's two ranks
    ref0 = [l for l in outs[0] if l.get("impl") == "reference"]
    ref1 = [l for l in outs[1] if l.get("impl") == "reference"]
    assert len(ref0) == 1 and not ref1
    line = ref0[0]
    assert line["n_gpus"] == 2 and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
