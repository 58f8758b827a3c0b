"""The benchmark's multi-rank path on CPU: two gloo ranks under torchrun agree on
the maximum of their timed regions (the value every rank reports), with the
barrier around it."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_dist_max_two_gloo_ranks(tmp_path):
    pytest.importorskip("torch.distributed")
    script = tmp_path / "ranks.py"
    script.write_text(
        "import json, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import torch\n"
        "import bench\n"
        "world, rank, local = bench.dist_setup()\n"
        "bench.dist_barrier(world)\n"
        "m = bench.dist_max(float(10 * rank + 3), world)\n"
        "bench.dist_barrier(world)\n"
        f"open({str(tmp_path)!r} + f'/rank{{rank}}.json', 'w').write("
        "json.dumps({'rank': rank, 'world': world, 'max': m}))\n"
        "torch.distributed.destroy_process_group()\n")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(script)]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=240)
    assert out.returncode == 0, out.stderr[-2000:]
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in (0, 1)]
    assert sorted(r["rank"] for r in res) == [0, 1]
    assert all(r["world"] == 2 and r["max"] == 13.0 for r in res)


def test_valid_pair_count_closed_form():
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    cu = np.array([0, 100, 256])
    assert bench.valid_pairs(cu, True) == 100 * 101 // 2 + 156 * 157 // 2
    assert bench.valid_pairs(cu, False) == 100 * 100 + 156 * 156


def test_item_pair_count_matches_oracle():
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import oracle
    rng = np.random.default_rng(0)
    for _ in range(200):
        T = int(rng.integers(1, 200))
        nd = int(rng.integers(1, min(T, 6) + 1))
        cuts = np.sort(rng.choice(np.arange(1, T), size=nd - 1, replace=False)) if nd > 1 else []
        cu = np.concatenate([[0], cuts, [T]]).astype(np.int32)
        qa = int(rng.integers(0, T))
        qb = int(rng.integers(qa + 1, T + 1))
        ka = int(rng.integers(0, T))
        kb = int(rng.integers(ka + 1, T + 1))
        for causal in (True, False):
            assert bench.valid_pairs_range(cu, causal, [0, 0, 0, qa, qb, ka, kb]) == \
                oracle.valid_pairs(cu, causal, qa, qb, ka, kb)
