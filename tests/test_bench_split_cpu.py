"""The benchmark's sequence-parallel split, on CPU with two gloo ranks under
torchrun: GPU g runs the schedule items of the virtual ranks r with
r mod N = g. Each rank computes its share of four workloads' schedules (Zigzag,
TASP, Ring; as built and cut at document boundaries); the test then checks
that every schedule item went to exactly one rank, that each rank's output
rows are exactly the Q chunks its virtual ranks own (no row written by two
GPUs, none left out), that the FLOP shares add up to the workload's, and that
the ranks' per-GPU times gather in rank order."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

WORKLOADS = [1, 2, 3, 4]  # the bf16 workloads: zigzag P=8, TASP P=8, ring P=16, TASP P=32


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _merge(spans):
    out = []
    for a, b in sorted(spans):
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return [tuple(x) for x in out]


def test_split_partitions_items_and_rows_two_gloo_ranks(tmp_path):
    pytest.importorskip("torch.distributed")
    import sequence_blockwise_gb300 as sb
    sb.load()  # build once here, not in both ranks at the same time
    script = tmp_path / "ranks.py"
    script.write_text(
        "import json, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import numpy as np, torch\n"
        "import bench\n"
        "import sequence_blockwise_gb300 as sb\n"
        "from sequence_blockwise_gb300 import workloads as wl\n"
        "world, rank, local = bench.dist_setup()\n"
        "res = {'rank': rank, 'world': world, 'gathered': bench.dist_gather(rank + 0.5, world), 'w': {}}\n"
        f"for i in {WORKLOADS!r}:\n"
        "    w = wl.WORKLOADS[i]\n"
        "    cu = wl.cu_seqlens(w)\n"
        "    built = sb.sp_schedule_build(w.kind, w.P, w.T, cu, w.causal, seed=w.seed)\n"
        "    for cut, items in ((0, built), (1, sb.sp_schedule_split_documents(built, cu, w.causal))):\n"
        "        mine = bench.split_items(items, world, rank)\n"
        "        res['w'][w.name + str(cut)] = {\n"
        "            'items': mine.tolist(),\n"
        "            'rows': bench.row_intervals(mine),\n"
        "            'pairs': int(sum(bench.valid_pairs_range(cu, w.causal, it) for it in mine))}\n"
        "bench.dist_barrier(world)\n"
        f"open({str(tmp_path)!r} + f'/rank{{rank}}.json', 'w').write(json.dumps(res))\n"
        "torch.distributed.destroy_process_group()\n")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(script)]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-3000:]
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in (0, 1)]
    assert [r["rank"] for r in res] == [0, 1] and all(r["world"] == 2 for r in res)
    assert all(r["gathered"] == [0.5, 1.5] for r in res)

    import bench
    from sequence_blockwise_gb300 import workloads as wl
    for i, cut in [(i, c) for i in WORKLOADS for c in (0, 1)]:
        w = wl.WORKLOADS[i]
        cu = wl.cu_seqlens(w)
        items = sb.sp_schedule_build(w.kind, w.P, w.T, cu, w.causal, seed=w.seed)
        if cut:  # the items as the benchmark runs them: cut at document boundaries
            items = sb.sp_schedule_split_documents(items, cu, w.causal)
        key_w = w.name + str(cut)
        got = [np.array(r["w"][key_w]["items"], dtype=np.int32).reshape(-1, 8) for r in res]
        # Every item exactly once, each on the GPU of its virtual rank.
        both = np.concatenate(got)
        assert len(both) == len(items)
        key = lambda a: sorted(map(tuple, a.tolist()))
        assert key(both) == key(items)
        for g, mine in enumerate(got):
            assert (mine[:, 0] % 2 == g).all()
        # Each GPU writes exactly the Q chunks its virtual ranks own.
        rows = [[tuple(x) for x in r["w"][key_w]["rows"]] for r in res]
        for g in range(2):
            own = _merge([c for vr in range(g, w.P, 2) for c in bench.owned_chunks(w.kind, w.P, w.T, vr)])
            assert rows[g] == own, (w.name, g)
        # The two GPUs' rows are disjoint and cover [0, T).
        assert _merge(rows[0] + rows[1]) == [(0, w.T)]
        assert sum(b - a for a, b in rows[0]) + sum(b - a for a, b in rows[1]) == w.T
        # FLOP shares add up to the workload's.
        assert sum(r["w"][key_w]["pairs"] for r in res) == bench.valid_pairs(cu, w.causal)


def test_owned_chunks_and_row_intervals():
    import bench
    # Zigzag P = 2 over 8 tokens: rank 0 owns chunks 0 and 3, rank 1 chunks 1 and 2.
    assert bench.owned_chunks(1, 2, 8, 0) == [(0, 2), (6, 8)]
    assert bench.owned_chunks(1, 2, 8, 1) == [(2, 4), (4, 6)]
    # Ring: the first T mod P chunks get one more token.
    assert [bench.owned_chunks(0, 3, 10, r) for r in range(3)] == [[(0, 4)], [(4, 7)], [(7, 10)]]
    items = np.array([[0, 0, 0, 0, 4, 0, 4, 0], [0, 1, 0, 0, 4, 7, 10, 0], [2, 0, 0, 7, 10, 7, 10, 0],
                      [2, 1, 0, 9, 12, 0, 4, 0]], dtype=np.int32)
    assert bench.row_intervals(items) == [(0, 4), (7, 12)]
    assert bench.split_items(items, 2, 0).tolist() == items.tolist()
    assert len(bench.split_items(items, 2, 1)) == 0
