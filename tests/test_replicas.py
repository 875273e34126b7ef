"""Host logic of the benchmark, on CPU: the replicas-only multi-GPU mode with two gloo ranks
(the job time is the maximum over ranks, the reference arm runs on rank 0 only), the
reference arm's JSON line, and the algorithmic byte count behind the roofline."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
sys.path.insert(0, sys.argv[1])
import torch, torch.distributed as dist
import bench
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo")
v = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
dist.barrier()
print(f"rank{rank} max={v}", flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = []
    for p in procs:
        out, _ = p.communicate(timeout=180)
        outs.append(out)
        assert p.returncode == 0, out
    for r, out in enumerate(outs):
        assert f"rank{r} max=15.0" in out, out


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25


def test_reference_arm_rank_nonzero_does_no_work(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        cpu_seconds, steps, warmup, gpus = 1.0, 1, 1, 2
    bench.run_reference(A(), None, rank=1)
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference on the host cores: one JSON line with the contract's keys,
    the oracle as the CPU baseline, no host-device traffic."""
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny-4k", "--steps", "2", "--warmup", "1", "--cpu-seconds", "0.5"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["config"]["workload"] == "tiny-4k"
    assert d["value"] > 0 and d["higher_is_better"] is False and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_bench_counts_algorithmic_bytes_from_the_selection():
    """The bench's byte count on a hand-made unit: the union of the heads' choices, the
    anchors of a grown window, and the residual items, checked against numbers worked out
    by hand (C = 3 clusters x L = 2 subclusters, G = 2 heads, top 2 x 1, P = 4 splits)."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench

    class Lay:
        units, c_max, l_max, group, sub_off_stride = 1, 3, 2, 2, 7

    class H:
        arrays = {"unit_info": np.array([[3, 2, 100, 21, 4, 90, 0, 0]], np.int32),
                  "sub_off": np.array([[0, 5, 8, 10, 14, 20, 21]], np.int32)}

        def layout(self):
            return Lay()

        def array(self, name, dtype, shape):
            return torch.from_numpy(self.arrays[name].reshape(shape))

        def splits(self):
            return 4

    class W:
        top_c, top_s = 2, 1

    # head 0 chose clusters 0 (subcluster 1) and 2 (subcluster 0); head 1 chose cluster 2
    # (subcluster 1) and nothing else
    sel = np.array([[0, 2, 1, 0], [2, -1, 1, -1]], np.int32)
    by = bench.bytes_from_selection(H(), W(), sel, np.array([100]), [100])
    # union rows 3 + 6 + 1 = 10, anchors 4 sinks + (100 - 90) recent = 14
    assert by["rows"] == 24
    assert by["select"] == 512 + 3 * 1028 + 2 * (2 * 1032 + 4) + 3 * 12 + 7 * 16
    assert by["attend"] == 512 + 3 * 12 + 10 * 4 + 24 * 512 + 7 * (512 + 16) + 4 * 2 * 132 * 4
    assert by["merge"] == 4 * 2 * 132 * 4 + 2 * 128 * 4
    assert by["step"] == by["select"] + by["attend"] + by["merge"]
    # fp8 summaries: 1 byte a mean or variance element, the terms' value means' high parts
    b8 = bench.bytes_from_selection(H(), W(), sel, np.array([100]), [100], sb=1)
    assert b8["select"] == 512 + 3 * (2 * 128 + 4) + 2 * (2 * (2 * 128 + 8) + 4) + 3 * 12 + 7 * 16
    assert b8["attend"] == 512 + 3 * 12 + 10 * 4 + 24 * 512 + 7 * (256 + 16) + 4 * 2 * 132 * 4
    # the feature-map residual: no Gaussian terms in the rows kernel; per head the unit's
    # feature sums and those of its chosen subclusters (32 x 132 floats each), 33 vectors out
    bf = bench.bytes_from_selection(H(), W(), sel, np.array([100]), [100], resid=2)
    row, vec = 32 * 132 * 4, 33 * 132 * 4
    assert bf["attend"] == 512 + 3 * 12 + 10 * 4 + 24 * 512 + 4 * 2 * 132 * 4
    assert bf["fm"] == (256 + 4 * 4 + 3 * row + vec) + (256 + 4 * 4 + 2 * row + vec)
    assert bf["merge"] == 4 * 2 * 132 * 4 + 2 * 128 * 4 + 2 * (vec + 4)
    assert bf["step"] == bf["select"] + bf["attend"] + bf["merge"] + bf["fm"]
