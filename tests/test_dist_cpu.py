"""Rank bookkeeping of bench.py's multi-GPU mode, on CPU with gloo (world size 2).

Sequences are independent, so N > 1 runs one replica per rank with its own
seeded batch and no collective on the data path; only the timing reduction
(max over ranks) and the barrier cross ranks.
"""
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import os, sys, json
    sys.path.insert(0, {root!r})
    import torch
    import bench
    from paged_kv_cache_493_b300 import workloads as W
    rank, world, local = bench.dist_setup()
    assert torch.distributed.get_backend() == "gloo"
    t = 1.0 + 2.0 * rank
    m = bench.reduce_max(t)
    bench.barrier()
    case = W.tiny_decode(seed=bench.replica_seed(1001, rank))
    print(json.dumps({{"rank": rank, "world": world, "max": m,
                      "q0": float(case.q.float().sum())}}))
    torch.distributed.destroy_process_group()
""")


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_rank_replicas_on_gloo(tmp_path):
    script = tmp_path / "child.py"
    script.write_text(CHILD.format(root=ROOT))
    port = free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err
        outs.append(__import__("json").loads(out.strip().splitlines()[-1]))
    assert {o["rank"] for o in outs} == {0, 1}
    assert all(o["world"] == 2 and o["max"] == 3.0 for o in outs)
    assert outs[0]["q0"] != outs[1]["q0"]          # each replica draws its own batch


def test_reference_arm_under_two_ranks_prints_one_line():
    """`bench.py --impl reference --gpus 2` starts two ranks itself (torchrun,
    gloo here); rank 0 alone times the oracle and prints one JSON line, rank
    1 exits 0 without work."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "1"], env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = __import__("json").loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["cores"] >= 1 and line["value"] > 0
