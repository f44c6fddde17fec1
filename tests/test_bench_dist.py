"""The multi-rank plumbing of bench.py on CPU: two ranks over gloo, launched
the way the benchmark driver launches N > 1 (torch.distributed.run on
127.0.0.1).  Each rank of the CUDA arm runs an independent replica; the only
cross-rank steps are the barriers around the timed region and the max of the
step time, which these tests exercise."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, extra_env=None, timeout=240):
    env = dict(os.environ, BENCH_BACKEND="gloo", PYTHONPATH=ROOT)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    if extra_env:
        env.update(extra_env)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_dist_max_and_barrier_over_two_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(
        "import sys, json\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "d = bench.Dist()\n"
        "assert d.world == 2\n"
        "d.barrier()\n"
        "v = d.max(10.0 + d.rank)\n"
        "d.barrier()\n"
        f"open({str(tmp_path)!r} + f'/rank{{d.rank}}.json', 'w').write(json.dumps({{'rank': d.rank, 'max': v}}))\n"
        "d.close()\n")
    r = _torchrun([str(script)])
    assert r.returncode == 0, r.stderr[-2000:]
    # each rank writes its own file (two processes share one stdout pipe)
    got = [json.loads((tmp_path / f"rank{k}.json").read_text()) for k in range(2)]
    assert sorted(g["rank"] for g in got) == [0, 1]
    assert all(g["max"] == 11.0 for g in got)


def test_reference_arm_prints_one_line_from_rank_zero():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                   "--warmup", "0", "--workload", "blobs_2k_d2"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"]["sample_points"] == 2000 and line["config"]["n"] == 2000
    # the value is pair evaluations per second of the points actually run
    assert line["value"] == pytest.approx(2000 * 2000 / (line["ms_per_step"] * 1e-3), rel=1e-9)
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_kernel_code_hash_ignores_comments_only():
    # the recorded ncu traffic stays valid across comment edits, not code edits
    import bench
    code = ["int f(int x) {\n    return x + 1;\n}\n", "#define N 4\n"]
    commented = ["// f adds one\nint f(int x) {   /* body */\n\n    return x + 1;  // done\n}\n",
                 "/* size\n   of it */\n#define N 4\n"]
    changed = ["int f(int x) {\n    return x + 2;\n}\n", "#define N 4\n"]
    assert bench.kernel_code_hash(code) == bench.kernel_code_hash(commented)
    assert bench.kernel_code_hash(code) != bench.kernel_code_hash(changed)
    assert bench.kernel_code_hash() == bench.kernel_code_hash(None)
