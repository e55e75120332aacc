"""Host-side logic of bench.py without a GPU: the replicas-only reductions
over ranks (world size 2, gloo) and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(world, 1.5 + rank), bench.sum_over_ranks(world, 10.0 * (rank + 1))))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_rank_reductions_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--reference-rows", "64"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_kernel_source_hash_ignores_comments_only():
    """traffic.json entries are keyed on the kernels' code: editing a comment
    or whitespace keeps the key, editing code changes it."""
    sys.path.insert(0, ROOT)
    import bench
    base = "int f(int x) {\n    return x + 1;  // one more\n}\n/* block\n comment */\n"
    assert bench.code_text(base) == bench.code_text(base.replace("// one more", "// another note"))
    assert bench.code_text(base) == bench.code_text(base.replace("    return", "\treturn"))
    assert bench.code_text(base) == bench.code_text(base.replace("/* block\n comment */", ""))
    assert bench.code_text(base) != bench.code_text(base.replace("x + 1", "x + 2"))
    assert bench.code_text(base) == "int f(int x) { return x + 1; }"
