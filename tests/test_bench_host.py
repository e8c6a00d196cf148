"""Host-side logic of bench.py on the CPU: the max-over-ranks reduction with
two gloo ranks, and the reference arm's JSON line (the oracle on the host)."""

import json
import os
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
    bench.barrier(world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    assert out == [(0, 15.0), (1, 15.0)]


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    # the same workload keys as the GPU arm's line, the default workload
    import bench
    from head_scaled_dot_gb300 import workloads
    w = workloads.WORKLOADS[3]
    lens = [int(x) for x in workloads.make_inputs(w)["valid_len"]]
    for k, v in bench.workload_config(w, lens).items():
        assert d["config"][k] == v, k
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True


def test_stored_traffic_entries_name_existing_sources_and_profiles():
    """profiles/traffic.json (the per-launch DRAM bytes the benchmark line
    reports beside its roofline) names, for every entry, a kernel source of
    the package, its hash and the committed ncu summary the bytes come from;
    the bench looks an entry up only while the hash matches the source."""
    sys.path.insert(0, ROOT)
    import bench
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    assert set(table) <= {"attention", "qkv_projection", "output_projection", "decode"}
    for kernel, entries in table.items():
        for workload, e in entries.items():
            src = os.path.join(ROOT, "head_scaled_dot_gb300", "csrc", e["source"])
            assert os.path.exists(src), (kernel, workload)
            assert len(e["source_sha256_16"]) == 16
            assert isinstance(e["dram_bytes_per_launch"], int) and e["dram_bytes_per_launch"] > 0
            summary = e["from"].split("profiles/")[-1]
            assert os.path.exists(os.path.join(ROOT, "profiles", summary)), summary
            got = bench.stored_traffic(kernel, workload)
            if bench.source_hash(src) == e["source_sha256_16"]:
                assert got == e["dram_bytes_per_launch"]
            else:
                assert got is None
