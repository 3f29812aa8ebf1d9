"""The multi-replica path of bench.py on CPU: two ranks over gloo (world size 2).

One process per GPU runs an independent replica; the job's time is the slowest rank's (a
max-reduction, the only collective) and its throughput counts every rank's tokens.  The
reference arm runs on rank 0 alone; other ranks return at once.
"""
import contextlib
import io
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        elapsed = 1.5 + rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed, "cpu")
        value = bench.whole_job_value(world, 4, 10, slowest)
        dist.barrier()
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_count_all_tokens():
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in out:
        assert slowest == 2.5
        assert value == 2 * 4 * 10 / 2.5


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.whole_job_value(1, 32, 100, 2.0) == 1600.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference"])
        bench.run_reference(bench.parse())
    assert buf.getvalue() == ""  # no work and no line on a non-zero rank


def test_reference_line_has_the_gpu_arm_config_and_its_own_time(monkeypatch):
    # the reference arm's line describes the GPU arm's workload (one function builds both
    # configs), and its ms_per_step is a step as it ran, so steps x ms_per_step fits in its time
    import json
    import bench
    import synth
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--workload", "tiny_f32",
                                         "--steps", "4", "--warmup", "1"])
        args = bench.parse()
        bench.run_reference(args)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    w = bench.WORKLOADS["tiny_f32"]
    blob = synth.model_blob(w.shape, w.seed_weights)
    assert line["config"] == bench.workload_config(w, args, 1, bench.blob_step_bytes(w, blob))
    assert line["impl"] == "reference" and line["steps"] == 4
    assert line["steps"] * line["ms_per_step"] <= line["wall_s"] * 1e3
    assert line["ms_per_token"] >= line["ms_per_step"]
    assert abs(line["value"] - 1e3 / line["ms_per_token"]) < 1e-9 * line["value"]


def test_step_roofline_fields():
    import bench
    # 15.28 GB per step at batch 1: 444.3 tok/s at the measured 6788 GB/s, 523.6 at 8 TB/s
    r = bench.step_roofline(15.28e9, 1, 6788.3, 352.7, 100, 100 * 15.28e9 / 5.389e12)
    assert abs(r["roofline_tok_s"] - 6788.3e9 / 15.28e9) < 1e-9
    assert abs(r["frac_of_roofline"] - 352.7 / (6788.3e9 / 15.28e9)) < 1e-12
    assert abs(r["roofline_tok_s_nominal_8tbs"] - 8000e9 / 15.28e9) < 1e-9
    assert abs(r["frac_of_nominal_8tbs"] - 352.7 * 15.28e9 / 8000e9) < 1e-12
    assert abs(r["hbm_gbs_achieved"] - 5389.0) < 1e-6


def test_kernel_function_text_finds_the_definition():
    import bench
    src = ("void k(int a);\n__global__ void __launch_bounds__(256, 1) k(const A a, int n) {\n"
           "  if (n) { f((n)); }\n}\nvoid other() {}\n")
    body = bench.kernel_function_text(src, "k")
    assert body.startswith("k(const A a, int n) {") and body.endswith("}") and "other" not in body
    assert bench.kernel_function_text(src, "missing") is None


def test_profile_summaries_are_self_describing():
    # every committed ncu summary names the command that made it (committed files only) and,
    # where the bench reads traffic from it, the kernel it measured and the bytes per launch
    import glob
    import os
    import re
    import bench
    files = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")))
    assert files
    for p in files:
        text = open(p).read()
        assert "```" in text and ("ncu " in text), p
        assert "_work" not in text and "_out/" not in text, p
        if "traffic_bytes_per_launch" in text:
            assert re.search(r"traffic_bytes_per_launch:\s*\d+", text), p
            assert re.search(r"kernel_function:\s*\w+", text) and re.search(r"kernel_function_sha256_16:\s*[0-9a-f]{16}", text), p
