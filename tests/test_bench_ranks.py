"""Host logic of the benchmark on CPU: every rank of a gloo run reports the
slowest rank's time (world size 2); the byte model; the traffic record's
source hash; the reference arm's JSON line and its rank handling."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_bench_byte_model():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from gated_deltanet_decode_gb300 import inputs as I
    s = I.QWEN_08B
    b = bench.layer_bytes(s, s.rows)
    state = 64 * 16 * 128 * 128 * 4 * 2
    assert state == 134217728
    assert state < b < state * 1.06          # conv, vectors and parameters add under 6%
    assert bench.layer_bytes(s, 0) < 0.01 * state   # padding rows move no state


def test_recorded_traffic_follows_kernel_source(tmp_path, monkeypatch):
    """The roofline's traffic figure is read from the ncu summary only while
    the summary's source hash matches the kernel sources."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    sha = bench.kernel_source_sha()
    p = tmp_path / "summary.md"
    p.write_text(f"text\n\n- traffic_per_launch_bytes: 1234\n- source_sha256: {sha}\n")
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(p))
    assert bench.recorded_traffic() == 1234
    p.write_text("- traffic_per_launch_bytes: 1234\n- source_sha256: " + "0" * 64 + "\n")
    assert bench.recorded_traffic() is None


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    import shutil
    import sys
    sys.path.insert(0, ROOT)
    import bench
    for p in bench.KERNEL_SOURCES:
        dst = tmp_path / p
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, p), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha()
    first = tmp_path / bench.KERNEL_SOURCES[0]
    text = first.read_text()
    first.write_text("// a new comment\n/* and a block\n   comment */\n\n" + text)
    assert bench.kernel_source_sha() == h0
    first.write_text(text.replace("kMaxStages = 8", "kMaxStages = 7"))
    assert bench.kernel_source_sha() != h0


def _run_reference(env_extra):
    import json
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_line():
    """The reference arm (the oracle on the host cores) prints one line with
    the same metric keys as the CUDA arm, its own CPU baseline and an
    end-to-end figure with no host-device traffic."""
    (line,) = _run_reference({"RANK": "0", "WORLD_SIZE": "1"})
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] and line["dtype"] == "f64" and line["data"] == "synthetic"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_no_work():
    """Under a multi-rank launch only rank 0 runs and prints the oracle."""
    assert _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
