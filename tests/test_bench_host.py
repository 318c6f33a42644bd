"""Host-side logic of bench.py, on CPU: the reference arm's JSON line, the
non-zero ranks of a multi-rank launch, the max-over-ranks reduction of the
timed region (gloo, world size 2), the kernel count per forward, the step
percentiles and the source-hash gate on recorded DRAM traffic."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True,
                       text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    return r.stdout


def test_reference_arm_prints_one_json_line():
    out = _run(["--impl", "reference", "--steps", "3", "--warmup", "3",
                "--reference-seconds", "3"])
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    out = _run(["--impl", "reference", "--steps", "3", "--warmup", "3"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.strip() == ""


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, cwd=ROOT)
    assert r.returncode != 0


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    q.put((rank, bench.max_over_ranks(10.0 + rank * 5.0, world)))
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    torch = pytest.importorskip("torch")
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get() for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_launch_count_per_forward():
    """gpu_launches counts three kernels per self-attention forward; cross-attention pairs its
    two projections in one bf16 launch only when both have more than 128 rows."""
    bench = _bench_module()
    from transformer_head_scaled_02_gb300 import workloads as wl
    assert bench.launches_per_step(wl.WORKLOADS["c3_bf16_causal"]) == 3
    assert bench.launches_per_step(wl.WORKLOADS["c5_bf16_cross"]) == 3
    few = wl.custom("few_q", B=2, T_q=64, T_kv=300, D=256, h=4, d_k=64, cross=True)
    assert bench.launches_per_step(few) == 4
    f32 = wl.custom("f32_cross", B=2, T_q=200, T_kv=300, D=64, h=4, d_k=16, dtype="f32", cross=True)
    assert bench.launches_per_step(f32) == 4


def test_step_percentiles():
    bench = _bench_module()
    s = bench.step_stats([0.1 * i for i in range(1, 11)])   # 0.1 .. 1.0
    assert s == {"p10": 0.19, "median": 0.55, "p90": 0.91}


def test_recorded_traffic_only_for_the_profiled_source(monkeypatch):
    """A DRAM figure is reported only while the kernel's source file hashes to the value the
    capture was taken on; any other source gives None."""
    bench = _bench_module()
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        d = json.load(f)
    e = d["c3_bf16_causal"]["attention"]
    assert bench.recorded_traffic("attention", "c3_bf16_causal", "attn_bf16.cu") == \
        (e["dram_bytes_per_launch"] if e["source_sha256_16"] == bench.kernel_source_hash("attn_bf16.cu")
         else None)
    assert bench.recorded_traffic("attention", "no_such_workload", "attn_bf16.cu") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda fname: "0" * 16)
    assert bench.recorded_traffic("attention", "c3_bf16_causal", "attn_bf16.cu") is None
