"""bench.py's multi-rank logic (independent replicas: barrier around the
timed region, max of the ranks' times, whole-job rate) with two gloo ranks on
the CPU, launched the way torchrun sets the environment."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    w, r, local = bench.dist_setup(world)
    bench.barrier(w)
    slowest = bench.barrier_max(w, 0.25 + 0.5 * r)  # rank 1 is the slow one
    rate = bench.job_rate(w, 1000, slowest)
    q.put((r, w, local, dist.get_backend(), slowest, rate))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for r, w, local, backend, slowest, rate in out:
        assert w == 2 and local == r and backend == "gloo"
        assert slowest == pytest.approx(0.75)       # max over ranks, seen by both
        assert rate == pytest.approx(2 * 1000 / 0.75)  # both replicas' units over the slowest time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.barrier_max(1, 0.5) == 0.5
    assert bench.job_rate(1, 300, 0.1) == pytest.approx(3000)


def test_traffic_records_match_source_and_shapes(tmp_path, monkeypatch):
    """roofline.traffic comes only from an ncu record of the same kernel source (sha256)
    and the same layer shapes; anything else gives no record (null traffic)."""
    import hashlib
    import json

    sys.path.insert(0, ROOT)
    import bench
    from ffn_side_attention_gb300 import synth

    src_dir = tmp_path / "ffn_side_attention_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src_dir / "gemm_tc.cu").write_bytes(b"kernel v1")
    sha = hashlib.sha256(b"kernel v1").hexdigest()
    recs = [dict(source_sha256=sha, H=4096, I=1536, dtype="bf16", workload="a", T=1),
            dict(source_sha256=sha, H=7168, I=5120, dtype="bf16", workload="b", T=2),
            dict(source_sha256="0" * 64, H=4096, I=1536, dtype="bf16", workload="c", T=3)]
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"gemm_tc.cu": recs}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    got = bench.recorded_traffic("gemm_tc.cu", synth.CONFIGS["qwen3_bf16"])
    assert [r["workload"] for r in got] == ["a"]
    assert [r["workload"] for r in bench.recorded_traffic("gemm_tc.cu", synth.CONFIGS["step3_bf16"])] == ["b"]
    assert bench.recorded_traffic("gemm_fp8.cu", synth.CONFIGS["qwen3_fp8"]) == []
    (src_dir / "gemm_tc.cu").write_bytes(b"kernel v2")  # the kernel changed since the capture
    assert bench.recorded_traffic("gemm_tc.cu", synth.CONFIGS["qwen3_bf16"]) == []


def test_gpus_flag_must_match_the_launch():
    """--gpus N without N ranks (WORLD_SIZE) is refused before any device work, instead of
    silently running one replica."""
    import subprocess

    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode != 0
    assert "--gpus 2 but WORLD_SIZE=1" in r.stderr


def test_per_batch_sweep_covers_every_decode_batch():
    """The default bench line's per_batch list: every (B, M) point of the Qwen3 bf16 layer,
    its fp8 variant, the three DeepSeek-V3 batches, Step3 as three micro-batches and the
    tiny fp32 layer -- 18 entries, no duplicates."""
    sys.path.insert(0, ROOT)
    import bench

    pts = bench.sweep_points()
    assert len(pts) == len(set(pts)) == 18
    q = {(b, m) for name, b, m, n in pts if name == "qwen3_bf16"}
    assert q == {(b, m) for b in (6, 48, 197, 395) for m in (1, 4, 8)}
    assert ("qwen3_fp8", 395, 4, 1) in pts and ("step3_bf16", 256, 8, 3) in pts and ("tiny_fp32", 32, 2, 1) in pts
    assert {(b, m) for name, b, m, n in pts if name == "dsv3_fp8"} == {(64, 8), (256, 8), (512, 8)}
