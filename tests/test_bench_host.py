"""Host-side logic of bench.py, on CPU: the algorithmic byte and flop counts, the rank plumbing of
multi-process runs (world size 2 over gloo), the reference arm's JSON line, and the lookup of
profiled DRAM traffic by source hash."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

import bench  # noqa: E402


def test_comba_byte_formula_matches_the_spec():
    # KBench comba_decode_step flops_src: at K = V = 128 the state is "99.1%" of the bytes.
    with open(os.path.join(GOLDEN, "comba_bytes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for K, V, pct in rows:
        K, V, pct = int(K), int(V), float(pct)
        for B, H in [(1, 1), (256, 32), (1024, 16)]:
            share = 100.0 * 2 * B * H * K * V * 4 / bench.comba_bytes(B, H, K, V)
            assert abs(share - pct) <= 0.1


def test_algorithmic_work_of_the_workloads():
    # byte counts written out by hand from the layouts in include/gdn.h
    assert bench.decode_bytes(64, 16, 32, 128, 128) == (
        2 * 64 * 32 * 128 * 128 * 4            # state read + write
        + 2 * 64 * 16 * 128 * 2                # q, k
        + 64 * 32 * 128 * 2 + 64 * 32 * 4 + 64 * 32 * 2   # v, g, beta
        + 64 * 32 * 128 * 2)                   # y
    assert bench.comba_bytes(256, 32, 128, 128) == 1_084_276_736
    T = 15360
    assert bench.prefill_bytes([4096, 2048, 1024, 8192], 16, 32, 128, 128) == (
        2 * T * 16 * 128 * 2 + T * 32 * 128 * 2 + 2 * T * 32 * 2 + T * 32 * 128 * 2
        + 2 * 4 * 32 * 128 * 128 * 4 + 4 * 8 + 5 * 8 + 2 * 32 * 4)
    chunks = 64 + 32 + 16 + 128
    assert bench.prefill_flops([4096, 2048, 1024, 8192], 32, 128, 128, 64) == (
        T * 32 * 2 * (3 * 64 * 128 + 2 * 64 * 128 + 3 * 128 * 128) + chunks * 32 * 64 ** 3 // 3)
    C = (2 * 16 + 48) * 128
    verify = 32 * 128 * 48 * 128 * 4 + (32 * 8 * C + 32 * C * 3 + 2 * 32 * 8 * 48
                                        + 2 * 32 * 8 * 48 * 128) * 4 + (C * 4 + 2 * 48 + 128) * 4
    assert bench.window_bytes(32, 16, 48, 128, 8, False) == verify
    assert bench.window_bytes(32, 16, 48, 128, 8, True) == verify + 32 * 128 * 48 * 128 * 4 + 32 * C * 3 * 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench as b
    d = b.Dist()
    d.barrier()
    m = d.max(float(rank + 1) * 1.5)
    d.close()
    q.put((rank, m))


def test_two_ranks_take_the_max_over_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 3.0), (1, 3.0)]


def test_reference_arm_prints_one_line():
    env = dict(os.environ)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # under torchrun, ranks other than 0 do no work and print nothing
    env.update(RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, env=env,
                       timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_traffic_rows_follow_their_sources(tmp_path, monkeypatch):
    # a row counts only while the hash of its source (one file, or several hashed in order) matches
    import hashlib
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cuh").write_bytes(b"kernel v1")
    (tmp_path / "k.cu").write_bytes(b"launch v1")
    one = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    two = hashlib.sha256(b"kernel v1" + b"launch v1").hexdigest()[:16]
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel sha bytes\n"
        f"single_kernel {one} 123 capture\n"
        f"pair_kernel {two} 456 capture\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("single_kernel", "k.cuh") == 123
    assert bench.profiled_traffic("pair_kernel", ("k.cuh", "k.cu")) == 456
    assert bench.profiled_traffic("pair_kernel", ("k.cu", "k.cuh")) is None  # order matters
    assert bench.profiled_traffic("pair_kernel", "k.cuh") is None
    (tmp_path / "k.cu").write_bytes(b"launch v2")  # the launch shape changed: the row is stale
    assert bench.profiled_traffic("pair_kernel", ("k.cuh", "k.cu")) is None
    assert bench.profiled_traffic("missing", "nope.cuh") is None
