"""Multi-process host logic of bench.py on CPU (world_size 2, gloo,
127.0.0.1): the barrier, the max over ranks of the timed region, and the
reference arm under torch.distributed.run (rank 0 alone runs and prints)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    ws, r, local = bench.dist_env()
    bench.barrier(ws)
    m = bench.max_over_ranks(1.5 + rank, ws)
    out.put((r, ws, local, m))
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 2.5), (1, 2, 1, 2.5)]


def test_reference_arm_prints_once_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_fingerprint_ignores_comments_only():
    # roofline.traffic is reported only while the kernel sources match the
    # capture: comment or whitespace edits keep the fingerprint, code edits do not
    sys.path.insert(0, ROOT)
    import bench
    src = {f: open(os.path.join(ROOT, "tiled_scaled_dot_gb300", "csrc", f)).read()
           for f in bench.KERNEL_SOURCES["backward"]}
    base = bench.kernel_fingerprint("backward", read=lambda f: src[f])
    assert base == bench.kernel_fingerprint("backward")
    f0 = bench.KERNEL_SOURCES["backward"][0]
    commented = dict(src)
    commented[f0] = "// a new comment\n/* and a block\n comment */\n" + src[f0].replace("\n", "\n\n", 3)
    assert bench.kernel_fingerprint("backward", read=lambda f: commented[f]) == base
    changed = dict(src)
    changed[f0] = src[f0].replace("constexpr int TR = 128;", "constexpr int TR = 64;")
    assert changed[f0] != src[f0]
    assert bench.kernel_fingerprint("backward", read=lambda f: changed[f]) != base
    # whitespace between tokens can be meaningful: `a - -b` is not `a--b`
    assert bench.source_tokens("x = a - -b;") != bench.source_tokens("x = a--b;")
    assert bench.source_tokens("x  =\n\ta - -b;  // c") == bench.source_tokens("x = a - -b;")
    # the launch parameters chosen in api.cu are part of every kernel's fingerprint
    assert all("api.cu" in srcs for srcs in bench.KERNEL_SOURCES.values())
