"""Host-side multi-rank logic of bench.py, on CPU with the gloo backend.

bench.py runs one independent replica per GPU (the layer is sharded by
nothing: replicas only) and takes the slowest rank's time; these tests check
that reduction and the barrier with two gloo ranks, and that the reference
(oracle) arm prints from rank 0 only.
"""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    m = bench.max_over_ranks(1.5 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, m))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 3.0), (1, 3.0)]


def test_reference_arm_prints_from_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--cpu-seconds", "0.1"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--cpu-seconds", "0.1"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_binding_roofline_picks_the_longer_time():
    # full-shape layer: 2,534,400 B per unique expert, 2*3*H*I flops per assignment
    sys.path.insert(0, ROOT)
    import bench
    per_assign = 2.0 * 3 * 2560 * 640
    peaks = dict(hbm_gbs=6771.0, tc_tflops=1890.5)
    # decode, one token: 10 experts' bytes against 10 assignments' flops
    assert bench.binding_roofline(10 * 2534400, 10 * per_assign, **peaks) == "hbm"
    # 512 Zipf-routed tokens on about 125 experts: still the bytes
    assert bench.binding_roofline(125 * 2534400, 5120 * per_assign, **peaks) == "hbm"
    # 4096 tokens on about 146 experts: the flops
    assert bench.binding_roofline(146 * 2534400, 40960 * per_assign, **peaks) == "tensor"
