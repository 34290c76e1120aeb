"""The multi-rank path of bench.py on the CPU: two gloo ranks on 127.0.0.1.

Under torchrun bench.py runs one process per GPU, each decoding its own
independent batch of the same shapes (weak scaling, no collective on the data
path); the only collectives are the barrier around the timed region and the
maximum of the step time over ranks, from which rank 0 reports the whole-job
throughput. These tests drive exactly those functions with gloo.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from sa_synth import config, make_workload
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        base = config(5, small=True)
        cfg = bench.rank_config(base, rank, world)
        wl = make_workload(cfg)
        # a fingerprint of this rank's inputs, gathered on every rank
        fp = torch.tensor([float(wl.q(0).astype(np.float64).sum()),
                           float(wl.k_pre.astype(np.float64).sum())], dtype=torch.float64)
        every = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(every, fp)
        dist.barrier()
        local_ms = 0.25 * (rank + 1)                 # rank-local mean step time
        worst = bench.dist_max(local_ms, world, "cpu")
        q.put(dict(rank=rank, worst=worst, value=bench.aggregate_steps_per_s(worst, world),
                   seed=cfg.seed, shapes=(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.ps, cfg.topk),
                   base_shapes=(base.B, base.H_q, base.H_kv, base.D, base.ps, base.topk),
                   q_shape=tuple(wl.q(0).shape), fps=[e.tolist() for e in every]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_batches_and_take_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort(key=lambda d: d["rank"])
    # the slowest rank's time on every rank, and the aggregate over both ranks
    assert [d["worst"] for d in got] == [0.5, 0.5]
    assert all(abs(d["value"] - 2 * 1000.0 / 0.5) < 1e-9 for d in got)
    # same shapes, different seeds and different data on the two ranks
    assert got[0]["shapes"] == got[1]["shapes"] == got[0]["base_shapes"]
    assert got[0]["q_shape"] == got[1]["q_shape"]
    assert got[0]["seed"] != got[1]["seed"]
    fps = got[0]["fps"]
    assert fps == got[1]["fps"] and fps[0] != fps[1]


def test_single_rank_keeps_the_base_workload():
    sys.path.insert(0, ROOT)
    import bench
    from sa_synth import config
    c = config(5, small=True)
    assert bench.rank_config(c, 0, 1) == c
    assert bench.dist_max(1.5, 1, "cpu") == 1.5
    assert bench.aggregate_steps_per_s(0.5, 1) == 2000.0


def test_reference_arm_is_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def _gather_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from sparse_paged_kv_page_gb300.shard import gather_slices, page_ranges
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the score rows of 3 requests x 2 KV heads over 12 pages, split by rank
        full = torch.arange(3 * 2 * 12, dtype=torch.float32).reshape(3, 2, 12)
        lo, hi = page_ranges(12, world)[rank]
        got = gather_slices(full[:, :, lo:hi].clone(), dim=2)
        q.put((rank, torch.equal(got, full)))
    finally:
        dist.destroy_process_group()


def test_sequence_shards_exchange_score_rows_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, True), (1, True)]


def test_page_ranges_cover_the_pages():
    sys.path.insert(0, ROOT)
    from sparse_paged_kv_page_gb300.shard import page_ranges
    for n, s in [(12, 2), (13, 5), (1, 1), (8194, 3)]:
        r = page_ranges(n, s)
        assert r[0][0] == 0 and r[-1][1] == n and all(a[1] == b[0] for a, b in zip(r, r[1:]))
        assert max(h - l for l, h in r) - min(h - l for l, h in r) <= 1
