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


def _spawn(target, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


def _seq_shard_main(rank, world, port, q):
    """One rank of a sequence-sharded page-level step, computed with the oracle:
    score its own page range, exchange the score slices, select over the whole
    rows, attend its part of the selection, exchange the partial states and
    merge them by log-sum-exp."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle as O
    from sa_synth import config, make_workload
    from sparse_paged_kv_page_gb300.shard import gather_slices, gather_states, page_ranges
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = config(5, small=True).replace(prefill=(2990, 2990))     # 187 pages: an odd count
        wl = make_workload(cfg)
        c = wl.cfg
        L = 2990
        n = O.num_pages(L, c.ps)
        lo, hi = page_ranges(n, world)[rank]
        sc = O.default_scale(c.D)
        qb = wl.q(0)
        local = torch.zeros((c.B, c.H_kv, hi - lo), dtype=torch.float64)
        for b in range(c.B):
            for h in range(c.H_kv):
                kh = wl.k_seq(b, head=h)
                # this rank's pages only: rows [lo * ps, min(hi * ps, L))
                mn, mx, me = O.head_meta(kh[lo * c.ps:], min(hi * c.ps, L) - lo * c.ps, c.ps, c.dtype)
                qg = O.decode_kdt(qb[b, h * c.G:(h + 1) * c.G], c.dtype)
                local[b, h] = torch.from_numpy(O.score_pages(mn, mx, me, qg, c.w_avg, c.w_peak))
        rows = gather_slices(local, dim=2)                     # exchange 1: whole score rows
        o_part = torch.zeros((c.B, c.H_q, c.D), dtype=torch.float64)
        l_part = torch.full((c.B, c.H_q), -float("inf"), dtype=torch.float64)
        sels = {}
        for b in range(c.B):
            for h in range(c.H_kv):
                sel = O.select_pages(rows[b, h].numpy(), n, c.topk)
                sels[(b, h)] = sel
                mine = sel[(sel >= lo) & (sel < hi)]
                pos = O.selected_positions(mine, L, c.ps)
                qg = O.decode_kdt(qb[b, h * c.G:(h + 1) * c.G], c.dtype)
                o, lse, _ = O.attention(qg, O.decode_kdt(wl.k_seq(b, head=h)[pos], c.dtype),
                                        O.decode_kdt(wl.v_seq(b, head=h)[pos], c.dtype), sc)
                o_part[b, h * c.G:(h + 1) * c.G] = torch.from_numpy(o)
                l_part[b, h * c.G:(h + 1) * c.G] = torch.from_numpy(lse)
        o_all, l_all = gather_states(o_part, l_part)           # exchange 2: partial states
        q.put((rank, (lo, hi), rows.numpy(), o_all.numpy(), l_all.numpy(), sels))
    finally:
        dist.destroy_process_group()


def test_sequence_shards_exchange_scores_and_states_over_two_gloo_ranks():
    """Two ranks over an odd page count (ranges 94 / 93): the gathered score
    rows equal the unsharded oracle's bit for bit, both ranks hold the same
    rows and selection, and the partial states merged by the oracle's
    log-sum-exp merge equal single-shot attention over the whole selection."""
    import oracle as O
    from sa_synth import config, make_workload
    got = _spawn(_seq_shard_main)
    (r0, rng0, rows0, o0, l0, sel0), (r1, rng1, rows1, o1, l1, sel1) = got
    assert rng0 == (0, 94) and rng1 == (94, 187)
    assert np.array_equal(rows0, rows1) and np.array_equal(o0, o1) and np.array_equal(l0, l1)
    cfg = config(5, small=True).replace(prefill=(2990, 2990))
    wl = make_workload(cfg)
    c = wl.cfg
    sc = O.default_scale(c.D)
    qb = wl.q(0)
    for b in range(c.B):
        for h in range(c.H_kv):
            kh, vh = wl.k_seq(b, head=h), wl.v_seq(b, head=h)
            qg = qb[b, h * c.G:(h + 1) * c.G]
            r = O.page_decode_unit(kh, vh, 2990, qg, ps=c.ps, topk=c.topk, w_avg=c.w_avg,
                                   w_peak=c.w_peak, dtype=c.dtype)
            assert np.array_equal(rows0[b, h], r["scores"])
            assert np.array_equal(sel0[(b, h)], r["sel"]) and np.array_equal(sel1[(b, h)], r["sel"])
            g = slice(h * c.G, (h + 1) * c.G)
            o, lse = O.merge_partials(o0[:, b, g], l0[:, b, g])
            assert np.allclose(o, r["out"], atol=1e-12) and np.allclose(lse, r["lse"], atol=1e-12)


def _kv_head_main(rank, world, port, q):
    """One rank of a KV-head-partitioned step: its heads' statistics, scores,
    selection and attention, with no exchange inside the step; the outputs of
    every rank are gathered only to compare them here."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle as O
    from sa_synth import config, make_workload
    from sparse_paged_kv_page_gb300.shard import kv_head_range
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = config(3, small=True).replace(H_q=12, H_kv=3)     # 3 KV heads over 2 ranks: 2 + 1
        wl = make_workload(cfg)
        c = wl.cfg
        h0, h1 = kv_head_range(c.H_kv, world, rank)
        qb = wl.q(0)
        out = torch.zeros((c.B, c.H_q, c.D), dtype=torch.float64)
        for b in range(c.B):
            L = int(wl.prefill_lens[b])
            for h in range(h0, h1):
                r = O.page_decode_unit(wl.k_seq(b, head=h), wl.v_seq(b, head=h), L,
                                       qb[b, h * c.G:(h + 1) * c.G], ps=c.ps, topk=c.topk,
                                       w_avg=c.w_avg, w_peak=c.w_peak, dtype=c.dtype)
                out[b, h * c.G:(h + 1) * c.G] = torch.from_numpy(r["out"])
        every = [torch.zeros_like(out) for _ in range(world)]
        dist.all_gather(every, out)
        q.put((rank, (h0, h1), [e.numpy() for e in every]))
    finally:
        dist.destroy_process_group()


def test_kv_head_partition_over_two_gloo_ranks():
    """KV heads 0-1 on rank 0 and 2 on rank 1: together the ranks' head rows
    are the unpartitioned step's output, row for row."""
    import oracle as O
    from sa_synth import config, make_workload
    got = _spawn(_kv_head_main)
    (_, rng0, every), (_, rng1, _) = got
    assert rng0 == (0, 2) and rng1 == (2, 3)
    cfg = config(3, small=True).replace(H_q=12, H_kv=3)
    wl = make_workload(cfg)
    c = wl.cfg
    qb = wl.q(0)
    for b in range(c.B):
        L = int(wl.prefill_lens[b])
        for h in range(c.H_kv):
            r = O.page_decode_unit(wl.k_seq(b, head=h), wl.v_seq(b, head=h), L,
                                   qb[b, h * c.G:(h + 1) * c.G], ps=c.ps, topk=c.topk,
                                   w_avg=c.w_avg, w_peak=c.w_peak, dtype=c.dtype)
            owner = 0 if h < 2 else 1
            assert np.array_equal(every[owner][b, h * c.G:(h + 1) * c.G], r["out"])
            assert not np.any(every[1 - owner][b, h * c.G:(h + 1) * c.G])


def test_page_ranges_cover_the_pages():
    sys.path.insert(0, ROOT)
    from sparse_paged_kv_page_gb300.shard import page_ranges
    for n, s in [(12, 2), (13, 5), (1, 1), (8194, 3)]:
        r = page_ranges(n, s)
        assert r[0][0] == 0 and r[-1][1] == n and all(a[1] == b[0] for a, b in zip(r, r[1:]))
        assert max(h - l for l, h in r) - min(h - l for l, h in r) <= 1
    assert page_ranges(8194, 3) == [(0, 2732), (2732, 5463), (5463, 8194)]


def _unequal_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from sparse_paged_kv_page_gb300.shard import gather_slices, page_ranges
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        full = torch.arange(2 * 3 * 8194, dtype=torch.float32).reshape(2, 3, 8194)
        lo, hi = page_ranges(8194, world)[rank]
        q.put((rank, torch.equal(gather_slices(full[:, :, lo:hi].clone(), dim=2), full)))
    finally:
        dist.destroy_process_group()


def test_gather_slices_takes_unequal_ranges_over_three_gloo_ranks():
    assert _spawn(_unequal_main, world=3) == [(0, True), (1, True), (2, True)]
