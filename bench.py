"""Benchmark of one decode step of page-selected sparse attention on GB300.

A step is the whole hot path over one batch: append k_new / v_new with the
page-statistics refresh, score every page, select top-k with the tail forced,
exact split-K attention over the selected pages with the LSE merge (page
level); for the token-level workload: append, attention over the retained
tokens, H2O fold and eviction. The default workload is the long-context GQA
decode (B=4, H_q=64, H_kv=8, D=128, page 16, 131072-token contexts, top-256
pages), whose per-step byte stream is the one the HBM roofline speaks to.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 5] [--impl ours|reference]

Timing: the step is one captured CUDA graph; each timed step (the graph
replay) is bracketed by CUDA events on the launching stream. Before the events
the step's inputs are copied from the HBM-resident input set into the step's
input buffers and L2 (129 MB) is flushed (a 256 MB write, then a 256 MB read).
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode steps/s and achieved HBM GB/s vs GB300 peak (score+select+attend)"
FALLBACK_HBM = 6800.0
NOMINAL_HBM = 8000.0      # GB300 HBM3e, nominal


# ---------------------------------------------------------------------------
# multi-rank host logic (one process per GPU; no data-path collective)
# ---------------------------------------------------------------------------
def rank_config(cfg, rank, world):
    """Each rank decodes its own independent batch of the same shapes (weak scaling)."""
    return cfg.replace(seed=cfg.rng_seed + 7919 * rank) if world > 1 else cfg


def dist_max(x: float, world: int, device) -> float:
    """Maximum of a rank-local float over all ranks (the slowest rank's time)."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_steps_per_s(max_ms: float, world: int) -> float:
    """Whole-job throughput: every rank runs one step of its own batch per step time."""
    return world * 1000.0 / max_ms


# ---------------------------------------------------------------------------
# byte model
# ---------------------------------------------------------------------------
def step_bytes(cfg, lens, per_query_head=False):
    """Algorithmic bytes of one page-level step: the 3 statistics rows of every
    page, the K and V of the selected pages (per KV head, or per query head
    with per-query-head selection), q and out (2-byte elements)."""
    e = 2
    tot = 0
    rows = cfg.H_q if per_query_head else cfg.H_kv
    for L in lens:
        n = -(-L // cfg.ps)
        tot += n * cfg.H_kv * 3 * cfg.D * e
        tot += min(cfg.topk, n) * rows * 2 * cfg.ps * cfg.D * e
    return tot + 2 * cfg.B * cfg.H_q * cfg.D * e


def entmax_step_bytes(cfg, lens, v_rows):
    """Page level with alpha-entmax: the statistics rows, K of the selected
    pages, V of the v_rows tokens some query head keeps (entmax is sparse: the
    rest is never read), q and out. The logits between the passes stay in L2."""
    e = 2
    tot = 0
    for L in lens:
        n = -(-L // cfg.ps)
        tot += n * cfg.H_kv * 3 * cfg.D * e
        tot += min(cfg.topk, n) * cfg.H_kv * cfg.ps * cfg.D * e
    return tot + v_rows * cfg.D * e + 2 * cfg.B * cfg.H_q * cfg.D * e


def gauss_step_bytes(cfg, lens, sel_pages, v_rows):
    """Gaussian-aware step: the k_mean and k_std rows of every page, K of the
    pages each query head selected, V of the rows each head keeps, q and out."""
    e = 2
    stats = sum(-(-L // cfg.ps) for L in lens) * cfg.H_kv * 2 * cfg.D * e
    return stats + sel_pages * cfg.ps * cfg.D * e + v_rows * cfg.D * e + 2 * cfg.B * cfg.H_q * cfg.D * e


def entmax_kept(dec, alpha):
    """V rows the last step read, and the mean support per query head, from
    the step's own logits and thresholds."""
    import numpy as np
    z = dec.logits.cpu().numpy().astype(np.float64)
    tau = dec.tau.cpu().numpy().astype(np.float64)
    cnt = dec.sel_cnt.cpu().numpy()
    B, Hq, R = z.shape
    G = Hq // cnt.shape[1]                    # 1 with a selection per query head
    with np.errstate(invalid="ignore"):
        keep = np.isfinite(z) & ((alpha - 1.0) * z - tau[:, :, None] > 0)
    rows, sup = 0, []
    for b in range(B):
        for h in range(cnt.shape[1]):
            n = int(cnt[b, h]) * dec.ps
            k = keep[b, h * G:(h + 1) * G, :n]
            rows += int(k.any(0).sum())
            sup.extend(k.sum(-1).tolist())
    return rows, float(np.mean(sup))


def h2o_step_bytes(cfg, cnts):
    """Token level: K and V of every retained token, its bf16 score read and
    written, q and out."""
    e = 2
    return sum(n * (2 * cfg.D * e + 2 * 2) for n in cnts) + 2 * cfg.B * cfg.H_q * cfg.D * e


def score_bytes(cfg, lens):
    """Algorithmic bytes of the page scorer: 3 * D * 2 per (page, KV head)."""
    return sum(-(-L // cfg.ps) for L in lens) * cfg.H_kv * 3 * cfg.D * 2


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


def traffic_from_profile(kernel_file, name):
    """Per-launch DRAM bytes from a committed ncu summary, used only if it was
    taken on the kernel source as it is now (sha256 of the .cu file)."""
    path = os.path.join(ROOT, "profiles", name)
    src = os.path.join(ROOT, "sparse_paged_kv_page_gb300", "csrc", kernel_file)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        vals = {}
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                v = v.strip()
                if v.startswith("`"):                      # `value` (comment)
                    v = v[1:].split("`", 1)[0]
                vals[k.strip().strip("-* `")] = v.split()[0] if v else v
        if vals.get("source_sha256") != sha:
            return None
        return float(vals["dram_bytes_per_launch_full_size"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.p, self.lines = index, None, []

    def __enter__(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.4)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            try:
                out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# CPU oracle leg: spawned workers map the prefill arrays from shared memory
# and each runs one (request, KV head) unit of a step per task.
# ---------------------------------------------------------------------------
_W = {}


def _worker_init(spec):
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    import numpy as np
    for name, path in spec.items():
        _W[name] = np.load(path, mmap_mode="r")


def _worker_task(task):
    import numpy as np
    import oracle as O
    b, h, lo, hi, extra_k, extra_v, L, qg, kind, kw, hh, pos = task
    ks = np.ascontiguousarray(_W["k"][lo:hi, h])
    vs = np.ascontiguousarray(_W["v"][lo:hi, h])
    if extra_k is not None:
        ks = np.concatenate([ks, extra_k], 0)
        vs = np.concatenate([vs, extra_v], 0)
    t = time.perf_counter()
    if kind == "page":
        O.page_decode_unit(ks, vs, L, qg, **kw)
    elif kind == "gauss":
        for g in range(qg.shape[0]):                        # each query head selects for itself
            O.gauss_decode_unit(ks, vs, L, qg[g], **kw)
    else:
        O.h2o_unit_step(hh, pos, ks, vs, qg, **kw)
    return time.perf_counter() - t


class OracleRunner:
    """The float64 oracle on the host cores, one unit per spawned worker."""

    def __init__(self, wl, workers, alpha=1.0, gaussian=False):
        import multiprocessing as mp
        import tempfile
        import numpy as np
        self.wl, self.workers, self.alpha, self.gaussian = wl, workers, alpha, gaussian
        self.dir = tempfile.mkdtemp(prefix="sa_oracle_")
        spec = {}
        for name, arr in (("k", wl.k_pre), ("v", wl.v_pre)):
            path = os.path.join(self.dir, name + ".npy")
            np.save(path, arr)
            spec[name] = path
        self.pool = mp.get_context("spawn").Pool(workers, initializer=_worker_init,
                                                 initargs=(spec,))

    def tasks(self, step, units):
        import numpy as np
        wl, c = self.wl, self.wl.cfg
        steps_done = step + 1 if c.decode_steps > 0 else 0
        qb = wl.q(step)
        out = []
        for b, h in units:
            L = wl.seq_len(b, steps_done)
            lo, hi = int(wl.pre_cu[b]), int(wl.pre_cu[b + 1])
            ek = ev = None
            if steps_done:
                ek = np.stack([wl.kv_new(t)[0][b, h] for t in range(steps_done)])
                ev = np.stack([wl.kv_new(t)[1][b, h] for t in range(steps_done)])
            qg = qb[b, h * c.G:(h + 1) * c.G]
            if c.ps == 1:
                n = min(L, c.budget + 1)
                kw = dict(dtype=c.dtype, decay=c.decay, budget=c.budget, n_sink=c.n_sink,
                          grace=c.grace, scale=c.scale)
                out.append((b, h, lo, hi, ek, ev, L, qg, "h2o", kw, np.zeros(n), np.arange(L - n, L)))
            elif self.gaussian:
                kw = dict(ps=c.ps, alpha=self.alpha, dtype=c.dtype, scale=c.scale)
                out.append((b, h, lo, hi, ek, ev, L, qg, "gauss", kw, None, None))
            else:
                kw = dict(ps=c.ps, topk=c.topk, w_avg=c.w_avg, w_peak=c.w_peak, dtype=c.dtype,
                          scale=c.scale, alpha=self.alpha)
                out.append((b, h, lo, hi, ek, ev, L, qg, "page", kw, None, None))
        return out

    def run(self, tasks):
        t0 = time.perf_counter()
        self.pool.map(_worker_task, tasks, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        import shutil
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)


def units_of(cfg):
    return [(b, h) for b in range(cfg.B) for h in range(cfg.H_kv)]


def cpu_baseline(wl, full_steps, workers, alpha=1.0, gaussian=False):
    """Full steps of the oracle (every unit), on `workers` processes."""
    r = OracleRunner(wl, workers, alpha, gaussian)
    try:
        r.run(r.tasks(0, units_of(wl.cfg)[:workers]))          # warm the workers
        walls = [r.run(r.tasks(s, units_of(wl.cfg))) for s in range(full_steps)]
    finally:
        r.close()
    return walls


def cpu_one_thread(wl, n_units, alpha=1.0, gaussian=False):
    """The oracle on one host thread: n_units (request, KV head) units of a
    step, returned as full steps per second (units / units per step / wall)."""
    r = OracleRunner(wl, 1, alpha, gaussian)
    try:
        units = units_of(wl.cfg)
        r.run(r.tasks(0, units[:1]))                            # warm the worker
        sample = [units[i % len(units)] for i in range(n_units)]
        wall = r.run(r.tasks(0, sample))
    finally:
        r.close()
    return (n_units / len(units)) / wall, wall


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def run_gpu(args, rank, world):
    import numpy as np
    import torch

    from sa_synth import config, make_workload, fill_stale
    from sparse_paged_kv_page_gb300.step import SparseDecoder
    import sparse_paged_kv_page_gb300 as S

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    cfg = rank_config(config(args.config), rank, world)
    append = cfg.decode_steps > 0
    # input schedule: 1 eager step, W warm-up replays, K timed, kernel reps, e2e steps
    n_in = 1 + args.warmup + args.steps + args.kernel_reps + args.e2e_steps + max(args.e2e_steps, 16)
    wl = make_workload(cfg, extra_steps=max(0, n_in + 2 - cfg.decode_steps))
    c = wl.cfg
    tdt = torch.bfloat16 if c.dtype == "bf16" else torch.float16

    def dbits(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(tdt)

    token = c.ps == 1
    kw = dict(batch=c.B, num_q_heads=c.H_q, num_kv_heads=c.H_kv, head_dim=c.D, page_size=c.ps,
              num_blocks=wl.num_blocks, bt_stride=wl.max_pages, dtype=tdt, scale=c.scale,
              device=dev)
    if token:
        kw.update(budget=c.budget, n_sink=c.n_sink, grace=c.grace, decay=c.decay,
                  ret_cap=int(wl.prefill_lens.max()) + n_in + 4)
    else:
        kw.update(topk=c.topk, w_avg=c.w_avg, w_peak=c.w_peak,
                  per_query_head=args.per_query_head,
                  alpha=(args.entmax or 1.5) if args.gaussian else (args.entmax or 1.0),
                  gaussian=args.gaussian)
    dec = SparseDecoder(**kw)
    fill_stale(dec.cache.k, "normal3", 11)
    fill_stale(dec.cache.v, "normal3", 12)
    if dec.cache.meta is not None:
        fill_stale(dec.cache.meta, "normal3", 13)
    dec.set_block_table(torch.from_numpy(wl.block_table))
    kp, vp = dbits(wl.k_pre), dbits(wl.v_pre)
    dec.prefill(kp, vp, wl.prefill_lens.tolist())
    del kp, vp
    torch.cuda.synchronize()

    # per-step inputs, resident in HBM before timing: row t = [q | k_new | v_new]
    nq, nk = c.B * c.H_q * c.D, c.B * c.H_kv * c.D
    host_in = np.zeros((n_in, nq + 2 * nk), dtype=np.uint16)
    for t in range(n_in):
        host_in[t, :nq] = wl.q(t).reshape(-1)
        if append:
            kn, vn = wl.kv_new(t)
            host_in[t, nq:nq + nk] = kn.reshape(-1)
            host_in[t, nq + nk:] = vn.reshape(-1)
    dev_in = dbits(host_in)
    inbuf = torch.empty(nq + 2 * nk, dtype=tdt, device=dev)
    dec.q_buf = inbuf[:nq].view(c.B, c.H_q, c.D)
    dec.k_buf = inbuf[nq:nq + nk].view(c.B, c.H_kv, c.D)
    dec.v_buf = inbuf[nq + nk:].view(c.B, c.H_kv, c.D)
    stream = torch.cuda.current_stream(dev)
    # L2 flush between steps: write a 256 MB buffer (twice L2), then read
    # another one, so the step starts with a cold L2 whose lines are clean --
    # otherwise the flush's ~129 MB of dirty lines would be written back to HBM
    # during the timed step.
    flush_w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    class _Flush:
        @staticmethod
        def zero_():
            flush_w.zero_()
            torch.amax(flush_r, dim=0, out=flush_sink)
    flush = _Flush

    t_next = 0
    # eager step 0 (loads modules, sets kernel attributes), then capture
    inbuf.copy_(dev_in[t_next]); t_next += 1
    dec.step(dec.q_buf, dec.k_buf if append else None, dec.v_buf if append else None)
    torch.cuda.synchronize()
    graph = dec.capture(append=append)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        inbuf.copy_(dev_in[t_next]); t_next += 1
        graph.replay()
    torch.cuda.synchronize()
    lens_start = [int(x) for x in dec.seq_lens.cpu().tolist()]
    cnt_start = dec.ret_cnt.cpu().numpy().reshape(-1).tolist() if token else None

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ahead = 100
    sleep_cycles = int(ahead * 150e-6 * 2.0e9)       # ~150 us of device time a step, ~2 GHz
    with ClockSampler(dev.index) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            # every `ahead` steps the device idles (outside the events) long
            # enough for the host to enqueue the next `ahead` steps, so a host
            # pause (scheduling, garbage collection) never lands between a
            # step's events
            if i % ahead == 0:
                torch.cuda._sleep(sleep_cycles)
            # this step's inputs into the step's input buffers, then the L2
            # flush, both before the events: the inputs are resident in HBM
            # when the timed step starts
            inbuf.copy_(dev_in[t_next]); t_next += 1
            flush.zero_()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(step_ms)
    ent = None
    if token:
        # retained tokens attended per (request, KV head): budget + 1 after the first step
        bytes_per_step = h2o_step_bytes(c, [min(n + 1, c.budget + 1) for n in cnt_start])
    elif args.gaussian:
        v_rows, support = entmax_kept(dec, dec.alpha)
        pages = int(dec.sel_cnt.sum().item())
        bytes_per_step = gauss_step_bytes(c, [L + args.steps for L in lens_start], pages, v_rows)
        ent = {"alpha": dec.alpha, "selection": "gaussian-aware, per query head",
               "pages_selected_last_step": pages,
               "mean_pages_per_query_head": pages / (c.B * c.H_q),
               "v_rows_read_last_step": v_rows, "mean_support_per_query_head": support}
    elif args.entmax:
        v_rows, support = entmax_kept(dec, args.entmax)
        bytes_per_step = entmax_step_bytes(c, [L + args.steps for L in lens_start], v_rows)
        ent = {"alpha": args.entmax, "v_rows_read_last_step": v_rows,
               "mean_support_per_query_head": support,
               "selected_tokens_per_kv_head": c.topk * c.ps}
    else:
        bytes_per_step = statistics.mean(
            step_bytes(c, [L + (i + 1 if append else 0) for L in lens_start], args.per_query_head)
            for i in range(args.steps))
    status = int(dec.dev_status.item())

    # per-kernel breakdown: the same C-ABI calls launched one by one and each
    # bracketed by events. A short device-side spin after the L2 flush keeps
    # the GPU busy while the host enqueues the calls, so the events time the
    # kernels back to back rather than the host.
    kern = {}
    names = (["append"] if append else []) + (["decode", "h2o"] if token else
                                               (["select", "decode"] if args.gaussian else ["score", "select", "decode"]))
    acc = {n: [] for n in names}
    lens_reps = [int(x) for x in dec.seq_lens.cpu().tolist()]
    for i in range(args.kernel_reps):
        inbuf.copy_(dev_in[t_next]); t_next += 1
        flush.zero_()
        torch.cuda._sleep(300000)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        j = 0
        e[j].record(stream)
        if append:
            dec.append(dec.k_buf, dec.v_buf)
            j += 1; e[j].record(stream)
        if token:
            S.sa_sparse_decode(dec.cache.struct, dec.batch, dec.q_buf, c.H_q, dec.ret_pos,
                               dec.ret_cnt, dec.ret_cap, c.scale, dec.out, lse=dec.lse,
                               logits=dec.logits, logits_stride=dec.ret_cap,
                               workspace=dec.workspace, dev_status=dec.dev_status)
            j += 1; e[j].record(stream)
            S.sa_h2o_update(dec.batch, c.H_kv, c.H_q, dec.logits, dec.ret_cap, dec.lse,
                            dec.cache.hh, dec.cache.hh.shape[0], dec.ret_pos, dec.ret_cnt,
                            dec.ret_cap, c.budget, c.n_sink, c.grace, c.decay,
                            evicted=dec.evicted, evicted_cnt=dec.evicted_cnt,
                            dev_status=dec.dev_status)
            j += 1; e[j].record(stream)
        elif args.gaussian:
            S.sa_gauss_select(dec.cache.struct, dec.batch, dec.q_buf, c.H_q, dec.alpha, c.scale,
                              dec.moments, dec.max_pages, dec.sel_idx, dec.sel_cnt, dec.sel_stride,
                              tau_hat=dec.tau_hat, dev_status=dec.dev_status)
            j += 1; e[j].record(stream)
            S.sa_sparse_decode_entmax_qh(dec.cache.struct, dec.batch, dec.q_buf, c.H_q, dec.sel_idx,
                                         dec.sel_cnt, dec.sel_stride, dec.alpha, c.scale, dec.out,
                                         tau=dec.tau, logits=dec.logits,
                                         logits_stride=dec.sel_stride * c.ps, workspace=dec.ent_ws,
                                         dev_status=dec.dev_status)
            j += 1; e[j].record(stream)
        else:
            qh = args.per_query_head
            (S.sa_score_pages_qh if qh else S.sa_score_pages)(
                dec.cache.struct, dec.batch, dec.q_buf, c.H_q, c.w_avg, c.w_peak,
                dec.scores, dec.max_pages, dev_status=dec.dev_status)
            j += 1; e[j].record(stream)
            S.sa_select_topk(dec.scores, dec.max_pages, dec.batch, c.ps, c.H_q if qh else c.H_kv,
                             c.topk, dec.sel_idx, dec.sel_cnt, dev_status=dec.dev_status)
            j += 1; e[j].record(stream)
            if args.entmax:
                S.sa_sparse_decode_entmax(
                    dec.cache.struct, dec.batch, dec.q_buf, c.H_q, dec.sel_idx, dec.sel_cnt,
                    c.topk, args.entmax, c.scale, dec.out, tau=dec.tau, logits=dec.logits,
                    logits_stride=c.topk * c.ps, workspace=dec.ent_ws, dev_status=dec.dev_status)
            else:
                (S.sa_sparse_decode_qh if qh else S.sa_sparse_decode)(
                    dec.cache.struct, dec.batch, dec.q_buf, c.H_q, dec.sel_idx,
                    dec.sel_cnt, c.topk, c.scale, dec.out, lse=dec.lse,
                    workspace=dec.workspace, dev_status=dec.dev_status)
            j += 1; e[j].record(stream)
        torch.cuda.synchronize()
        for k, n in enumerate(names):
            acc[n].append(e[k].elapsed_time(e[k + 1]))
    if args.kernel_reps:
        kern = {n: statistics.mean(v) for n, v in acc.items()}
    # mean statistics bytes the scorer read per rep (lengths grow by one per rep)
    score_ab = (statistics.mean(score_bytes(c, [L + (i + 1 if append else 0) for L in lens_reps])
                                for i in range(args.kernel_reps))
                if args.kernel_reps and not token else 0)

    # end to end through the public API: pinned host inputs in, the output back
    e2e = None
    if args.e2e_steps > 0:
        pin_in = torch.from_numpy(host_in.view(np.int16)).pin_memory()
        pin_out = torch.empty((c.B, c.H_q, c.D), dtype=torch.int16).pin_memory()
        marks = []
        for i in range(args.e2e_steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            inbuf.view(torch.int16).copy_(pin_in[t_next], non_blocking=True); t_next += 1
            graph.replay()
            pin_out.copy_(dec.out.view(torch.int16), non_blocking=True)
            b.record(stream)
            marks.append((a, b))
        torch.cuda.synchronize()
        serial_ms = dist_max(statistics.mean(x.elapsed_time(y) for x, y in marks), world, dev)

        # Pipelined, as a serving loop runs: groups of G steps are captured,
        # with their copies, into one CUDA graph (two graphs alternating). In
        # a group, step j's inputs are copied in from pinned host slot j on a
        # copy branch (the copy for step j + 1 overlaps step j), the step runs
        # on its own input buffer into its own output buffer, and its output
        # is copied back to pinned slot j on the copy branch while step j + 1
        # runs. The host refills a graph's pinned input slots with the inputs
        # of the steps it runs next only after that graph's previous launch
        # has finished. Steps run back to back without the L2 flush: a step
        # streams about twice L2 (the flush changes the device time by ~2%).
        G = 8
        N = (args.e2e_steps // G) * G
        if N < 2 * G:
            N = 2 * G
        copy = torch.cuda.Stream(device=dev)
        saved_out = dec.out
        groups = []
        for gi in range(2):
            ins = [torch.empty_like(inbuf) for _ in range(G)]
            outs = [torch.empty_like(dec.out) for _ in range(G)]
            pins = torch.empty((G, nq + 2 * nk), dtype=torch.int16).pin_memory()
            pouts = torch.empty((G, c.B, c.H_q, c.D), dtype=torch.int16).pin_memory()
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(device=dev)
            cap.wait_stream(stream)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cap):
                h_ev = [torch.cuda.Event() for _ in range(G)]
                r_ev = [torch.cuda.Event() for _ in range(G)]
                copy.wait_stream(cap)
                with torch.cuda.stream(copy):
                    for j in range(G):
                        ins[j].view(torch.int16).copy_(pins[j], non_blocking=True)
                        h_ev[j].record(copy)
                for j in range(G):
                    cap.wait_event(h_ev[j])
                    dec.out = outs[j]
                    dec.step(ins[j][:nq].view(c.B, c.H_q, c.D),
                             ins[j][nq:nq + nk].view(c.B, c.H_kv, c.D) if append else None,
                             ins[j][nq + nk:].view(c.B, c.H_kv, c.D) if append else None)
                    r_ev[j].record(cap)
                    copy.wait_event(r_ev[j])
                    with torch.cuda.stream(copy):
                        pouts[j].copy_(outs[j].view(torch.int16), non_blocking=True)
                cap.wait_stream(copy)
            groups.append((g, pins, pouts, ins, outs))
        dec.out = saved_out
        torch.cuda.synchronize()
        done = [None, None]

        def fill(gi, k):                                   # group k's inputs into graph gi's slots
            groups[gi][1].copy_(pin_in[t_next + k * G:t_next + (k + 1) * G])

        fill(0, 0)
        fill(1, 1)
        ev = lambda: torch.cuda.Event(enable_timing=True)
        t0, t1 = ev(), ev()
        t0.record(stream)
        for k in range(N // G):
            gi = k % 2
            if k >= 2:
                done[gi].synchronize()                     # its previous launch has read its slots
                fill(gi, k)
            groups[gi][0].replay()
            done[gi] = torch.cuda.Event()
            done[gi].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        t_next += N
        em = dist_max(t0.elapsed_time(t1) / N, world, dev)
        e2e = {"value": aggregate_steps_per_s(em, world), "unit": "steps/s",
               "h2d_bytes_per_step": int((nq + 2 * nk if append else nq) * 2),
               "d2h_bytes_per_step": int(c.B * c.H_q * c.D * 2), "ms_per_step": em,
               "mode": "pipelined: groups of 8 steps captured with their copies into CUDA graphs "
                       "(two alternating); every step copies its own inputs in from pinned host "
                       "memory and its output back on a copy branch that overlaps the neighbouring "
                       "steps; the host refills a graph's pinned input slots after its previous "
                       "launch; steps back to back without the L2 flush",
               "serial": {"value": aggregate_steps_per_s(serial_ms, world), "ms_per_step": serial_ms,
                          "mode": "one step at a time: L2 flush, H2D, step, D2H inside the events"}}
    status |= int(dec.dev_status.item())

    max_ms = dist_max(ms, world, dev)
    max_median_ms = dist_max(statistics.median(step_ms), world, dev)
    launches = (1 if append else 0) + (2 if token else (5 if args.gaussian else 3)) + \
        (3 if args.entmax and not args.gaussian else 0)
    return dict(ent=ent, ms=ms, max_ms=max_ms, wall=wall, clocks=clk.summary(), bytes=bytes_per_step,
                kern=kern, status=status, score_ab=score_ab, e2e=e2e, cfg=c, wl=wl,
                launches_per_step=launches, step_ms_min=min(step_ms), step_ms_max=max(step_ms),
                step_ms_median=statistics.median(step_ms), max_median_ms=max_median_ms)


def run_h2o_prefill(args):
    """The prefill-side H2O (each key as its own query) of the token-level
    workload's whole prefill: sa_h2o_prefill timed alone, the pool already
    holding the prefill's keys, the retained lists emptied before each rep."""
    import numpy as np
    import torch
    from sa_synth import config, make_workload
    from sparse_paged_kv_page_gb300.step import SparseDecoder
    import sparse_paged_kv_page_gb300 as S
    dev = torch.device("cuda", 0)
    c = config(4).replace(decode_steps=0)
    wl = make_workload(c)
    dec = SparseDecoder(batch=c.B, num_q_heads=c.H_q, num_kv_heads=c.H_kv, head_dim=c.D, page_size=1,
                        num_blocks=wl.num_blocks, bt_stride=wl.max_pages, budget=c.budget,
                        n_sink=c.n_sink, grace=c.grace, decay=c.decay, scale=c.scale,
                        ret_cap=int(wl.prefill_lens.max()) + 4, device=dev)
    dec.set_block_table(torch.from_numpy(wl.block_table))
    kv = torch.from_numpy(np.ascontiguousarray(wl.k_pre).view(np.int16)).to(dev).view(torch.bfloat16)
    vv = torch.from_numpy(np.ascontiguousarray(wl.v_pre).view(np.int16)).to(dev).view(torch.bfloat16)
    cu = torch.from_numpy(wl.pre_cu.astype(np.int32)).to(dev)
    S.sa_append_kv(dec.cache.struct, dec.batch, kv, vv, cu, int(wl.prefill_lens.max()), hh=dec.cache.hh,
                   dev_status=dec.dev_status)
    torch.cuda.synchronize()
    times = []
    for i in range(args.warmup + max(1, args.steps)):
        dec.ret_cnt.zero_()
        dec.cache.hh.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        S.sa_h2o_prefill(dec.cache.struct, dec.batch, cu, dec.cache.hh, dec.cache.hh.shape[0],
                         dec.ret_pos, dec.ret_cnt, dec.ret_cap, c.budget, c.n_sink, c.grace, c.decay,
                         c.scale, dev_status=dec.dev_status)
        b.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(a.elapsed_time(b))
    ms = statistics.mean(times)
    toks = int(wl.prefill_lens.sum())
    assert int(dec.dev_status.item()) == 0
    assert bool((dec.ret_cnt == c.budget).all())
    print(json.dumps({"metric": "prefill-side H2O absorb + eviction (key as query), tokens/s",
                      "value": toks / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
                      "steps": len(times), "warmup": args.warmup, "ms_per_step": ms,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                      "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": describe(c) + f", {toks} prefill tokens per call",
                                 "timing": "CUDA events around each sa_h2o_prefill call"},
                      "gpu_launches": len(times)}))


def run_also(args, rank, world, hbm_peak, peak_kind):
    """The batched GQA workload (the second one the 60% bar names) timed the
    same way as the headline line: the fused step replayed as a CUDA graph,
    L2 flushed between steps, CUDA events on the launching stream, and the
    scorer alone for its roofline."""
    import copy
    import torch
    a = copy.copy(args)
    a.config = 3
    a.steps = max(20, min(args.steps, 200))
    a.warmup = max(3, args.warmup)
    a.e2e_steps = 0
    a.kernel_reps = max(10, min(args.kernel_reps, 30))
    torch.cuda.empty_cache()
    res = run_gpu(a, rank, world)
    c = res["cfg"]
    step_gbs = res["bytes"] / (res["ms"] * 1e-3) / 1e9
    ach = res["score_ab"] / (res["kern"]["score"] * 1e-3) / 1e9 if res["kern"] else None
    out = {"workload": describe(c), "value": aggregate_steps_per_s(res["max_ms"], world),
           "unit": "steps/s", "steps": a.steps, "warmup": a.warmup, "ms_per_step": res["max_ms"],
           "step_ms_median": res["step_ms_median"],
           "hbm_gbs": step_gbs, "hbm_frac": step_gbs / hbm_peak, "hbm_peak_kind": peak_kind,
           "hbm_frac_nominal": step_gbs / NOMINAL_HBM,
           "algorithmic_bytes_per_step": res["bytes"],
           "roofline": None if ach is None else {
               "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
               "frac": ach / hbm_peak, "traffic": None, "kernel": "score_kernel (sa_score_pages)",
               "peak_kind": peak_kind, "algorithmic_bytes_per_launch": res["score_ab"],
               "kernel_ms": res["kern"]},
           "clocks": res["clocks"], "dev_status": res["status"],
           "gpu_launches": res["launches_per_step"] * a.steps}
    del res
    torch.cuda.empty_cache()
    return out


def describe(c):
    base = f"{c.name}: B={c.B}, H_q={c.H_q}, H_kv={c.H_kv}, D={c.D}, page_size={c.ps}, {c.dtype}"
    if c.ps == 1:
        return base + (f", prefill {c.prefill[0]}, budget {c.budget} (sink {c.n_sink}, "
                       f"grace {c.grace}), decay {c.decay}")
    ctx = f"context {c.prefill[0]}" if c.prefill else f"context U{list(c.len_range)}"
    return base + f", {ctx}, top-{c.topk} pages incl. tail, w=({c.w_avg}, {c.w_peak})"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--kernel-reps", type=int, default=100)
    ap.add_argument("--cpu-steps", type=int, default=2)
    ap.add_argument("--workers", type=int, default=0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-also", action="store_true",
                    help="skip the batched GQA workload reported beside the long-context line")
    ap.add_argument("--h2o-prefill", action="store_true",
                    help="time the prefill-side H2O absorb / eviction of the token-level workload")
    ap.add_argument("--entmax", type=float, default=0.0,
                    help="attend the selection with alpha-entmax (1 < alpha <= 2) instead of softmax")
    ap.add_argument("--gaussian", action="store_true",
                    help="Gaussian-aware adaptive selection per query head, attended with "
                         "alpha-entmax (alpha = --entmax, default 1.5)")
    ap.add_argument("--per-query-head", action="store_true",
                    help="select pages per query head (score, select, attend one row per query head)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    from sa_synth import config, make_workload
    cfg = config(args.config)
    workers = args.workers or max(1, min(16, os.cpu_count() or 1))

    if args.impl == "reference":
        # the float64 oracle on the host cores; each step is a bounded sample:
        # one (request, KV head) unit, units cycled, steps spread over workers
        if rank != 0:
            return
        wl = make_workload(cfg, extra_steps=2)
        r = OracleRunner(wl, workers, (args.entmax or 1.5) if args.gaussian else (args.entmax or 1.0),
                         args.gaussian)
        alpha = (args.entmax or 1.5) if args.gaussian else (args.entmax or 1.0)
        units = units_of(cfg)
        try:
            r.run(r.tasks(0, units[:workers]))
            warm = [units[i % len(units)] for i in range(args.warmup)]
            if warm:
                r.run(r.tasks(0, warm))
            timed = [units[i % len(units)] for i in range(args.steps)]
            wall = r.run(r.tasks(0, timed))
        finally:
            r.close()
        # the timed work is args.steps unit samples = args.steps / units full steps
        full = args.steps / len(units)
        v = full / wall                                  # full steps per second
        v1, wall1 = cpu_one_thread(wl, min(4, len(units)), alpha, args.gaussian)
        sample = (f"{args.steps} (request, KV head) unit samples of the {len(units)} in a full "
                  f"step = {full:g} full steps, cycling over the units, on {workers} spawned "
                  f"single-threaded workers")
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s",
                "n_gpus": args.gpus, "steps": full, "warmup": args.warmup,
                "ms_per_step": 1000.0 * wall / full, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": describe(cfg),
                           "sample": sample + "; steps counts the full steps timed, so "
                                     "steps x ms_per_step is the timed wall"},
                "timed_wall_s": wall, "unit_samples": args.steps,
                "cpu_baseline": {"value": v, "unit": "steps/s", "cores": workers, "kind": "oracle",
                                 "sample": sample,
                                 "one_thread": {"value": v1, "unit": "steps/s", "cores": 1,
                                                "sample": f"{min(4, len(units))} unit samples on one "
                                                          f"worker ({wall1:.2f} s)"}},
                "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if args.h2o_prefill:
        if rank == 0:
            run_h2o_prefill(args)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, rank, world)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    c = res["cfg"]
    hbm_peak, peak_kind = peaks()
    value = aggregate_steps_per_s(res["max_ms"], world)
    step_gbs = res["bytes"] / (res["ms"] * 1e-3) / 1e9
    roof = None
    if res["kern"]:
        if args.gaussian:
            ab = res["score_ab"] * 2 // 3                   # k_mean and k_std rows, not k_min / k_max
            kms = res["kern"]["select"]
            tm = traffic_from_profile("gauss.cu", "gauss_moments.long_context_gqa.md") if args.config == 5 else None
            ts = traffic_from_profile("gauss.cu", "gauss_select.long_context_gqa.md") if args.config == 5 else None
            tr = tm + ts if tm is not None and ts is not None else None
            mk = "gauss_moments_mma_kernel" if c.dtype == "bf16" else "gauss_moments_kernel"
            kname = mk + " + gauss_select_kernel (sa_gauss_select)"
        elif c.ps > 1 and args.per_query_head:
            ab = res["score_ab"]
            kms = res["kern"]["score"]
            tr = traffic_from_profile("score.cu", "score_qh.long_context_gqa.md") \
                if args.config == 5 and c.H_q // c.H_kv <= 8 else None
            kname = ("score_qh_kernel" if c.H_q // c.H_kv <= 8 else "score_kernel<per-head>") + " (sa_score_pages_qh)"
        elif c.ps > 1:
            ab = res["score_ab"]
            kms = res["kern"]["score"]
            tr = traffic_from_profile("score.cu", "score_pages.long_context_gqa.md") \
                if args.config == 5 else None
            kname = "score_kernel (sa_score_pages)"
        else:
            ab = 2 * c.D * 2 * (c.budget + 1) * c.B * c.H_kv
            kms = res["kern"]["decode"]
            tr = None
            kname = "decode_kernel (sa_sparse_decode)"
        ach = ab / (kms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                "frac": ach / hbm_peak, "traffic": tr, "kernel": kname,
                "peak_kind": peak_kind, "algorithmic_bytes_per_launch": ab,
                "kernel_ms": res["kern"]}
    cpu = None
    if world == 1 and not args.no_cpu:
        alpha = (args.entmax or 1.5) if args.gaussian else (args.entmax or 1.0)
        walls = cpu_baseline(res["wl"], args.cpu_steps, workers, alpha, args.gaussian)
        n1 = min(4, c.B * c.H_kv)
        v1, wall1 = cpu_one_thread(res["wl"], n1, alpha, args.gaussian)
        cpu = {"value": 1.0 / statistics.mean(walls), "unit": "steps/s", "cores": workers,
               "kind": "oracle",
               "sample": (f"{len(walls)} full step(s): all {c.B * c.H_kv} (request, KV head) "
                          f"units, float64 numpy oracle, one unit per task on {workers} "
                          f"spawned single-threaded workers"),
               "one_thread": {"value": v1, "unit": "steps/s", "cores": 1,
                              "sample": f"{n1} of the {c.B * c.H_kv} units of a step on one worker "
                                        f"({wall1:.2f} s), scaled to full steps"}}
    also = None
    if (world == 1 and args.config == 5 and not (args.gaussian or args.entmax or args.per_query_head)
            and not args.no_also):
        also = {"batched_gqa_ragged": run_also(args, rank, world, hbm_peak, peak_kind)}
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["max_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": c.dtype, "data": "synthetic",
        "config": {"workload": describe(c) + (", pages selected per query head"
                                              if args.per_query_head else "")
                   + (", Gaussian-aware selection per query head, "
                      f"{args.entmax or 1.5}-entmax" if args.gaussian else
                      (f", {args.entmax}-entmax instead of softmax" if args.entmax else "")),
                   "l2": "flushed between steps outside the events: 256 MB write, then a 256 MB read so the flush's dirty lines are written back before the step",
                   "timing": "CUDA events around each step (graph replay); the step's q / k_new / v_new are copied from the HBM-resident input set into its input buffers before the events; every 100 steps a device-side sleep outside the events lets the host enqueue ahead",
                   "parallelism": f"independent batch per GPU x{world}"},
        "hbm_gbs": step_gbs, "hbm_frac": step_gbs / hbm_peak, "hbm_peak_kind": peak_kind,
        "hbm_frac_nominal": step_gbs / NOMINAL_HBM,
        "algorithmic_bytes_per_step": res["bytes"],
        "step_ms_min": res["step_ms_min"], "step_ms_max": res["step_ms_max"],
        "step_ms_median": res["step_ms_median"],
        "steps_per_s_median": aggregate_steps_per_s(res["max_median_ms"], world),
        "roofline": roof, "cpu_baseline": cpu, "e2e": res["e2e"], "also": also,
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": res["clocks"], "dev_status": res["status"],
    }
    if res["ent"]:
        line["entmax"] = res["ent"]
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
