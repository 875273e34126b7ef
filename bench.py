#!/usr/bin/env python
"""MoG decode benchmark: microseconds per decode step per layer, and achieved HBM GB/s of
the dominant decode kernel against the measured HBM roofline.

Workload (default): the 1M-token layer -- 32 query heads over 8 KV heads, d = 128,
N = 1048576 bf16 keys per KV head from the planted-centre generator (4096 centres,
sigma 0.5), 1024 clusters x 20 subclusters, top-16 clusters x top-8 subclusters, 4 sink +
512 recent anchors.  The build runs once before timing (prefill time); a step is one
mog_decode of the whole layer.  Before every timed step L2 is made cold: a 256 MB write,
then a 256 MB read.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mog|reference] [--workload W]

--impl reference times the CPU oracle (the plain fp64 statement of the method) on the
host cores, on every KV head and query head of the same layer, for K steps after W.
Under torchrun every rank runs an independent replica (the method has no cross-GPU
exchange); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from serving_mog_decode_gb300 import workloads as wl  # noqa: E402

METRIC = "MoG decode us/step/layer at 32K-1M ctx; achieved HBM GB/s vs roofline"
D = 128
FLUSH_BYTES = 256 << 20
APPEND_STEPS = 36         # appends timed with --sliding (the first four are warm-up)
CUSHION_CYCLES = 200_000   # GPU-side spin before each timed step (~0.1 ms): the host
                           # finishes enqueueing the step before the start event is reached


def args_():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mog", choices=["mog", "reference"])
    ap.add_argument("--workload", default="ctx-1m", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="budget of the oracle timing sample (decode steps of the whole layer)")
    ap.add_argument("--no-ablation", action="store_true",
                    help="skip the top-only and score-mode-1 arms")
    ap.add_argument("--settle-seconds", type=float, default=0.5,
                    help="decode loop before the timings, to settle the clocks")
    ap.add_argument("--phase-steps", type=int, default=0,
                    help="steps of the per-kernel timing (0: max(20, min(steps, 200)))")
    ap.add_argument("--no-dense", action="store_true",
                    help="skip the dense_decode comparison (profiling runs)")
    ap.add_argument("--sliding", action="store_true",
                    help="sliding recent window; the cache gets room for the append timing "
                         "that follows the decode timing")
    ap.add_argument("--group-select", action="store_true",
                    help="group-shared selection: the query heads of a KV head select once, "
                         "by the log-sum-exp of their scores")
    ap.add_argument("--paged", type=int, default=0, metavar="ROWS",
                    help="hold the cache as pages of ROWS rows (a power of two) in a random "
                         "order behind a block table")
    ap.add_argument("--bf16-summaries", action="store_true",
                    help="selection scores and residual terms from the summaries rounded to bf16")
    ap.add_argument("--fm-residual", action="store_true",
                    help="the feature-map residual (random features) instead of the Gaussian one")
    ap.add_argument("--kmeanspp", action="store_true",
                    help="first-level k-means++ seeds (draws from the input generator)")
    ap.add_argument("--fp8-summaries", action="store_true",
                    help="selection scores and residual terms from the summaries rounded to fp8 e4m3")
    ap.add_argument("--union-exact", action="store_true",
                    help="GQA union-exact mode: every query head attends the union of the "
                         "chosen subclusters of its KV group")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


DECODE_SOURCES = ("attend.cuh", "common.cuh", "decode.cu", "internal.h")


def kernel_hash():
    """Hash of the sources the decode kernels are compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "serving_mog_decode_gb300", "csrc")
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def stored_traffic(workload, kernel):
    """dram bytes per launch of `kernel` from a committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(workload, {}).get(kernel)
        if e and e.get("source_hash") == kernel_hash():
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


class Clocks:
    """nvidia-smi sampling (200 ms) around the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", str(dev_index)], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------ the oracle

def oracle_layer(w, arrays=None):
    """Per-unit inputs and oracle summaries of the whole layer (untimed set-up).  Small
    layers use the oracle's own two-level k-means; for larger ones (whose fp64 k-means
    takes hours) every unit gets a planted-centre/position partition: clusters by planted
    centre, subclusters by position.  `arrays` = (K, V, q) of the batch, if already drawn.
    Returns (units, how the partition was made) with units = [(K, V, n, q[G], summ)]."""
    import oracle
    lens = wl.lengths(w)
    own = w.batch * w.h_kv * int(lens.max()) <= (1 << 18)
    G, units = w.group, []
    for b in range(w.batch):
        n = int(lens[b])
        Cn, L = wl.clusters_for(w, n)
        for h in range(w.h_kv):
            u = wl.UnitDraw(w, b, h, n)
            if arrays is None:
                K, V = u.keys_values()
                q = u.q
            else:
                K, V = arrays[0][b, h, :n], arrays[1][b, h, :n]
                q = arrays[2][b, h * G:(h + 1) * G]
            S, R = w.n_sink, w.n_recent
            if own:
                summ = oracle.build_unit(K, V, n, S, R, Cn, L)
            else:
                pos = np.arange(S, max(S, n - R))
                lab = (u.z[pos] % Cn) * L + (pos % L)
                order = np.argsort(lab, kind="stable")
                perm = pos[order].astype(np.int32)
                sub_off = np.searchsorted(lab[order], np.arange(Cn * L + 1)).astype(np.int32)
                summ = oracle.stats(K, V, perm, sub_off, Cn, L)
                summ.update(perm=perm, sub_off=sub_off, C=Cn, L=L, n_build=n, S=S, R=R)
            units.append((K, V, n, q, summ))
    how = ("the oracle's own two-level k-means" if own else
           "a planted-centre/position partition (the fp64 k-means of this layer is out of budget)")
    return units, how


def oracle_decode_sample(w, budget_s, steps=None, warmup=0, arrays=None, dense_steps=0):
    """Time the oracle's decode step (selection + exact + residual) of the whole layer:
    every query head of every KV head, spread over a thread pool of all host cores (each
    oracle call is single-threaded and releases the interpreter lock).  Runs `steps`
    steps after `warmup` (or, with steps None, as many as fit in budget_s).  With
    dense_steps > 0 the oracle's dense attention of the layer is timed too.
    Returns (us per step per layer, cores, description, per-step list, dense us or None)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    oracle.build()
    units, how = oracle_layer(w, arrays)
    cores = os.cpu_count() or 1
    tasks = [(i, g) for i in range(len(units)) for g in range(w.group)]

    def head(t):
        K, V, n, q, summ = units[t[0]]
        oracle.mog_head(K, V, n, q[t[1]], summ, w.top_c, w.top_s)

    def dense_head(t):
        K, V, n, q, _ = units[t[0]]
        oracle.dense(K, V, n, q[t[1]])

    with ThreadPoolExecutor(max_workers=cores) as ex:
        def one(fn):
            t0 = time.perf_counter()
            list(ex.map(fn, tasks))
            return (time.perf_counter() - t0) * 1e6

        for _ in range(warmup):
            one(head)
        times = []
        t_end = time.perf_counter() + budget_s
        while (steps is None and (time.perf_counter() < t_end or len(times) < 3)) or \
                (steps is not None and len(times) < steps):
            times.append(one(head))
            if steps is None and len(times) >= 1000:
                break
        dense_us = statistics.mean(one(dense_head) for _ in range(dense_steps)) if dense_steps else None
    desc = (f"the whole layer ({len(units)} KV heads x {w.group} query heads), oracle decode step "
            f"timed {len(times)}x on a pool of {cores} threads; summaries from {how}, untimed")
    if dense_us is not None:
        desc += f"; the oracle's dense attention of the layer timed {dense_steps}x"
    return statistics.mean(times), cores, desc, times, dense_us


# ------------------------------------------------------------------------ GPU path

def summary_bytes(a):
    """Bytes per element of the summaries' means and variances the decode reads."""
    return 1 if a.fp8_summaries else 2 if a.bf16_summaries else 4


def bytes_from_selection(h, w, sel, lens, n_now, sb=4, resid=1):
    """Algorithmic bytes of one decode step, per kernel: all cluster summaries and the
    subcluster summaries of each unit's union of selected clusters (selection); the K/V
    rows (+ index) of the union of selected subclusters, the anchors and the residual terms
    (rows); the partials and the output (merge).  sb: bytes per element of the summaries'
    means and variances (4 fp32, 2 bf16, 1 fp8); the residual terms' value means take 4
    (bf16 high and low parts) with fp32 summaries, else 2 (the high part).  resid: 1 the
    Gaussian residual's terms (rows kernel), 0 none, 2 the feature-map residual (its own
    kernel: per head the unit's total and the chosen subclusters' feature sums, 32 x 132
    floats each, and FM_NCH + 1 vectors out, which the merge reads)."""
    import torch
    lay = h.layout()
    U, cm, lm, G = lay.units, lay.c_max, lay.l_max, lay.group
    info = h.array("unit_info", torch.int32, (U, 8)).cpu().numpy()
    off = h.array("sub_off", torch.int32, (U, lay.sub_off_stride)).cpu().numpy()
    tc, ts = w.top_c, w.top_s
    sel = sel.reshape(U, G, -1)
    tot = dict(select=0, attend=0, merge=0, rows=0, fm=0)
    fm_row = 32 * 132 * 4   # one feature sum (all features), bytes
    fm_vec = 33 * 132 * 4   # the vectors one head's CTAs write
    for u in range(U):
        Cn, L, nb, S, rlo, b = info[u, 0], info[u, 1], info[u, 2], info[u, 4], info[u, 5], info[u, 6]
        ucl, usub = set(), set()
        for g in range(G):
            for i in range(tc):
                c = sel[u, g, i]
                if c < 0:
                    continue
                ucl.add(int(c))
                for r in range(ts):
                    l = sel[u, g, tc + i * ts + r]
                    if l >= 0:
                        usub.add((int(c), int(l)))
        Uk = sum(int(off[u, c * L + l + 1] - off[u, c * L + l]) for c, l in usub)
        anchors = min(S, n_now[b]) + max(0, n_now[b] - rlo)
        items = len(ucl) * L + Cn  # residual terms: the union's subclusters, then clusters
        gp = (G + 3) // 4 * 4
        P = h.splits()
        vb = 4 if sb == 4 else 2  # bytes per value-mean element of a residual term
        # selection kernel: query, cluster summaries (mean, variance, count), the union's
        # subcluster summaries and offsets; writes the segments and the residual exponents
        tot["select"] += G * D * 2 + Cn * (2 * sb * D + 4) + len(ucl) * (L * (2 * sb * D + 8) + 4)
        tot["select"] += len(usub) * 12 + items * gp * 4
        # rows kernel: query, segments, perm index and K, V rows (bf16) of the chosen rows and
        # the anchors, the residual terms (bf16 high/low value means and exponents), partials
        tot["attend"] += G * D * 2 + len(usub) * 12 + Uk * 4 + (Uk + anchors) * 4 * D
        if resid == 1:
            tot["attend"] += items * (vb * D + gp * 4)
        tot["attend"] += P * G * (D + 4) * 4
        if resid == 2:
            for g in range(G):
                nsel = sum(1 for i in range(tc) if sel[u, g, i] >= 0
                           for r in range(ts) if sel[u, g, tc + i * ts + r] >= 0)
                tot["fm"] += D * 2 + 4 * (tc + tc * ts) + (1 + nsel) * fm_row + fm_vec
                tot["merge"] += fm_vec + 4
        # merge kernel: partials in, the output (fp32) out
        tot["merge"] += P * G * (D + 4) * 4 + G * D * 4
        tot["rows"] += Uk + anchors
    tot["step"] = tot["select"] + tot["attend"] + tot["merge"] + tot["fm"]
    return tot


def run_gpu(a, w, rank, world):
    import torch

    import serving_mog_decode_gb300 as mog
    from serving_mog_decode_gb300 import buildlib

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(mog.LIB_PATH):
        buildlib.build()
    if world > 1:
        torch.distributed.barrier()

    lens = wl.lengths(w)
    K, V, q, _ = wl.make_batch(w)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)

    if a.sliding:  # room for the appends timed after the decode steps
        pad = ((0, 0), (0, 0), (0, APPEND_STEPS), (0, 0))
        K, V = np.pad(K, pad), np.pad(V, pad)
    Kd, Vd, qd = bf(K), bf(V), bf(q)
    host_arrays = (K, V, q)  # kept for the oracle's timing sample (rank 0)
    if a.paged:  # the same cache as pages in a random order behind a block table
        pr = a.paged
        B, H, ncap = Kd.shape[0], Kd.shape[1], Kd.shape[2]
        pps = -(-ncap // pr)
        order = torch.randperm(B * pps, generator=torch.Generator().manual_seed(5)).to(dev)
        pools = []
        for X in (Kd, Vd):
            Xp = torch.nn.functional.pad(X, (0, 0, 0, pps * pr - ncap))
            Xp = Xp.view(B, H, pps, pr, D).permute(0, 2, 1, 3, 4).reshape(B * pps, H, pr, D)
            pool = torch.empty_like(Xp)
            pool[order] = Xp
            pools.append(pool)
        del Xp
        Kd = mog.PagedKV(pools[0], pools[1], order.view(B, pps).to(torch.int32).contiguous(), pr)
        Vd = None
        torch.cuda.empty_cache()
    n_cap = K.shape[2]
    prm = mog.make_params(w.batch, w.h_kv, w.h_q, n_cap, n_clusters=w.n_clusters, n_sub=w.n_sub,
                          top_c=w.top_c, top_s=w.top_s, n_sink=w.n_sink, n_recent=w.n_recent,
                          union_exact=int(a.union_exact), sliding=int(a.sliding),
                          group_select=int(a.group_select), bf16_summaries=int(a.bf16_summaries),
                          fp8_summaries=int(a.fp8_summaries), kmeanspp=int(a.kmeanspp),
                          residual=2 if a.fm_residual else 1)
    omega = (torch.from_numpy(wl.fm_omega(mog.FM_FEATURES, D, w.seed + 200)).to(torch.float32).to(dev)
             if a.fm_residual else None)
    draws = None
    if a.kmeanspp:
        tl = mog.trace_layout(prm, lens)
        draws = torch.from_numpy(wl.seed_draws(tl.units, tl.c_max, w.seed + 100)).to(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def cold_l2():
        """Write a buffer larger than L2, then read another one: L2 ends cold for the step's
        inputs and clean (no write-back of the flush data inside the timed step)."""
        flush.zero_()
        flush_rd.sum()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    # ---- build (once, prefill time) ----
    torch.cuda.synchronize()
    b0, b1 = ev(), ev()
    b0.record()
    h = mog.build(Kd, Vd, lens, prm, draws=draws)
    b1.record()
    torch.cuda.synchronize()
    build_ms = b0.elapsed_time(b1)
    fm_ms = None
    if a.fm_residual:   # the feature-map summary, also at prefill time
        b0.record()
        h.feature_map(omega)
        b1.record()
        torch.cuda.synchronize()
        fm_ms = b0.elapsed_time(b1)
    assert h.sync_status() == 0
    lay = h.layout()
    steps1 = h.array("l1_steps", torch.int32, (lay.units,)).cpu().numpy()
    info = h.array("unit_info", torch.int32, (lay.units, 8)).cpu().numpy()
    l1_flop = float(sum(2.0 * info[u, 3] * D * info[u, 0] * steps1[u] for u in range(lay.units)))
    l2_flop = float(sum(2.0 * info[u, 3] * D * info[u, 1] * 10 for u in range(lay.units)))

    out = torch.empty(qd.shape, dtype=torch.float32, device=dev)
    SW = w.top_c + w.top_c * w.top_s
    sel = torch.empty((lay.units * lay.group, max(SW, 1)), dtype=torch.int32, device=dev)
    h.decode(qd, out, sel_out=sel)
    torch.cuda.synchronize()
    n_now = [int(x) for x in lens]
    by = bytes_from_selection(h, w, sel.cpu().numpy(), lens, n_now, summary_bytes(a), prm.residual)

    clocks = Clocks(local)
    # ---- settle clocks, then dense_decode (the full scan) for comparison ----
    t_end = time.time() + a.settle_seconds
    while time.time() < t_end:
        for _ in range(50):
            h.decode(qd, out)
        torch.cuda.synchronize()
    dense_out = torch.empty_like(out)
    dscratch = torch.empty(mog.dense_scratch_bytes(w.batch, w.h_kv, w.h_q, int(lens.max())),
                           dtype=torch.uint8, device=dev)
    dense_ms = []
    for i in range(1 if a.no_dense else 3 + 10):  # (one untimed call for the error below)
        cold_l2()
        torch.cuda._sleep(CUSHION_CYCLES)
        s0, s1 = ev(), ev()
        s0.record()
        mog.dense_decode(Kd, Vd, h.lengths_dev, int(lens.max()), qd, dense_out, dscratch)
        s1.record()
        torch.cuda.synchronize()
        if i >= 3 and not a.no_dense:
            dense_ms.append(s0.elapsed_time(s1))
    dense_bytes = float(sum(int(lens[u // w.h_kv]) for u in range(lay.units))) * 4 * D
    # approximation error of the MoG output against the full scan, per query head
    h.decode(qd, out)
    torch.cuda.synchronize()
    o, dn = out.reshape(-1, D).double(), dense_out.reshape(-1, D).double()
    err = ((o - dn).norm(dim=1) / dn.norm(dim=1).clamp_min(1e-30)).cpu().numpy()
    approx = {"median_rel_l2": float(np.median(err)), "p90_rel_l2": float(np.percentile(err, 90)),
              "max_rel_l2": float(err.max()), "heads": int(err.size)}
    # ---- ablations on the same partition: top-only (no residual) and score mode 1 ----
    ablation = None
    if not a.no_ablation:
        perm_t = h.array("perm", torch.int32, (lay.units, lay.n_cap)).clone()
        off_t = h.array("sub_off", torch.int32, (lay.units, lay.sub_off_stride)).clone()
        ablation = {}
        for name, over in (("top_only", dict(residual=0)), ("score_mode_1", dict(score_mode=1))):
            kw = dict(n_clusters=w.n_clusters, n_sub=w.n_sub, top_c=w.top_c, top_s=w.top_s,
                      n_sink=w.n_sink, n_recent=w.n_recent, union_exact=int(a.union_exact),
                      sliding=int(a.sliding), group_select=int(a.group_select),
                      bf16_summaries=int(a.bf16_summaries),
                      fp8_summaries=int(a.fp8_summaries))
            kw.update(over)
            kw.setdefault("residual", 2 if a.fm_residual else 1)
            pv = mog.make_params(w.batch, w.h_kv, w.h_q, n_cap, **kw)
            hv = mog.build(Kd, Vd, lens, pv, partition=(perm_t, off_t))
            if pv.residual == 2:
                hv.feature_map(omega)
            sv = torch.empty_like(sel)
            ov = hv.decode(qd, sel_out=sv)
            torch.cuda.synchronize()
            assert hv.sync_status() == 0
            ev_ = ((ov.reshape(-1, D).double() - dn).norm(dim=1) / dn.norm(dim=1).clamp_min(1e-30)).cpu().numpy()
            byv = bytes_from_selection(hv, w, sv.cpu().numpy(), lens, n_now, summary_bytes(a), pv.residual)
            tv = []
            for i in range(3 + 20):
                cold_l2()
                torch.cuda._sleep(CUSHION_CYCLES)
                s0, s1 = ev(), ev()
                s0.record()
                hv.decode(qd, ov)
                s1.record()
                torch.cuda.synchronize()
                if i >= 3:
                    tv.append(s0.elapsed_time(s1))
            ablation[name] = {
                "us": round(statistics.mean(tv) * 1e3, 2),
                "kv_rows_read": int(byv["rows"]),
                "kv_read_fraction": round(byv["rows"] / float(sum(n_now[u // w.h_kv] for u in range(lay.units))), 4),
                "approx_vs_dense": {"median_rel_l2": round(float(np.median(ev_)), 6),
                                    "p90_rel_l2": round(float(np.percentile(ev_, 90)), 6),
                                    "max_rel_l2": round(float(ev_.max()), 6)}}
            del hv, ov, sv
        del perm_t, off_t
    # ---- the timed decode steps ----
    for _ in range(a.warmup):
        cold_l2()
        h.decode(qd, out)
    starts = [ev() for _ in range(a.steps)]
    ends = [ev() for _ in range(a.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(a.steps):
        cold_l2()
        torch.cuda._sleep(CUSHION_CYCLES)
        starts[i].record()
        h.decode(qd, out)
        ends[i].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # ---- per-kernel times (events around the selection, rows and merge kernels) ----
    # Events between the kernels stop each from starting early, so the rows and merge
    # kernels would fetch their code from DRAM after the L2 flush with nothing to overlap
    # it (in the step they load it while their predecessor runs).  The data stays cold;
    # a decode on a small side handle after the flush brings the kernels' code back.
    side = None
    try:
        sw = wl.Workload("side", batch=1, h_kv=w.h_kv, h_q=w.h_q, n=4096, centres=32, seed=7)
        sK, sV, sq, sl = wl.make_batch(sw)
        sL = min(w.n_sub if w.n_sub > 0 else 8, 8)
        sp = mog.make_params(1, w.h_kv, w.h_q, 4096, n_clusters=32, n_sub=sL, top_c=min(w.top_c, 16),
                             top_s=min(w.top_s, sL), n_sink=4, n_recent=64,
                             union_exact=int(a.union_exact), group_select=int(a.group_select),
                             bf16_summaries=int(a.bf16_summaries),
                             fp8_summaries=int(a.fp8_summaries), residual=prm.residual)
        sKd, sVd, sqd = bf(sK), bf(sV), bf(sq)
        sh = mog.build(sKd, sVd, sl, sp)
        if sp.residual == 2:
            sh.feature_map(omega)
        side = (sh, sqd, torch.empty(sqd.shape, dtype=torch.float32, device=dev))
    except Exception:
        side = None
    phase = [[], [], []]
    for i in range(a.phase_steps if a.phase_steps > 0 else max(20, min(a.steps, 200))):
        cold_l2()
        if side is not None:
            side[0].decode(side[1], side[2])
        torch.cuda._sleep(CUSHION_CYCLES)
        evs = [ev() for _ in range(4)]
        h.decode_phased(qd, out, evs)
        torch.cuda.synchronize()
        for k in range(3):
            phase[k].append(evs[k].elapsed_time(evs[k + 1]))
    # ---- end to end through the C ABI with host buffers ----
    q_host = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    e2e_ms = []
    for i in range(a.warmup + a.steps):
        cold_l2()
        s0, s1 = ev(), ev()
        s0.record()
        qd.copy_(q_host, non_blocking=True)
        h.decode(qd, out)
        out_host.copy_(out, non_blocking=True)
        s1.record()
        torch.cuda.synchronize()
        if i >= a.warmup:
            e2e_ms.append(s0.elapsed_time(s1))
    clk = clocks.stop()
    assert h.sync_status() == 0
    append = None
    if a.sliding:  # mog_append: the new rows, then each KV head's oldest recent key moves in
        kn = torch.randn(w.batch, w.h_kv, D, device=dev).to(torch.bfloat16)
        vn = torch.randn(w.batch, w.h_kv, D, device=dev).to(torch.bfloat16)
        app_ms = []
        for i in range(APPEND_STEPS):
            s0, s1 = ev(), ev()
            s0.record()
            h.append(kn, vn)
            s1.record()
            torch.cuda.synchronize()
            if i >= 4:
                app_ms.append(s0.elapsed_time(s1))
        assert h.sync_status() == 0
        append = {"us_median": round(statistics.median(app_ms) * 1e3, 2), "appends": len(app_ms),
                  "what": "mog_append with the sliding window, events around the call (launch overhead included)"}

    mean_ms = max_over_ranks(statistics.mean(step_ms), dev)
    pm = [statistics.mean(p) for p in phase]
    names = ["k_mog_decode", "k_mog_rows", "k_mog_merge"]
    kbytes = [by["select"], by["attend"], by["merge"]]
    dom = max(range(3), key=lambda i: pm[i])
    peak, peak_kind = peaks()
    achieved = kbytes[dom] / (pm[dom] * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(mean_ms * 1e3 / world, 3),
        "unit": "us/step/layer",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": round(mean_ms, 5),
        "step_us_median": round(statistics.median(step_ms) * 1e3, 3),
        "step_us_min": round(min(step_ms) * 1e3, 3),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (planted-centre keys, Gaussian values; seeded)",
        "config": {"workload": w.name, "batch": w.batch, "h_kv": w.h_kv, "h_q": w.h_q, "d": D,
                   "context": int(lens.max()), "clusters": w.n_clusters, "subclusters": w.n_sub,
                   "top_c": w.top_c, "top_s": w.top_s, "n_sink": w.n_sink, "n_recent": w.n_recent,
                   "mode": ("group-shared selection" if a.group_select else "per-head selection")
                           + (", union-exact" if a.union_exact else "")
                           + (", bf16 summaries" if a.bf16_summaries else "")
                           + (", fp8 summaries" if a.fp8_summaries else "")
                           + (", k-means++ seeds" if a.kmeanspp else "")
                           + (", feature-map residual" if a.fm_residual else "")
                           + (f", paged cache ({a.paged}-row pages)" if a.paged else ""),
                   "recent_window": "sliding" if a.sliding else "growing",
                   "l2": "cold before every timed step (256 MB write, then 256 MB read)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": stored_traffic(w.name, names[dom]),
                     "algorithmic_bytes_per_launch": int(kbytes[dom]),
                     "launch_us": round(pm[dom] * 1e3, 3)},
        "kernels_us": {names[i]: round(pm[i] * 1e3, 3) for i in range(3)},
        "kernels_timing": ("mog_decode_phased: events around each kernel (no overlap between the "
                           "kernels, no warm-up passes); data cold (L2 flushed); the kernels' code "
                           "re-warmed by a decode on a small side handle" if side is not None else
                           "mog_decode_phased: events around each kernel; data and code cold (L2 flushed)"),
        "kernels_GBps": {names[i]: round(kbytes[i] / (pm[i] * 1e-3) / 1e9, 1) for i in range(3)},
        "step_bytes": int(by["step"]),
        "step_GBps": round(by["step"] / (mean_ms * 1e-3) / 1e9, 1),
        "step_frac_of_peak": round(by["step"] / (mean_ms * 1e-3) / 1e9 / peak, 4),
        "kv_rows_read": int(by["rows"]),
        "kv_read_fraction": round(by["rows"] / float(sum(n_now[u // w.h_kv] for u in range(lay.units))), 4),
        "dense_decode": ({"us": round(statistics.mean(dense_ms) * 1e3, 2),
                          "GBps": round(dense_bytes / (statistics.mean(dense_ms) * 1e-3) / 1e9, 1),
                          "frac": round(dense_bytes / (statistics.mean(dense_ms) * 1e-3) / 1e9 / peak, 4)}
                         if dense_ms else None),
        "speedup_vs_dense": round(statistics.mean(dense_ms) / mean_ms, 2) if dense_ms else None,
        "approx_vs_dense": {k: (round(v, 6) if isinstance(v, float) else v) for k, v in approx.items()},
        "approx_vs_dense_top_only": ablation["top_only"]["approx_vs_dense"] if ablation else None,
        "ablation": ablation,
        "build": {"ms": round(build_ms, 2), "l1_flop": l1_flop, "l2_flop": l2_flop,
                  "TFLOPs": round((l1_flop + l2_flop) / (build_ms * 1e-3) / 1e12, 3),
                  # k-means++ reads every mid key once per seed (2 bytes x d each)
                  "kmeanspp_key_bytes": (sum(float(info[u, 3]) * 2 * D * float(info[u, 0]) for u in range(lay.units))
                                         if a.kmeanspp else None),
                  "feature_map_ms": round(fm_ms, 2) if fm_ms is not None else None},
        "e2e": {"value": round(statistics.mean(e2e_ms) * 1e3 / world, 3), "unit": "us/step/layer",
                "h2d_bytes_per_step": int(q_host.numel() * 2), "d2h_bytes_per_step": int(out_host.numel() * 4)},
        "append": append,
        # selection, rows and merge kernels per step (and the feature-map kernel with it)
        "gpu_launches": (4 if a.fm_residual else 3) * a.steps,
        "clocks": clk,
    }
    if rank == 0 and a.cpu_seconds <= 0:   # timing experiments only: no CPU baseline
        print(json.dumps(res), flush=True)
    elif rank == 0:
        mu, cores, desc, _, dense_cpu = oracle_decode_sample(w, a.cpu_seconds, arrays=host_arrays,
                                                             dense_steps=2)
        res["cpu_baseline"] = {"value": round(mu, 1), "unit": "us/step/layer", "cores": cores,
                               "kind": "oracle", "sample": desc,
                               "dense_us": round(dense_cpu, 1) if dense_cpu else None}
        print(json.dumps(res), flush=True)


def max_over_ranks(value, device):
    """The maximum of `value` over all ranks of the default process group (the value itself
    when no group is initialised): the job's time is its slowest replica's."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_reference(a, w, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    mu, cores, desc, times, _ = oracle_decode_sample(w, a.cpu_seconds, steps=a.steps, warmup=a.warmup)
    res = {"metric": METRIC, "impl": "reference", "value": round(mu, 1), "unit": "us/step/layer",
           "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
           "ms_per_step": round(mu / 1e3, 4), "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (planted-centre keys; seeded)",
           "config": {"workload": w.name},
           "cpu_baseline": {"value": round(mu, 1), "unit": "us/step/layer", "cores": cores,
                            "kind": "oracle", "sample": desc},
           "e2e": {"value": round(mu, 1), "unit": "us/step/layer", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    a = args_()
    w = wl.WORKLOADS[a.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if a.impl == "reference":
        run_reference(a, w, rank)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    run_gpu(a, w, rank, world)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
