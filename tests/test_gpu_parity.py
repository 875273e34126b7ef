"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the same
seeded inputs.  Oracle state (centroids, partitions, selections) is injected into the
GPU, never the other way round.

Tolerances:
  k-means assignments           bit-exact given the same (fp32) centroids
  summaries (count exact)       per-group relative L2 <= 1e-5 for mean, variance, value mean
  selection                     identical except where the score gap to the cut-off < 1e-4
  outputs (same selection)      per-head relative L2 <= 1e-3
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle as ora
import serving_mog_decode_gb300 as mog
from serving_mog_decode_gb300 import buildlib
from serving_mog_decode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
D = 128
DEV = torch.device("cuda:0")
TIE = 1e-4
OUT_TOL = 1e-3
STAT_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    buildlib.build()
    ora.build()
    mog.lib()


def bf(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-30))


def small_workload(n, centres=64, **kw):
    base = dict(batch=1, h_kv=1, h_q=1, n=n, centres=centres, n_clusters=16, n_sub=6, top_c=4,
                top_s=3, n_sink=4, n_recent=32, seed=11)
    base.update(kw)
    return wl.Workload("test", **base)


# --------------------------------------------------------------------------- dense

@pytest.mark.parametrize("lens,G", [((1300, 777), 4), ((64,), 1), ((200, 5000, 1), 5)])
def test_dense_decode_matches_oracle(lens, G):
    B, Hkv = len(lens), 2
    w = small_workload(max(lens), batch=B, h_kv=Hkv, h_q=Hkv * G)
    n_cap = max(lens) + 3
    K = np.zeros((B, Hkv, n_cap, D), np.uint16)
    V = np.zeros_like(K)
    q = np.zeros((B, Hkv * G, D), np.uint16)
    for b in range(B):
        for h in range(Hkv):
            u = wl.UnitDraw(w, b, h, lens[b])
            u.keys_values(K[b, h], V[b, h])
            q[b, h * G:(h + 1) * G] = u.q
    ld = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = mog.dense_decode(bf(K), bf(V), ld, max(lens), bf(q)).cpu().numpy()
    for b in range(B):
        for hq in range(Hkv * G):
            ref = ora.dense(K[b, hq // G], V[b, hq // G], lens[b], q[b, hq])
            assert rel(out[b, hq], ref) < OUT_TOL, (b, hq)


# --------------------------------------------------------------------------- k-means

def _assign_steps(Kmid, k, T):
    _, _, steps, hist = ora.lloyd(Kmid, k, T, history=True)
    x = bf(Kmid)
    total_fb = 0
    for t in range(steps):
        c32 = hist[t].astype(np.float32)
        gpu, fb = mog.kmeans_assign(x, torch.from_numpy(c32).to(DEV))
        ref = ora.assign(Kmid, c32.astype(np.float64))
        assert np.array_equal(gpu.cpu().numpy(), ref), f"step {t}"
        total_fb += fb
    return steps, total_fb


def test_l1_assign_bit_exact_tiny():
    w = wl.WORKLOADS["tiny-4k"]
    K, _, _ = wl.make_unit(w)
    mid = K[w.n_sink:w.n - w.n_recent]
    steps, fb = _assign_steps(mid, w.n_clusters, 10)
    assert steps >= 3
    print(f"tiny: {steps} steps, {fb} rows decided by the fp64 fallback")


def test_l1_assign_bit_exact_with_ties_and_ragged_tail():
    g = np.random.default_rng(5)
    base = g.standard_normal((40, D))
    X = wl.to_bf16(np.repeat(base, 3, axis=0)[:117])          # exact duplicate rows, ragged
    cent = np.concatenate([base[:10], base[:10], g.standard_normal((13, D))]).astype(np.float32)
    gpu, fb = mog.kmeans_assign(bf(X), torch.from_numpy(cent).to(DEV))
    ref = ora.assign(X, cent.astype(np.float64))
    assert np.array_equal(gpu.cpu().numpy(), ref)
    assert fb > 0       # duplicated centroids tie exactly and must go to the fp64 rule


def test_l1_assign_bit_exact_qwen3_4b_unit():
    """A full 32K-key KV head of the Qwen3-4B-shaped workload (181 centroids)."""
    w = wl.WORKLOADS["qwen3-4b-32k"]
    K, _, _ = wl.make_unit(w, 0, 3)
    mid = K[w.n_sink:w.n - w.n_recent]
    _assign_steps(mid, w.n_clusters, 2)


def test_l1_assign_tensor_core_pass_decides_most_rows():
    """The tensor-core scores decide almost every row of a full 32K-key head; the rest go
    through the direct fp32 pass (and, if needed, the fp64 rule) and still match."""
    w = wl.WORKLOADS["qwen3-4b-32k"]
    K, _, _ = wl.make_unit(w, 0, 5)
    mid = K[w.n_sink:w.n - w.n_recent]
    _, _, steps, hist = ora.lloyd(mid, w.n_clusters, 2, history=True)
    c32 = hist[steps - 1].astype(np.float32)
    gpu, fb, rc = mog.kmeans_assign(bf(mid), torch.from_numpy(c32).to(DEV), with_recheck=True)
    assert np.array_equal(gpu.cpu().numpy(), ora.assign(mid, c32.astype(np.float64)))
    print(f"32K head: {rc} of {mid.shape[0]} rows rechecked, {fb} by the fp64 rule")
    assert rc < 0.05 * mid.shape[0]


def test_l1_assign_bit_exact_many_chunks_ragged_outliers():
    """More than 256 centroids (several tensor-core groups, the last one ragged), a row
    count that is not a multiple of the 128-row tile, and keys scaled x4 (large norms)."""
    g = np.random.default_rng(11)
    centres = g.standard_normal((700, D))
    z = g.integers(0, 700, size=3001)
    X = centres[z] + 0.5 * g.standard_normal((3001, D))
    X[g.choice(3001, size=30, replace=False)] *= 4.0
    Xb = wl.to_bf16(X)
    cent = (centres[:301] + 0.05 * g.standard_normal((301, D))).astype(np.float32)
    gpu, fb, rc = mog.kmeans_assign(bf(Xb), torch.from_numpy(cent).to(DEV), with_recheck=True)
    assert np.array_equal(gpu.cpu().numpy(), ora.assign(Xb, cent.astype(np.float64)))
    assert rc < 3001


def test_l1_assign_single_centroid_and_single_row():
    g = np.random.default_rng(12)
    X = wl.to_bf16(g.standard_normal((1, D)))
    cent = g.standard_normal((1, D)).astype(np.float32)
    gpu, fb = mog.kmeans_assign(bf(X), torch.from_numpy(cent).to(DEV))
    assert gpu.cpu().numpy().tolist() == [0]
    cent5 = g.standard_normal((5, D)).astype(np.float32)
    gpu, fb = mog.kmeans_assign(bf(X), torch.from_numpy(cent5).to(DEV))
    assert np.array_equal(gpu.cpu().numpy(), ora.assign(X, cent5.astype(np.float64)))


def test_l2_segmented_assign_bit_exact():
    w = wl.WORKLOADS["tiny-4k"]
    K, V, _ = wl.make_unit(w)
    b = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    perm, off, L = b["perm"], b["sub_off"], w.n_sub
    rows, seg, cents = [], [0], []
    for c in range(w.n_clusters):
        mem = np.sort(perm[off[c * L]:off[(c + 1) * L]])
        if mem.size == 0:
            continue
        _, _, st, hist = ora.lloyd(K, L, 4, rows=mem, history=True)
        for t in range(st):
            rows.append(mem)
            seg.append(seg[-1] + mem.size)
            cents.append(hist[t].astype(np.float32))
    rows = np.concatenate(rows).astype(np.int32)
    cents = np.stack(cents)
    gpu = mog.kmeans_assign_segments(bf(K), torch.from_numpy(rows).to(DEV),
                                     torch.tensor(seg, dtype=torch.int32, device=DEV),
                                     torch.from_numpy(cents).to(DEV)).cpu().numpy()
    for s in range(len(seg) - 1):
        ref = ora.assign(K, cents[s].astype(np.float64), rows=rows[seg[s]:seg[s + 1]])
        assert np.array_equal(gpu[seg[s]:seg[s + 1]], ref), s


# ---------------------------------------------------------------- injected partitions

class Injected:
    """A batch whose (cluster, subcluster) partition is given: the oracle's own build of
    each unit (small cases) or a rule applied to positions (large cases)."""

    def __init__(self, w, lens=None, mode="oracle", n_cap=None, union_exact=0, sliding=0,
                 group_select=0, score_mode=0, residual=1, bf16_summaries=0, fp8_summaries=0):
        self.w = w
        self.score_mode, self.residual = score_mode, residual
        lens = wl.lengths(w) if lens is None else np.asarray(lens, np.int32)
        self.lens = lens
        self.n_cap = int(lens.max()) if n_cap is None else n_cap
        B, Hkv, G = w.batch, w.h_kv, w.group
        self.K = np.zeros((B, Hkv, self.n_cap, D), np.uint16)
        self.V = np.zeros_like(self.K)
        self.q = np.zeros((B, Hkv * G, D), np.uint16)
        self.summ = {}
        self.prm = mog.make_params(B, Hkv, Hkv * G, self.n_cap, n_clusters=w.n_clusters,
                                   n_sub=w.n_sub, top_c=w.top_c, top_s=w.top_s, n_sink=w.n_sink,
                                   n_recent=w.n_recent, union_exact=union_exact, sliding=sliding,
                                   group_select=group_select, score_mode=score_mode,
                                   residual=residual, bf16_summaries=bf16_summaries,
                                   fp8_summaries=fp8_summaries)
        stride = mog.sub_off_stride(self.prm, lens)
        perm_all = np.zeros((B * Hkv, self.n_cap), np.int32)
        off_all = np.zeros((B * Hkv, stride), np.int32)
        for b in range(B):
            n = int(lens[b])
            Cn, L = wl.clusters_for(w, n)
            for h in range(Hkv):
                u = wl.UnitDraw(w, b, h, n)
                u.keys_values(self.K[b, h], self.V[b, h])
                self.q[b, h * G:(h + 1) * G] = u.q
                S, R = w.n_sink, w.n_recent
                if mode == "oracle":
                    s = ora.build_unit(self.K[b, h], self.V[b, h], n, S, R, Cn, L)
                else:   # clusters by planted centre, subclusters by position
                    nm = max(0, n - S - R)
                    pos = np.arange(S, S + nm)
                    lab = (u.z[pos] % Cn) * L + (pos % L)
                    order = np.argsort(lab, kind="stable")
                    perm = pos[order].astype(np.int32)
                    sub_off = np.searchsorted(lab[order], np.arange(Cn * L + 1)).astype(np.int32)
                    s = ora.stats(self.K[b, h], self.V[b, h], perm, sub_off, Cn, L)
                    s.update(perm=perm, sub_off=sub_off, C=Cn, L=L, n_build=n, S=S, R=R)
                self.summ[(b, h)] = s
                perm_all[b * Hkv + h, :s["perm"].size] = s["perm"]
                off_all[b * Hkv + h, :Cn * L + 1] = s["sub_off"]
        self.h = mog.build(bf(self.K), bf(self.V), lens, self.prm,
                           partition=(torch.from_numpy(perm_all).to(DEV),
                                      torch.from_numpy(off_all).to(DEV)))
        self.qd = bf(self.q)

    def gpu_summaries(self):
        lay = self.h.layout()
        U, cm, lm = lay.units, lay.c_max, lay.l_max
        return dict(
            cl_n=self.h.array("cl_n", torch.int32, (U, cm)).cpu().numpy(),
            cl_ms=self.h.array("cl_ms", torch.float32, (U, cm, 2, D)).cpu().numpy(),
            cl_vbar=self.h.array("cl_vbar", torch.float32, (U, cm, D)).cpu().numpy(),
            sub_n=self.h.array("sub_n", torch.int32, (U, cm * lm)).cpu().numpy(),
            sub_ms=self.h.array("sub_ms", torch.float32, (U, cm * lm, 2, D)).cpu().numpy(),
            sub_vbar=self.h.array("sub_vbar", torch.float32, (U, cm * lm, D)).cpu().numpy())


def _check_stats(inj):
    g = inj.gpu_summaries()
    worst = 0.0
    for (b, h), s in inj.summ.items():
        u = b * inj.w.h_kv + h
        Cn, L = s["C"], s["L"]
        assert np.array_equal(g["cl_n"][u, :Cn], s["cl_n"])
        assert np.array_equal(g["sub_n"][u, :Cn * L], s["sub_n"])
        for name, gpu, ref, n in (("mu", g["cl_ms"][u, :Cn, 0], s["cl_mu"], s["cl_n"]),
                                  ("var", g["cl_ms"][u, :Cn, 1], s["cl_var"], s["cl_n"]),
                                  ("vbar", g["cl_vbar"][u, :Cn], s["cl_vbar"], s["cl_n"]),
                                  ("smu", g["sub_ms"][u, :Cn * L, 0], s["sub_mu"], s["sub_n"]),
                                  ("svar", g["sub_ms"][u, :Cn * L, 1], s["sub_var"], s["sub_n"]),
                                  ("svbar", g["sub_vbar"][u, :Cn * L], s["sub_vbar"], s["sub_n"])):
            idx = np.nonzero(n > 0)[0]
            if idx.size == 0:
                continue
            nr = np.linalg.norm(ref[idx], axis=1)
            diff = np.linalg.norm(gpu[idx] - ref[idx], axis=1)
            err = np.where(nr > 0, diff / np.where(nr > 0, nr, 1.0), np.abs(gpu[idx]).max(axis=1))
            worst = max(worst, float(err.max()))
            bad = np.nonzero(err > STAT_TOL)[0]
            assert bad.size == 0, (name, u, idx[bad[:5]], err[bad[:5]])
    return worst


def _selection_vs_oracle(inj, heads=None):
    """The GPU's own selection against the oracle's, head by head (differences only at
    near-ties).  Returns (the oracle's selections [U*G][SW], near-tie count)."""
    w, G = inj.w, inj.w.group
    SW = w.top_c + w.top_c * w.top_s
    U = w.batch * w.h_kv
    sel_out = torch.full((U * G, max(SW, 1)), -7, dtype=torch.int32, device=DEV)
    inj.h.decode(inj.qd, sel_out=sel_out)
    gsel = sel_out.cpu().numpy()
    ties = 0
    sel_ref = np.full((U * G, max(SW, 1)), -1, np.int32)
    heads = range(U * G) if heads is None else heads
    for hq in heads:
        u, g = hq // G, hq % G
        b, h = u // w.h_kv, u % w.h_kv
        s = inj.summ[(b, h)]
        sc, ss, cs, sscore = ora.select(inj.q[b, h * G + g], s, w.top_c, w.top_s,
                                        getattr(inj, "score_mode", 0))
        sel_ref[hq, :w.top_c] = sc
        sel_ref[hq, w.top_c:SW] = ss.reshape(-1)
        gc = gsel[hq, :w.top_c]
        if not np.array_equal(gc, sc):
            cut = cs[sc[sc >= 0]].min() if (sc >= 0).any() else -np.inf
            for c in set(gc.tolist()) ^ set(sc.tolist()):
                assert c >= 0 and abs(cs[c] - cut) < TIE, ("cluster selection", hq, c)
            ties += 1
            continue
        gs = gsel[hq, w.top_c:SW].reshape(w.top_c, w.top_s)
        for i in range(w.top_c):
            if not np.array_equal(gs[i], ss[i]):
                cut = sscore[i][ss[i][ss[i] >= 0]].min()
                for l in set(gs[i].tolist()) ^ set(ss[i].tolist()):
                    assert l >= 0 and abs(sscore[i][l] - cut) < TIE, ("sub selection", hq, i, l)
                ties += 1
    return sel_ref, ties


def _check_decode(inj, n_now=None, sample_heads=None):
    w, G = inj.w, inj.w.group
    SW = w.top_c + w.top_c * w.top_s
    U = w.batch * w.h_kv
    heads = range(U * G) if sample_heads is None else sample_heads
    sel_ref, ties = _selection_vs_oracle(inj, heads)
    # outputs under the oracle's selection
    sin = torch.from_numpy(sel_ref).to(DEV)
    out = inj.h.decode(inj.qd, sel_in=sin).cpu().numpy().reshape(U * G, D)
    worst = 0.0
    for hq in heads:
        u, g = hq // G, hq % G
        b, h = u // w.h_kv, u % w.h_kv
        s = inj.summ[(b, h)]
        nn = int(inj.lens[b]) if n_now is None else n_now[b]
        ref, _ = ora.decode(inj.K[b, h], inj.V[b, h], nn, inj.q[b, h * G + g], s,
                            sel_ref[hq, :w.top_c], sel_ref[hq, w.top_c:SW].reshape(w.top_c, w.top_s),
                            residual=bool(getattr(inj, "residual", 1)))
        e = rel(out[hq], ref)
        worst = max(worst, e)
        assert e <= OUT_TOL, (hq, e)
    assert inj.h.sync_status() == 0
    return ties, worst


def test_stats_and_decode_tiny_oracle_partition():
    inj = Injected(wl.WORKLOADS["tiny-4k"])
    print("stats worst", _check_stats(inj), "decode", _check_decode(inj))


def test_stats_and_decode_gqa_ragged():
    w = small_workload(0, batch=2, h_kv=2, h_q=8, centres=48, n_clusters=0, n_sub=0, top_c=3,
                       top_s=2, n_recent=40, n_range=(2500, 3100), seed=21)
    inj = Injected(w)
    assert len(set(inj.lens.tolist())) == 2
    _check_stats(inj)
    _check_decode(inj)


@pytest.mark.parametrize("tc,ts", [(0, 0), (16, 0), (16, 6), (1, 1), (5, 6)])
def test_decode_selection_extremes(tc, ts):
    w = small_workload(3000, h_kv=2, h_q=10, top_c=tc, top_s=ts, seed=31)
    inj = Injected(w)
    _check_decode(inj)


@pytest.mark.parametrize("tc,ts", [(4, 3), (16, 6), (0, 0)])
def test_decode_top_only_matches_oracle(tc, ts):
    """residual = 0 (the top-clusters-only ablation of the residual): the anchors and the
    chosen subclusters' rows alone, against the oracle's decode without residual terms."""
    w = small_workload(3000, h_kv=2, h_q=8, top_c=tc, top_s=ts, seed=33)
    inj = Injected(w, residual=0)
    print("top-only decode", _check_decode(inj))


def test_decode_score_mode_1_matches_oracle():
    """score_mode = 1 (groups ranked by tau q.mu alone): the GPU's selection against the
    oracle's selection under the same rule, and the outputs under it."""
    w = small_workload(3000, batch=2, h_kv=2, h_q=8, n_range=(2500, 3000), top_c=5, top_s=3,
                       seed=34, n_clusters=0, n_sub=0)
    inj = Injected(w, score_mode=1)
    ties, worst = _check_decode(inj)
    _check_stats(inj)
    # the rule changes what is chosen on this data
    w0 = small_workload(3000, batch=2, h_kv=2, h_q=8, n_range=(2500, 3000), top_c=5, top_s=3,
                        seed=34, n_clusters=0, n_sub=0)
    sel0 = _selection_vs_oracle(Injected(w0), None)[0]
    sel1 = _selection_vs_oracle(inj, None)[0]
    assert not np.array_equal(sel0, sel1)
    print("score mode 1 decode", ties, worst)


def test_full_size_qwen3_4b_injected_partition():
    """The benchmark's workload (8 KV heads x 32K keys, 181 x 15 groups) with a
    position-rule partition: statistics and the whole decode step against the oracle."""
    w = wl.WORKLOADS["qwen3-4b-32k"]
    inj = Injected(w, mode="rule")
    _check_stats(inj)
    ties, worst = _check_decode(inj)
    print(f"qwen3-4b-32k: {ties} near-tie heads, worst rel-L2 {worst:.2e}")


# ------------------------------------------------------------------ whole pipeline

def _gpu_build(w, lens=None, n_cap=None, **over):
    lens = wl.lengths(w) if lens is None else np.asarray(lens, np.int32)
    K, V, q, _ = wl.make_batch(w, n_cap=n_cap)
    kw = dict(n_clusters=w.n_clusters, n_sub=w.n_sub, top_c=w.top_c, top_s=w.top_s,
              n_sink=w.n_sink, n_recent=w.n_recent)
    kw.update(over)
    prm = mog.make_params(w.batch, w.h_kv, w.h_q, K.shape[2], **kw)
    Kd, Vd = bf(K), bf(V)
    h = mog.build(Kd, Vd, lens, prm)
    return h, K, V, q, lens, Kd, Vd


def _partition(h, u, lens_b, w):
    lay = h.layout()
    info = h.array("unit_info", torch.int32, (lay.units, 8)).cpu().numpy()[u]
    Cn, L, nm, S = info[0], info[1], info[3], info[4]
    perm = h.array("perm", torch.int32, (lay.units, lay.n_cap)).cpu().numpy()[u, :nm]
    off = h.array("sub_off", torch.int32, (lay.units, lay.sub_off_stride)).cpu().numpy()[u, :Cn * L + 1]
    return Cn, L, nm, S, perm, off


def test_build_partition_properties_and_identities():
    w = wl.WORKLOADS["tiny-4k"]
    h, K, V, q, lens, _, _ = _gpu_build(w)
    Cn, L, nm, S, perm, off = _partition(h, 0, lens[0], w)
    assert np.array_equal(np.sort(perm), np.arange(S, S + nm))
    assert off[0] == 0 and off[-1] == nm and np.all(np.diff(off) >= 0)
    for g in range(Cn * L):
        assert np.all(np.diff(perm[off[g]:off[g + 1]]) > 0)
    g = Injected.gpu_summaries(type("X", (), {"h": h})())
    X = wl.from_bf16(K[0, 0]).astype(np.float64)
    for c in range(Cn):
        sl = slice(c * L, (c + 1) * L)
        ns = g["sub_n"][0, sl].astype(np.float64)
        assert g["cl_n"][0, c] == ns.sum() == off[(c + 1) * L] - off[c * L]
        if ns.sum() == 0:
            continue
        mem = perm[off[c * L]:off[(c + 1) * L]]
        np.testing.assert_allclose(g["cl_ms"][0, c, 0], X[mem].mean(0), rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(g["cl_ms"][0, c, 1], X[mem].var(0), rtol=1e-4, atol=1e-5)
        within = (ns[:, None] * g["sub_ms"][0, sl, 1]).sum(0) / ns.sum()
        between = (ns[:, None] * (g["sub_ms"][0, sl, 0] - g["cl_ms"][0, c, 0]) ** 2).sum(0) / ns.sum()
        np.testing.assert_allclose(g["cl_ms"][0, c, 1], within + between, rtol=1e-4, atol=1e-5)


def test_full_pipeline_approximation_error_close_to_oracle():
    w = wl.WORKLOADS["tiny-4k"]
    h, K, V, q, lens, _, _ = _gpu_build(w)
    out = h.decode(bf(q)).cpu().numpy()[0, 0]
    ref = ora.dense(K[0, 0], V[0, 0], w.n, q[0, 0])
    ob = ora.build_unit(K[0, 0], V[0, 0], w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    om, _, _, _ = ora.mog_head(K[0, 0], V[0, 0], w.n, q[0, 0], ob, w.top_c, w.top_s)
    top, _, _, _ = ora.mog_head(K[0, 0], V[0, 0], w.n, q[0, 0], ob, w.top_c, w.top_s, residual=False)
    e_gpu, e_ora, e_top = rel(out, ref), rel(om, ref), rel(top, ref)
    print(f"MoG vs dense: gpu {e_gpu:.3e} oracle {e_ora:.3e} (top-only {e_top:.3e})")
    assert e_gpu < max(1.5 * e_ora, e_ora + 0.01)


@pytest.mark.parametrize("name", ["tiny-4k", "qwen3-4b-32k"])
def test_all_groups_selected_equals_dense(name):
    w = wl.WORKLOADS[name]
    h, K, V, q, lens, Kd, Vd = _gpu_build(w, top_c=w.n_clusters, top_s=w.n_sub)
    out = h.decode(bf(q)).cpu().numpy()
    G = w.group
    for hq in range(0, w.h_q, max(1, w.h_q // 8)):
        ref = ora.dense(K[0, hq // G], V[0, hq // G], w.n, q[0, hq])
        assert rel(out[0, hq], ref) < OUT_TOL, hq
    assert h.sync_status() == 0


def test_append_joins_recent_anchors():
    w = small_workload(3000, h_kv=2, h_q=8, seed=41)
    steps = 5
    h, K, V, q, lens, Kd, Vd = _gpu_build(w, n_cap=3000 + steps, top_c=w.n_clusters, top_s=w.n_sub)
    rng = np.random.default_rng(3)
    for t in range(steps):
        kn = wl.to_bf16(rng.standard_normal((1, 2, D)))
        vn = wl.to_bf16(rng.standard_normal((1, 2, D)))
        h.append(bf(kn), bf(vn))
        K[0, :, 3000 + t] = kn[0]
        V[0, :, 3000 + t] = vn[0]
    out = h.decode(bf(q)).cpu().numpy()
    assert np.array_equal(Kd.view(torch.int16).cpu().numpy().view(np.uint16), K)
    for hq in range(8):
        ref = ora.dense(K[0, hq // 4], V[0, hq // 4], 3000 + steps, q[0, hq])
        assert rel(out[0, hq], ref) < OUT_TOL
    with pytest.raises(mog.MogError, match="CAPACITY"):
        h.append(bf(kn), bf(vn))


def test_many_units_many_slots_per_split():
    """256 KV heads with up to 24 selected clusters each: four rows-kernel CTAs per unit
    over several waves, each streaming many union slots and residual terms."""
    w = small_workload(1200, batch=16, h_kv=16, h_q=16, centres=24, n_clusters=36, n_sub=4,
                       top_c=24, top_s=2, n_recent=16, seed=51)
    inj = Injected(w)
    assert inj.h.splits() == 4
    _check_decode(inj, sample_heads=range(0, 256, 7))


def _check_decode_union(inj):
    """Union-exact mode: each head's own selection (checked against the oracle), then
    every head of a KV group attends the union of the group's chosen subclusters."""
    w, G = inj.w, inj.w.group
    tc, ts, SW = w.top_c, w.top_s, w.top_c + w.top_c * w.top_s
    U = w.batch * w.h_kv
    sel_ref, ties = _selection_vs_oracle(inj)
    out = inj.h.decode(inj.qd, sel_in=torch.from_numpy(sel_ref).to(DEV)).cpu().numpy().reshape(U * G, D)
    worst, grew = 0.0, 0
    for u in range(U):
        b, h = u // w.h_kv, u % w.h_kv
        s = inj.summ[(b, h)]
        sels = [(sel_ref[u * G + g, :tc], sel_ref[u * G + g, tc:SW].reshape(tc, ts)) for g in range(G)]
        uc, us = ora.union_selection(sels, s["L"])
        for g in range(G):
            ref, diag = ora.decode(inj.K[b, h], inj.V[b, h], int(inj.lens[b]), inj.q[b, h * G + g], s, uc, us)
            own = ora.decode(inj.K[b, h], inj.V[b, h], int(inj.lens[b]), inj.q[b, h * G + g], s, *sels[g])[1]
            grew += diag[2] > own[2]
            e = rel(out[u * G + g], ref)
            worst = max(worst, e)
            assert e <= OUT_TOL, (u, g, e)
    assert grew > 0   # the union adds rows for some heads: the mode is exercised
    assert inj.h.sync_status() == 0
    return ties, worst


def test_union_exact_gqa_matches_oracle():
    w = small_workload(2500, h_kv=2, h_q=8, top_c=5, top_s=3, seed=71)
    inj = Injected(w, union_exact=1)
    print("union-exact decode", _check_decode_union(inj))


def test_union_exact_sixteen_heads_many_units():
    w = small_workload(1500, batch=3, h_kv=2, h_q=32, centres=40, n_clusters=30, n_sub=6,
                       top_c=6, top_s=2, n_recent=32, seed=72)
    inj = Injected(w, union_exact=1)
    print("union-exact decode", _check_decode_union(inj))


def _slide_steps(inj, n0, steps, seed):
    """Append `steps` random tokens to a sliding-window handle; after each, check that the
    key that moved into every KV head's clusters went to the exact argmin under the GPU's
    own means, and replay the move in the oracle."""
    w = inj.w
    rng = np.random.default_rng(seed)
    L, U = w.n_sub, w.batch * w.h_kv
    for t in range(steps):
        before = inj.gpu_summaries()
        kn = wl.to_bf16(rng.standard_normal((w.batch, w.h_kv, D)))
        vn = wl.to_bf16(rng.standard_normal((w.batch, w.h_kv, D)))
        inj.h.append(bf(kn), bf(vn))
        inj.K[:, :, n0 + t], inj.V[:, :, n0 + t] = kn, vn
        after = inj.gpu_summaries()
        for u in range(U):
            b, h = u // w.h_kv, u % w.h_kv
            s = inj.summ[(b, h)]
            Cn = s["C"]
            moved = np.nonzero(after["sub_n"][u, :Cn * L] != before["sub_n"][u, :Cn * L])[0]
            assert moved.size == 1, (t, u, moved)
            c, l = divmod(int(moved[0]), L)
            p = max(s["S"], s["n_build"] - s["R"])
            x = inj.K[b, h, p:p + 1]
            full = np.nonzero(before["cl_n"][u, :Cn] > 0)[0]
            means = before["cl_ms"][u, full, 0].astype(np.float64)
            assert full[ora.assign(x, means)[0]] == c, (t, u)
            subs = np.nonzero(before["sub_n"][u, c * L:(c + 1) * L] > 0)[0]
            smeans = before["sub_ms"][u, c * L + subs, 0].astype(np.float64)
            assert subs[ora.assign(x, smeans)[0]] == l, (t, u)
            inj.summ[(b, h)], _ = ora.slide(inj.K[b, h], inj.V[b, h], s, force=(c, l))


def _check_partition(inj):
    w, lay = inj.w, inj.h.layout()
    L, U = w.n_sub, w.batch * w.h_kv
    info = inj.h.array("unit_info", torch.int32, (U, 8)).cpu().numpy()
    perm = inj.h.array("perm", torch.int32, (U, lay.n_cap)).cpu().numpy()
    off = inj.h.array("sub_off", torch.int32, (U, lay.sub_off_stride)).cpu().numpy()
    for u in range(U):
        s = inj.summ[(u // w.h_kv, u % w.h_kv)]
        Cn = s["C"]
        assert info[u, 5] == max(s["S"], s["n_build"] - s["R"]) and info[u, 3] == s["perm"].size
        assert np.array_equal(off[u, :Cn * L + 1], s["sub_off"])
        for g in range(Cn * L):
            a, e = s["sub_off"][g], s["sub_off"][g + 1]
            assert np.array_equal(np.sort(perm[u, a:e]), np.sort(s["perm"][a:e])), (u, g)


def test_sliding_window_matches_oracle():
    """Sliding recent window: after each append the oldest recent key of every KV head
    joins a cluster.  The GPU's choice is the exact argmin under its own means at that
    moment; the oracle replays the same moves (Welford in fp64); statistics, partition,
    window and decode then agree."""
    steps, n0 = 40, 3000
    w = small_workload(n0, batch=2, h_kv=2, h_q=8, n_recent=32, seed=81)
    inj = Injected(w, n_cap=n0 + steps, sliding=1)
    _slide_steps(inj, n0, steps, seed=8)
    _check_partition(inj)
    print("sliding: stats worst", _check_stats(inj))
    print("sliding: decode", _check_decode(inj, n_now=[n0 + steps] * w.batch))


def test_sliding_window_large_partition_cluster_of_ctas():
    """A 256 x 20 partition (5120 subclusters): the slide runs as a cluster of several CTAs
    per KV head (slices of the cluster search, batches of the partition update)."""
    steps, n0 = 16, 12000
    w = small_workload(n0, batch=1, h_kv=2, h_q=4, centres=300, n_clusters=256, n_sub=20,
                       top_c=6, top_s=4, n_recent=24, seed=83)
    inj = Injected(w, mode="planted", n_cap=n0 + steps, sliding=1)
    _slide_steps(inj, n0, steps, seed=10)
    _check_partition(inj)
    print("sliding, large partition: stats worst", _check_stats(inj))
    print("sliding, large partition: decode", _check_decode(inj, n_now=[n0 + steps] * w.batch))


def test_sliding_window_union_exact_ragged_batch():
    """Both variants at once on a ragged batch: a 2600-key sequence slides its window into
    the clusters, a 40-key one has no cluster and keeps a growing window; the decode is
    then checked under the union-exact rule."""
    steps = 24
    w = small_workload(2600, batch=2, h_kv=2, h_q=8, n_recent=48, seed=82)
    lens = np.array([2600, 40], np.int32)
    inj = Injected(w, lens=lens, n_cap=2600 + steps, sliding=1, union_exact=1)
    rng = np.random.default_rng(9)
    L, U = w.n_sub, w.batch * w.h_kv
    for t in range(steps):
        before = inj.gpu_summaries()
        kn = wl.to_bf16(rng.standard_normal((w.batch, w.h_kv, D)))
        vn = wl.to_bf16(rng.standard_normal((w.batch, w.h_kv, D)))
        inj.h.append(bf(kn), bf(vn))
        for b in range(w.batch):
            inj.K[b, :, lens[b] + t], inj.V[b, :, lens[b] + t] = kn[b], vn[b]
        after = inj.gpu_summaries()
        for u in range(U):
            b, h = u // w.h_kv, u % w.h_kv
            s = inj.summ[(b, h)]
            Cn = s["C"]
            moved = np.nonzero(after["sub_n"][u, :Cn * L] != before["sub_n"][u, :Cn * L])[0]
            if not (s["cl_n"] > 0).any():
                assert moved.size == 0
                assert ora.slide(inj.K[b, h], inj.V[b, h], s)[1] is None
                continue
            assert moved.size == 1, (t, u, moved)
            c, l = divmod(int(moved[0]), L)
            inj.summ[(b, h)], _ = ora.slide(inj.K[b, h], inj.V[b, h], s, force=(c, l))
    info = inj.h.array("unit_info", torch.int32, (U, 8)).cpu().numpy()
    for u in range(U):
        s = inj.summ[(u // w.h_kv, u % w.h_kv)]
        assert info[u, 5] == max(s["S"], s["n_build"] - s["R"])
    inj.lens = lens + steps
    print("sliding + union-exact: stats", _check_stats(inj), "decode", _check_decode_union(inj))


def _check_decode_group(inj, om64=None):
    """Group-shared selection: the GPU's selection against the oracle's group selection
    (differences only at near-ties), repeated for every head; then every head's output
    under the oracle's group selection (with om64: the oracle's feature-map decode)."""
    w, G = inj.w, inj.w.group
    tc, ts, SW = w.top_c, w.top_s, w.top_c + w.top_c * w.top_s
    U = w.batch * w.h_kv
    sel_out = torch.full((U * G, SW), -7, dtype=torch.int32, device=DEV)
    inj.h.decode(inj.qd, sel_out=sel_out)
    gsel = sel_out.cpu().numpy()
    sel_ref = np.full((U * G, SW), -1, np.int32)
    ties = 0
    for u in range(U):
        b, h = u // w.h_kv, u % w.h_kv
        s = inj.summ[(b, h)]
        sc, ss, gc, gsc = ora.group_selection(inj.q[b, h * G:(h + 1) * G], s, tc, ts)
        for g in range(G):
            sel_ref[u * G + g, :tc] = sc
            sel_ref[u * G + g, tc:] = ss.reshape(-1)
            assert np.array_equal(gsel[u * G + g], gsel[u * G])   # the group's lists, repeated
        if not np.array_equal(gsel[u * G, :tc], sc):
            cut = gc[sc[sc >= 0]].min()
            for c in set(gsel[u * G, :tc].tolist()) ^ set(sc.tolist()):
                assert c >= 0 and abs(gc[c] - cut) < TIE, ("group cluster selection", u, c)
            ties += 1
            continue
        gs = gsel[u * G, tc:].reshape(tc, ts)
        for i in range(tc):
            if sc[i] >= 0 and not np.array_equal(gs[i], ss[i]):
                row = gsc[sc[i]]
                cut = row[ss[i][ss[i] >= 0]].min()
                for l in set(gs[i].tolist()) ^ set(ss[i].tolist()):
                    assert l >= 0 and abs(row[l] - cut) < TIE, ("group sub selection", u, i, l)
                ties += 1
    out = inj.h.decode(inj.qd, sel_in=torch.from_numpy(sel_ref).to(DEV)).cpu().numpy().reshape(U * G, D)
    worst = 0.0
    for u in range(U):
        b, h = u // w.h_kv, u % w.h_kv
        s = inj.summ[(b, h)]
        for g in range(G):
            args = (inj.K[b, h], inj.V[b, h], int(inj.lens[b]), inj.q[b, h * G + g], s,
                    sel_ref[u * G + g, :tc], sel_ref[u * G + g, tc:].reshape(tc, ts))
            ref, _ = ora.decode(*args) if om64 is None else ora.decode_fm(*args, om64)
            e = rel(out[u * G + g], ref)
            worst = max(worst, e)
            assert e <= OUT_TOL, (u, g, e)
    assert inj.h.sync_status() == 0
    return ties, worst


def test_group_shared_selection_matches_oracle():
    w = small_workload(2500, h_kv=2, h_q=8, top_c=5, top_s=3, seed=91)
    inj = Injected(w, group_select=1)
    print("group-shared decode", _check_decode_group(inj))


def test_group_shared_selection_sixteen_heads_ragged():
    w = small_workload(1800, batch=2, h_kv=2, h_q=32, centres=40, n_clusters=30, n_sub=6,
                       top_c=6, top_s=2, n_recent=32, seed=92)
    inj = Injected(w, lens=np.array([1800, 900], np.int32), group_select=1, union_exact=1)
    print("group-shared decode, 16 heads", _check_decode_group(inj))


def test_sixteen_query_heads_per_kv_head():
    w = small_workload(2500, h_kv=1, h_q=16, top_c=5, top_s=3, seed=61)
    inj = Injected(w)
    _check_stats(inj)
    _check_decode(inj)


# ------------------------------------------------- full-size heads of the large workloads

class FromBuild:
    """One KV head of a workload, clustered by the library's own build; the oracle's
    summaries are recomputed from the partition the GPU chose."""

    def __init__(self, name, steps=0):
        import dataclasses
        base = wl.WORKLOADS[name]
        self.unit = wl.UnitDraw(base, 0, 0, base.n)
        self.w = dataclasses.replace(base, batch=1, h_kv=1, h_q=base.group)
        n = base.n
        self.lens = np.array([n], np.int32)
        self.n_cap = n + steps
        K = np.zeros((1, 1, self.n_cap, D), np.uint16)
        V = np.zeros_like(K)
        self.unit.keys_values(K[0, 0], V[0, 0])
        self.K, self.V = K, V
        self.q = self.unit.q[None].copy()
        prm = mog.make_params(1, 1, base.group, self.n_cap, n_clusters=base.n_clusters,
                              n_sub=base.n_sub, top_c=base.top_c, top_s=base.top_s,
                              n_sink=base.n_sink, n_recent=base.n_recent)
        self.Kd, self.Vd = bf(K), bf(V)
        self.h = mog.build(self.Kd, self.Vd, self.lens, prm)
        Cn, L, nm, S, perm, off = _partition(self.h, 0, n, self.w)
        s = ora.stats(K[0, 0], V[0, 0], perm, off, Cn, L)
        s.update(perm=perm, sub_off=off, C=Cn, L=L, n_build=n, S=S, R=base.n_recent)
        self.summ = {(0, 0): s}
        self.qd = bf(self.q)

    gpu_summaries = Injected.gpu_summaries


def test_full_size_1m_head_build_and_decode():
    """A 1M-key KV head of the 1M workload (1024 x 20 groups, top 16 x 8, 4 query heads):
    the GPU's own two-level clustering, its statistics against the oracle's on that
    partition, the selection and the decode step."""
    fb = FromBuild("ctx-1m")
    Cn, L, nm, S, perm, off = _partition(fb.h, 0, fb.lens[0], fb.w)
    assert np.array_equal(np.sort(perm), np.arange(S, S + nm))
    worst_s = _check_stats(fb)
    ties, worst = _check_decode(fb)
    print(f"1M head: stats worst {worst_s:.2e}, {ties} near-tie heads, decode worst {worst:.2e}")


class FromBuildBatch:
    """A whole workload batch clustered by the library's own build (automatic C and L per
    sequence); the oracle's summaries of every unit are recomputed from the partition the
    GPU chose."""

    def __init__(self, name):
        self.w = w = wl.WORKLOADS[name]
        K, V, q, lens = wl.make_batch(w, n_cap=int(wl.lengths(w).max()))
        self.K, self.V, self.q, self.lens = K, V, q, lens
        prm = mog.make_params(w.batch, w.h_kv, w.h_q, K.shape[2], n_clusters=w.n_clusters,
                              n_sub=w.n_sub, top_c=w.top_c, top_s=w.top_s, n_sink=w.n_sink,
                              n_recent=w.n_recent)
        self.h = mog.build(bf(K), bf(V), lens, prm)
        self.summ = {}
        for u in range(w.batch * w.h_kv):
            b, h = divmod(u, w.h_kv)
            Cn, L, nm, S, perm, off = _partition(self.h, u, lens[b], w)
            assert (Cn, L) == wl.clusters_for(w, int(lens[b]))
            assert np.array_equal(np.sort(perm), np.arange(S, S + nm))
            s = ora.stats(K[b, h], V[b, h], perm, off, Cn, L)
            s.update(perm=perm, sub_off=off, C=Cn, L=L, n_build=int(lens[b]), S=S, R=w.n_recent)
            self.summ[(b, h)] = s
        self.qd = bf(q)

    gpu_summaries = Injected.gpu_summaries


def test_full_size_olmo3_7b_varlen_build_and_decode():
    """The Olmo-3-7B-shaped batch at full size: 8 sequences x 32 MHA heads, N_b from
    U[16384, 65536], round(sqrt N_b) clusters x ceil(log2 N_b) subclusters per sequence.
    The GPU's own build of all 256 heads; every head's statistics against the oracle's on
    that partition; selection and decode on four heads of every sequence."""
    fb = FromBuildBatch("olmo3-7b-varlen")
    assert len(set(fb.lens.tolist())) == fb.w.batch
    worst_s = _check_stats(fb)
    heads = [b * fb.w.h_q + h for b in range(fb.w.batch) for h in (0, 9, 18, 27)]
    ties, worst = _check_decode(fb, sample_heads=heads)
    print(f"olmo3 varlen: lengths {fb.lens.tolist()}, stats worst {worst_s:.2e}, "
          f"{ties} near-tie heads, decode worst {worst:.2e}")


def test_append_64_steps_qwen3_14b_head():
    """The Qwen3-14B-shaped head (131072 keys, 362 x 17 groups, top 12 x 8, 5 query heads)
    over 64 decode steps that each append one key and value: appended keys join the
    recent anchors and every 16th step is checked against the oracle."""
    steps = 64
    fb = FromBuild("qwen3-14b-128k", steps=steps)
    n = int(fb.lens[0])
    worst = 0.0
    for t in range(1, steps + 1):
        kn, vn, qt = fb.unit.step(t)
        fb.h.append(bf(kn[None, None]), bf(vn[None, None]))
        fb.K[0, 0, n + t - 1] = kn
        fb.V[0, 0, n + t - 1] = vn
        fb.q = qt[None]
        fb.qd = bf(fb.q)
        if t % 16 == 0:
            _, w_t = _check_decode(fb, n_now=[n + t])
            worst = max(worst, w_t)
    assert np.array_equal(fb.Kd.view(torch.int16).cpu().numpy().view(np.uint16), fb.K)
    print(f"64 appending steps: decode worst {worst:.2e}")


# ------------------------------------------------------------------- failure paths

def test_bounded_wait_gives_up_and_the_context_survives():
    """The mbarrier wait of the tensor-core build gives up after its poll limit, records
    MOG_ERR_TIMEOUT and returns; the next kernels run normally."""
    scratch = torch.zeros(4, dtype=torch.int32, device=DEV)
    assert mog.check_bounded_wait(2000, True, scratch) == 0
    assert mog.check_bounded_wait(2000, False, scratch) == 6       # MOG_ERR_TIMEOUT
    assert mog.check_bounded_wait(2000, True, scratch) == 0
    w = small_workload(700, seed=13)
    K, V, q = wl.make_unit(w)
    ld = torch.tensor([700], dtype=torch.int32, device=DEV)
    out = mog.dense_decode(bf(K)[None, None], bf(V)[None, None], ld, 700, bf(q)[None]).cpu().numpy()
    assert rel(out[0, 0], ora.dense(K, V, 700, q[0])) < OUT_TOL


def _corrupt_build(mutate):
    """mog_build_from_partition on the oracle's partition of a small head after
    `mutate(perm, sub_off, S, nm)` edits it in place; returns the device status code."""
    w = small_workload(1500, seed=14)
    K, V, q = wl.make_unit(w)
    s = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    prm = mog.make_params(1, 1, 1, w.n, n_clusters=w.n_clusters, n_sub=w.n_sub, top_c=w.top_c,
                          top_s=w.top_s, n_sink=w.n_sink, n_recent=w.n_recent)
    stride = mog.sub_off_stride(prm, [w.n])
    perm = np.zeros((1, w.n), np.int32)
    off = np.zeros((1, stride), np.int32)
    nm = s["perm"].size
    perm[0, :nm] = s["perm"]
    off[0, :s["sub_off"].size] = s["sub_off"]
    mutate(perm[0], off[0], w.n_sink, nm)
    h = mog.build(bf(K)[None, None], bf(V)[None, None], [w.n], prm,
                  partition=(torch.from_numpy(perm).to(DEV), torch.from_numpy(off).to(DEV)))
    return h.sync_status()


def test_corrupt_partition_is_reported():
    """A partition whose positions leave the mid region, or whose offsets run backwards,
    is caught on the device: the status word reads MOG_ERR_DEVICE_CHECK and the summaries
    are not computed from it."""
    assert _corrupt_build(lambda p, o, S, nm: None) == 0
    def bad_position(p, o, S, nm):
        p[nm // 2] = S + nm + 3
    def backwards(p, o, S, nm):
        o[5], o[6] = o[6] + 1, o[5]
    def short_total(p, o, S, nm):
        o[16 * 6] = nm - 1
    for mutate in (bad_position, backwards, short_total):
        assert _corrupt_build(mutate) == 5, mutate.__name__      # MOG_ERR_DEVICE_CHECK


# ------------------------------------------------------------ bf16 summaries (variant)

def _bf16_bits_to_f64(a):
    return (np.asarray(a).astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_bf16_copies(inj):
    """The GPU's bf16 copies of the key means and variances (and the value means' high
    parts) against the oracle's rounding of its own statistics: equal, except one bf16 ulp
    where the fp32 value sits on a rounding tie (the GPU's and the oracle's fp32 values may
    differ in their last bits)."""
    lay = inj.h.layout()
    U, cm, lm = lay.units, lay.c_max, lay.l_max
    cl16 = _bf16_bits_to_f64(inj.h.array("cl_ms16", torch.int16, (U, cm, 2, D)).cpu().numpy())
    sb16 = _bf16_bits_to_f64(inj.h.array("sub_ms16", torch.int16, (U, cm * lm, 2, D)).cpu().numpy())
    total, off_by_one = 0, 0
    for (b, h), s in inj.summ.items():
        u = b * inj.w.h_kv + h
        Cn, L = s["C"], s["L"]
        for gpu, ref, n in ((cl16[u, :Cn, 0], s["cl_mu"], s["cl_n"]), (cl16[u, :Cn, 1], s["cl_var"], s["cl_n"]),
                            (sb16[u, :Cn * L, 0], s["sub_mu"], s["sub_n"]),
                            (sb16[u, :Cn * L, 1], s["sub_var"], s["sub_n"])):
            keep = n > 0
            g, r = gpu[keep], ora.bf16_round(ref[keep])
            total += g.size
            bad = g != r
            if bad.any():
                ulp = np.abs(r[bad]) * 2.0 ** -7
                assert np.all(np.abs(g[bad] - r[bad]) <= ulp * 1.0001), "more than one bf16 ulp"
                f32 = ref[keep][bad].astype(np.float32).astype(np.float64)
                mid = (g[bad] + r[bad]) / 2
                assert np.all(np.abs(f32 - mid) <= np.abs(mid) * 2.0 ** -20), "not at a rounding tie"
                off_by_one += int(bad.sum())
    assert off_by_one <= max(2, total // 10000), (off_by_one, total)
    return total, off_by_one


def test_bf16_summaries_match_oracle():
    """MOG_FLAG_BF16_SUMMARIES on the oracle's partition: the fp32 summaries as usual, their
    bf16 copies against the oracle's rounding, then the selection and the decode against the
    oracle on the rounded summaries."""
    w = small_workload(3000, batch=2, h_kv=2, h_q=8, top_c=5, top_s=3, seed=35)
    inj = Injected(w, bf16_summaries=1)
    _check_stats(inj)
    total, ob1 = _check_bf16_copies(inj)
    inj.summ = {k: ora.summaries_bf16(s) for k, s in inj.summ.items()}
    ties, worst = _check_decode(inj)
    print(f"bf16 summaries: {total} values, {ob1} one ulp off at ties; {ties} near-tie heads, "
          f"decode worst {worst:.2e}")


def test_bf16_summaries_full_size_qwen3_4b():
    """The 32K workload at full size with bf16 summaries (position-rule partition)."""
    w = wl.WORKLOADS["qwen3-4b-32k"]
    inj = Injected(w, mode="rule", bf16_summaries=1)
    _check_bf16_copies(inj)
    inj.summ = {k: ora.summaries_bf16(s) for k, s in inj.summ.items()}
    print("bf16 summaries 32K", _check_decode(inj))


def test_bf16_summaries_follow_the_sliding_window():
    """With the sliding window the Welford updates keep the bf16 copies equal to the
    rounding of the updated fp32 summaries."""
    steps, n0 = 12, 3000
    w = small_workload(n0, batch=1, h_kv=2, h_q=4, n_recent=32, seed=84)
    inj = Injected(w, n_cap=n0 + steps, sliding=1, bf16_summaries=1)
    _slide_steps(inj, n0, steps, seed=12)
    lay = inj.h.layout()
    U, cm, lm = lay.units, lay.c_max, lay.l_max
    g = inj.gpu_summaries()
    cl16 = _bf16_bits_to_f64(inj.h.array("cl_ms16", torch.int16, (U, cm, 2, D)).cpu().numpy())
    sb16 = _bf16_bits_to_f64(inj.h.array("sub_ms16", torch.int16, (U, cm * lm, 2, D)).cpu().numpy())
    as_bf = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(cl16, as_bf(g["cl_ms"]))
    assert np.array_equal(sb16, as_bf(g["sub_ms"]))
    inj.summ = {k: ora.summaries_bf16(s) for k, s in inj.summ.items()}
    print("bf16 + sliding decode", _check_decode(inj, n_now=[n0 + steps] * w.batch))


# ------------------------------------------------------------- fp8 summaries (variant)

def _e4m3_bits_to_f64(a):
    """fp8 e4m3 bytes -> their values, decoded from the format's fields (sign, 4 exponent
    bits with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals)."""
    a = np.asarray(a).astype(np.uint8).astype(np.int64)
    sgn = np.where(a & 0x80, -1.0, 1.0)
    e, m = (a >> 3) & 0xF, a & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e - 7))
    return sgn * mag


def _fp8_arrays(inj):
    lay = inj.h.layout()
    U, cm, lm = lay.units, lay.c_max, lay.l_max
    cl8 = _e4m3_bits_to_f64(inj.h.array("cl_ms8", torch.uint8, (U, cm, 2, D)).cpu().numpy())
    sb8 = _e4m3_bits_to_f64(inj.h.array("sub_ms8", torch.uint8, (U, cm * lm, 2, D)).cpu().numpy())
    return cl8, sb8


def _check_fp8_copies(inj):
    """The GPU's e4m3 copies of the key means and variances against the oracle's rounding of
    its own statistics: equal, except where the fp32 value sits on a rounding tie of e4m3
    (the GPU's and the oracle's fp32 statistics may differ in their last bits); there the
    GPU holds one of the tie's two neighbours."""
    cl8, sb8 = _fp8_arrays(inj)
    total, off_by_one = 0, 0
    for (b, h), s in inj.summ.items():
        u = b * inj.w.h_kv + h
        Cn, L = s["C"], s["L"]
        for gpu, ref, n in ((cl8[u, :Cn, 0], s["cl_mu"], s["cl_n"]), (cl8[u, :Cn, 1], s["cl_var"], s["cl_n"]),
                            (sb8[u, :Cn * L, 0], s["sub_mu"], s["sub_n"]),
                            (sb8[u, :Cn * L, 1], s["sub_var"], s["sub_n"])):
            keep = n > 0
            g, r = gpu[keep], ora.fp8_round(ref[keep])
            total += g.size
            bad = g != r
            if bad.any():
                mid = (g[bad] + r[bad]) / 2
                f32 = ref[keep][bad].astype(np.float32).astype(np.float64)
                assert np.all(np.abs(f32 - mid) <= np.abs(mid) * 2.0 ** -18), "not at a rounding tie"
                lo, hi = ora.fp8_round(mid * (1 - 2.0 ** -10)), ora.fp8_round(mid * (1 + 2.0 ** -10))
                assert np.all(((g[bad] == lo) & (r[bad] == hi)) | ((g[bad] == hi) & (r[bad] == lo))), \
                    "not the tie's neighbours"
                off_by_one += int(bad.sum())
    assert total > 0 and off_by_one <= max(2, total // 10000), (off_by_one, total)
    return total, off_by_one


def test_fp8_summaries_match_oracle():
    """MOG_FLAG_FP8_SUMMARIES on the oracle's partition: the fp32 summaries as usual, their
    e4m3 copies against the oracle's rounding, then the selection and the decode (whose
    residual terms read the rounded value means) against the oracle on the rounded
    summaries."""
    w = small_workload(3000, batch=2, h_kv=2, h_q=8, top_c=5, top_s=3, seed=36)
    inj = Injected(w, fp8_summaries=1)
    _check_stats(inj)
    total, ob1 = _check_fp8_copies(inj)
    lay = inj.h.layout()
    assert lay.cl_ms16 == 0 and lay.sub_ms16 == 0
    inj.summ = {k: ora.summaries_fp8(s) for k, s in inj.summ.items()}
    ties, worst = _check_decode(inj)
    print(f"fp8 summaries: {total} values, {ob1} off at ties; {ties} near-tie heads, decode worst {worst:.2e}")


def test_fp8_summaries_full_size_qwen3_4b():
    """The 32K workload at full size with fp8 summaries (position-rule partition)."""
    w = wl.WORKLOADS["qwen3-4b-32k"]
    inj = Injected(w, mode="rule", fp8_summaries=1)
    _check_fp8_copies(inj)
    inj.summ = {k: ora.summaries_fp8(s) for k, s in inj.summ.items()}
    print("fp8 summaries 32K", _check_decode(inj))


def test_fp8_summaries_follow_the_sliding_window():
    """With the sliding window the Welford updates keep the e4m3 copies equal to the
    rounding of the updated fp32 summaries (torch's e4m3 conversion, nearest-even)."""
    steps, n0 = 12, 3000
    w = small_workload(n0, batch=1, h_kv=2, h_q=4, n_recent=32, seed=85)
    inj = Injected(w, n_cap=n0 + steps, sliding=1, fp8_summaries=1)
    _slide_steps(inj, n0, steps, seed=13)
    g = inj.gpu_summaries()
    cl8, sb8 = _fp8_arrays(inj)
    as_f8 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(cl8, as_f8(np.clip(g["cl_ms"], -448, 448)))
    assert np.array_equal(sb8, as_f8(np.clip(g["sub_ms"], -448, 448)))
    inj.summ = {k: ora.summaries_fp8(s) for k, s in inj.summ.items()}
    print("fp8 + sliding decode", _check_decode(inj, n_now=[n0 + steps] * w.batch))


# ------------------------------------------------------------ k-means++ seeding (variant)

def test_kmeanspp_ragged_batch_paged_and_bad_draws():
    """k-means++ seeding over a ragged batch (units of different lengths and numbers of
    clusters): every unit's seeds equal the oracle's with that unit's draws; a paged copy
    of the cache gives the same seeds and partition bit for bit; a draw outside [0, 1) is
    reported by the status word."""
    w = small_workload(0, batch=2, h_kv=2, h_q=8, centres=48, n_clusters=0, n_sub=0, top_c=3,
                       top_s=2, n_recent=40, n_range=(2500, 3100), seed=22)
    K, V, q, lens = wl.make_batch(w)
    n_cap = K.shape[2]
    prm = mog.make_params(2, 2, 8, n_cap, top_c=3, top_s=2, n_sink=4, n_recent=40, kmeanspp=1)
    tl = mog.trace_layout(prm, lens)
    draws = wl.seed_draws(tl.units, tl.c_max, 23)
    h = mog.build(bf(K), bf(V), lens, prm, draws=draws)
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    lay = h.layout()
    U = lay.units
    pp = h.array("pp_idx", torch.int32, (U, lay.c_max)).cpu().numpy()
    info = h.array("unit_info", torch.int32, (U, 8)).cpu().numpy()
    assert len(set(info[:, 0].tolist())) == 2          # two numbers of clusters
    for u in range(U):
        b, hh = divmod(u, 2)
        Cn, nm, S = int(info[u, 0]), int(info[u, 3]), int(info[u, 4])
        ref = ora.kmeanspp(K[b, hh, S:S + nm], Cn, draws[u])
        assert np.array_equal(pp[u, :Cn], ref), u
    pk, _ = _paged_copy(K, V, 64, True, seed=24)
    hp = mog.build(pk, None, lens, prm, draws=draws)
    torch.cuda.synchronize()
    assert hp.sync_status() == 0
    ppp = hp.array("pp_idx", torch.int32, (U, lay.c_max)).cpu().numpy()
    assert np.array_equal(pp, ppp)                      # (entries past a unit's C stay -1)
    assert all(np.all(pp[u, info[u, 0]:] == -1) for u in range(U))
    for u in range(U):
        nm, used = int(info[u, 3]), int(info[u, 0] * info[u, 1] + 1)
        for name, width in (("perm", nm), ("sub_off", used)):
            stride = lay.n_cap if name == "perm" else lay.sub_off_stride
            a, c = (x.array(name, torch.int32, (U, stride))[u, :width] for x in (h, hp))
            assert torch.equal(a, c), (name, u)
    bad = draws.copy()
    bad[1, 3] = 1.5
    hb = mog.build(bf(K), bf(V), lens, prm, draws=bad)
    assert hb.sync_status() == 5                        # MOG_ERR_DEVICE_CHECK
    with pytest.raises(ValueError):
        mog.build(bf(K), bf(V), lens, prm)               # the draws are required


# ---------------------------------------------------- feature-map residual (variant)

FM_M = mog.FM_FEATURES


def _omega(seed):
    """The frequencies as the GPU holds them (float32), and as float64 for the oracle."""
    om32 = wl.fm_omega(FM_M, D, seed).astype(np.float32)
    return om32, om32.astype(np.float64)


def _check_fm_sums(inj, om64):
    """The GPU's per-subcluster feature sums (scaled by exp(-(|w_i|^2/2 - 40))) against the
    oracle's unscaled sums, feature row by feature row; and the unit totals against the
    oracle's sums over all subclusters."""
    lay = inj.h.layout()
    U, cm, lm = lay.units, lay.c_max, lay.l_max
    z = inj.h.array("fm_z", torch.float32, (U, cm * lm, FM_M, D + 4)).cpu().numpy().astype(np.float64)
    t = inj.h.array("fm_t", torch.float32, (U, FM_M, D + 4)).cpu().numpy().astype(np.float64)
    mi = 0.5 * np.sum(om64 * om64, axis=1) - 40.0
    scale = np.exp(mi)[None, :, None]
    worst = 0.0
    for (b, h), s in inj.summ.items():
        u = b * inj.w.h_kv + h
        Cn, L = s["C"], s["L"]
        ref = ora.fm_sums(inj.K[b, h], inj.V[b, h], s, om64)           # [C*L, m, d+1]
        gz = z[u, :Cn * L, :, :D + 1] * scale
        for g in range(Cn * L):
            if s["sub_n"][g] == 0:
                assert np.all(gz[g] == 0), g
                continue
            e = np.abs(gz[g] - ref[g]).max(axis=1) / np.abs(ref[g]).max(axis=1)
            worst = max(worst, float(e.max()))
        tot = ref.sum(axis=0)
        e = np.abs(t[u, :, :D + 1] * scale[0] - tot).max(axis=1) / np.abs(tot).max(axis=1)
        worst = max(worst, float(e.max()))
    assert worst < 2e-4, worst
    return worst


def _check_decode_fm(inj, om64, sample_heads=None):
    """Outputs under the oracle's selection against the oracle's decode with the
    feature-map residual."""
    w, G = inj.w, inj.w.group
    SW = w.top_c + w.top_c * w.top_s
    U = w.batch * w.h_kv
    heads = range(U * G) if sample_heads is None else sample_heads
    sel_ref, ties = _selection_vs_oracle(inj, heads)
    out = inj.h.decode(inj.qd, sel_in=torch.from_numpy(sel_ref).to(DEV)).cpu().numpy().reshape(U * G, D)
    worst = 0.0
    for hq in heads:
        u, g = hq // G, hq % G
        b, h = u // w.h_kv, u % w.h_kv
        ref, diag = ora.decode_fm(inj.K[b, h], inj.V[b, h], int(inj.lens[b]), inj.q[b, h * G + g], inj.summ[(b, h)],
                                  sel_ref[hq, :w.top_c], sel_ref[hq, w.top_c:SW].reshape(w.top_c, w.top_s), om64)
        e = rel(out[hq], ref)
        worst = max(worst, e)
        assert e <= OUT_TOL, (hq, e)
    assert inj.h.sync_status() == 0
    return ties, worst


def test_fm_residual_sums_and_decode_match_oracle():
    """residual = 2 on the oracle's partition: every subcluster's feature sums and the unit
    totals against the oracle's, then the decode against the oracle's feature-map decode."""
    w = small_workload(3000, batch=2, h_kv=2, h_q=8, top_c=5, top_s=3, seed=41)
    inj = Injected(w, residual=2)
    om32, om64 = _omega(42)
    with pytest.raises(mog.MogError, match="INVALID_ARG"):
        inj.h.decode(inj.qd)                       # the summary is not built yet
    inj.h.feature_map(om32)
    print("fm sums worst", _check_fm_sums(inj, om64))
    print("fm decode (near-ties, worst)", _check_decode_fm(inj, om64))


def test_fm_residual_with_group_selection():
    """residual = 2 with the group-shared selection: every head subtracts the group's chosen
    subclusters; outputs against the oracle's feature-map decode under the group's
    selection."""
    w = small_workload(2500, batch=2, h_kv=2, h_q=8, top_c=5, top_s=3, seed=48)
    inj = Injected(w, group_select=1, residual=2)
    om32, om64 = _omega(49)
    inj.h.feature_map(om32)
    print("fm + group-shared decode", _check_decode_group(inj, om64))


def test_fm_residual_full_size_qwen3_4b():
    """The 32K workload at full size (position-rule partition): sums and every head."""
    w = wl.WORKLOADS["qwen3-4b-32k"]
    inj = Injected(w, mode="rule", residual=2)
    om32, om64 = _omega(43)
    inj.h.feature_map(om32)
    print("fm sums 32K worst", _check_fm_sums(inj, om64))
    print("fm decode 32K", _check_decode_fm(inj, om64))


def test_fm_residual_paged_recluster_and_misuse():
    """A paged copy gives bit-identical sums and outputs; re-clustering redoes the sums for
    the new partition (equal to a fresh build's); the summary is refused for another
    residual mode."""
    n0, steps = 3000, 8
    w = small_workload(n0, batch=2, h_kv=2, h_q=8, top_c=5, top_s=3, n_recent=32, seed=44)
    K, V, q, lens = wl.make_batch(w, n_cap=n0 + steps)
    prm = mog.make_params(2, 2, 8, n0 + steps, n_clusters=w.n_clusters, n_sub=w.n_sub, top_c=5, top_s=3,
                          n_sink=4, n_recent=32, residual=2)
    om32, _ = _omega(45)
    Kd, Vd, qd = bf(K), bf(V), bf(q)
    hc = mog.build(Kd, Vd, lens, prm)
    hc.feature_map(om32)
    pk, _ = _paged_copy(K, V, 64, False, seed=46)
    hp = mog.build(pk, None, lens, prm)
    hp.feature_map(om32)
    lay = hc.layout()
    U, cm, lm = lay.units, lay.c_max, lay.l_max
    zc = hc.array("fm_z", torch.float32, (U, cm * lm, FM_M, D + 4))[..., :D + 1]
    zp = hp.array("fm_z", torch.float32, (U, cm * lm, FM_M, D + 4))[..., :D + 1]
    assert torch.equal(zc, zp)
    assert torch.equal(hc.decode(qd), hp.decode(qd))
    rng = np.random.default_rng(47)
    for t in range(steps):
        kn = wl.to_bf16(rng.standard_normal((2, 2, D)))
        vn = wl.to_bf16(rng.standard_normal((2, 2, D)))
        hc.append(bf(kn), bf(vn))
        K[:, :, n0 + t], V[:, :, n0 + t] = kn, vn
    hc.recluster()
    fresh = mog.build(Kd, Vd, lens + steps, prm)
    fresh.feature_map(om32)
    torch.cuda.synchronize()
    zr = hc.array("fm_z", torch.float32, (U, cm * lm, FM_M, D + 4))[..., :D + 1]
    zf = fresh.array("fm_z", torch.float32, (U, cm * lm, FM_M, D + 4))[..., :D + 1]
    info = hc.array("unit_info", torch.int32, (U, 8)).cpu().numpy()
    for u in range(U):
        used = int(info[u, 0] * info[u, 1])
        assert torch.equal(zr[u, :used], zf[u, :used]), u
    assert torch.equal(hc.decode(qd), fresh.decode(qd))
    g = mog.build(Kd, Vd, lens, mog.make_params(2, 2, 8, n0 + steps, n_clusters=w.n_clusters, n_sub=w.n_sub,
                                                top_c=5, top_s=3, n_sink=4, n_recent=32))
    with pytest.raises(mog.MogError, match="INVALID_ARG"):
        g.feature_map(om32)
    assert hc.sync_status() == 0 and hp.sync_status() == 0


# -------------------------------------------------------------- periodic re-clustering

@pytest.mark.parametrize("sliding,kpp", [(0, 0), (1, 0), (0, 1)])
def test_recluster_equals_fresh_build_and_matches_oracle(sliding, kpp):
    """mog_recluster after 40 appended tokens: the partition, the summaries and the window
    equal a fresh mog_build over the grown sequences (with the build's C and L), bit for
    bit -- also when the sliding window had moved keys into the clusters.  The statistics
    and the decode then match the oracle on that partition."""
    n0, steps = 3000, 40
    w = small_workload(n0, batch=2, h_kv=2, h_q=8, top_c=5, top_s=3, n_recent=32, seed=36)
    K, V, q, lens = wl.make_batch(w, n_cap=n0 + steps)
    rng = np.random.default_rng(37)
    prm = mog.make_params(2, 2, 8, n0 + steps, n_clusters=w.n_clusters, n_sub=w.n_sub, top_c=5,
                          top_s=3, n_sink=4, n_recent=32, sliding=sliding, kmeanspp=kpp)
    Kd, Vd = bf(K), bf(V)
    draws = wl.seed_draws(4, w.n_clusters, 38) if kpp else None   # k-means++: reused by recluster
    h = mog.build(Kd, Vd, lens, prm, draws=draws)
    for t in range(steps):
        kn = wl.to_bf16(rng.standard_normal((2, 2, D)))
        vn = wl.to_bf16(rng.standard_normal((2, 2, D)))
        h.append(bf(kn), bf(vn))
        K[:, :, n0 + t], V[:, :, n0 + t] = kn, vn
    h.recluster()
    fresh = mog.build(Kd, Vd, lens + steps, mog.make_params(
        2, 2, 8, n0 + steps, n_clusters=w.n_clusters, n_sub=w.n_sub, top_c=5, top_s=3, n_sink=4,
        n_recent=32, sliding=sliding, kmeanspp=kpp), draws=draws)
    torch.cuda.synchronize()
    assert h.sync_status() == 0 and fresh.sync_status() == 0
    lay = h.layout()
    U, cm, lm = lay.units, lay.c_max, lay.l_max
    for name, dt, shape in (("unit_info", torch.int32, (U, 8)), ("perm", torch.int32, (U, lay.n_cap)),
                            ("sub_off", torch.int32, (U, lay.sub_off_stride)), ("cl_n", torch.int32, (U, cm)),
                            ("cl_ms", torch.float32, (U, cm, 2, D)), ("cl_vbar", torch.float32, (U, cm, D)),
                            ("sub_n", torch.int32, (U, cm * lm)), ("sub_ms", torch.float32, (U, cm * lm, 2, D)),
                            ("sub_vbar", torch.float32, (U, cm * lm, D))):
        a = h.array(name, dt, shape).cpu().numpy()
        b = fresh.array(name, dt, shape).cpu().numpy()
        info = h.array("unit_info", torch.int32, (U, 8)).cpu().numpy()
        if name == "perm":   # only the mid region of each unit is defined
            for u in range(U):
                assert np.array_equal(a[u, :info[u, 3]], b[u, :info[u, 3]]), (name, u)
        elif name == "sub_off":   # C*L + 1 offsets per unit (the row stride is padded)
            for u in range(U):
                used = info[u, 0] * info[u, 1] + 1
                assert np.array_equal(a[u, :used], b[u, :used]), (name, u)
        else:
            assert np.array_equal(a, b), name
    assert int(h.array("unit_info", torch.int32, (U, 8)).cpu().numpy()[0, 2]) == n0 + steps
    # against the oracle, on the partition the GPU chose
    w2 = wl.Workload("recluster", batch=2, h_kv=2, h_q=8, n=n0 + steps, centres=64, n_clusters=w.n_clusters,
                     n_sub=w.n_sub, top_c=5, top_s=3, n_sink=4, n_recent=32, seed=36)
    chk = type("Chk", (), {})()
    chk.w, chk.h, chk.K, chk.V, chk.q, chk.qd = w2, h, K, V, q, bf(q)
    chk.lens = lens + steps
    chk.summ = {}
    for u in range(U):
        b, hh = divmod(u, 2)
        Cn, L, nm, S, perm, off = _partition(h, u, n0 + steps, w2)
        s = ora.stats(K[b, hh], V[b, hh], perm, off, Cn, L)
        s.update(perm=perm, sub_off=off, C=Cn, L=L, n_build=n0 + steps, S=S, R=32)
        chk.summ[(b, hh)] = s
    chk.gpu_summaries = lambda: Injected.gpu_summaries(chk)
    _check_stats(chk)
    print("recluster decode", _check_decode(chk))


# ------------------------------------------------------------------ paged KV cache

def _paged_copy(K, V, page_rows, heads_first, seed):
    """A paged copy of a contiguous cache [B, H, n_cap, d]: pages handed out in a random
    order, plus spare pages, in either page layout; returns (PagedKV, block table)."""
    B, H, n_cap, d = K.shape
    pps = -(-n_cap // page_rows)
    n_pages = B * pps + 5
    order = np.random.default_rng(seed).permutation(n_pages)[:B * pps].reshape(B, pps).astype(np.int32)
    shape = (n_pages, H, page_rows, d) if heads_first else (n_pages, page_rows, H, d)
    Kp = np.zeros(shape, np.uint16)
    Vp = np.zeros(shape, np.uint16)
    for b in range(B):
        for pg in range(pps):
            lo, hi = pg * page_rows, min(n_cap, (pg + 1) * page_rows)
            for h in range(H):
                if heads_first:
                    Kp[order[b, pg], h, :hi - lo], Vp[order[b, pg], h, :hi - lo] = K[b, h, lo:hi], V[b, h, lo:hi]
                else:
                    Kp[order[b, pg], :hi - lo, h], Vp[order[b, pg], :hi - lo, h] = K[b, h, lo:hi], V[b, h, lo:hi]
    bt = torch.from_numpy(order).to(DEV)
    return mog.PagedKV(bf(Kp), bf(Vp), bt, page_rows, heads_first=heads_first), order


@pytest.mark.parametrize("page_rows,heads_first", [(64, True), (16, False)])
def test_paged_cache_is_bit_identical_to_contiguous(page_rows, heads_first):
    """The same cache stored contiguously and as scattered pages behind a block table:
    build (the paged one without the tensor-core pass, which needs contiguous rows),
    decode, append and dense_decode give bit-identical partitions, summaries, selections
    and outputs."""
    steps = 6
    w = small_workload(2900, batch=2, h_kv=2, h_q=8, top_c=5, top_s=3, n_recent=32, seed=38)
    K, V, q, lens = wl.make_batch(w, n_cap=2900 + steps)
    lens = np.array([2900, 2750], np.int32)
    K[1, :, 2750:] = 0
    V[1, :, 2750:] = 0
    prm = mog.make_params(2, 2, 8, 2900 + steps, n_clusters=w.n_clusters, n_sub=w.n_sub, top_c=5,
                          top_s=3, n_sink=4, n_recent=32)
    Kd, Vd = bf(K), bf(V)
    pk, order = _paged_copy(K, V, page_rows, heads_first, seed=39)
    hc = mog.build(Kd, Vd, lens, prm)
    hp = mog.build(pk, None, lens, prm)
    qd = bf(q)
    SW = 5 + 15
    rng = np.random.default_rng(40)
    for t in range(steps + 1):
        sc = torch.empty((2 * 8, SW), dtype=torch.int32, device=DEV)
        sp = torch.empty_like(sc)
        oc = hc.decode(qd, sel_out=sc)
        op = hp.decode(qd, sel_out=sp)
        torch.cuda.synchronize()
        assert torch.equal(sc, sp), t
        assert torch.equal(oc, op), t
        if t == 0:
            lay = hc.layout()
            info = hc.array("unit_info", torch.int32, (lay.units, 8)).cpu().numpy()
            for u in range(lay.units):
                a_p, b_p = (x.array("perm", torch.int32, (lay.units, lay.n_cap))[u, :info[u, 3]] for x in (hc, hp))
                a_o, b_o = (x.array("sub_off", torch.int32, (lay.units, lay.sub_off_stride))[u, :info[u, 0] * info[u, 1] + 1]
                            for x in (hc, hp))
                assert torch.equal(a_p, b_p) and torch.equal(a_o, b_o), u
            for name, dt, shape in (("cl_ms", torch.float32, (lay.units, lay.c_max, 2, D)),
                                    ("sub_ms", torch.float32, (lay.units, lay.c_max * lay.l_max, 2, D)),
                                    ("sub_vbar", torch.float32, (lay.units, lay.c_max * lay.l_max, D))):
                assert torch.equal(hc.array(name, dt, shape), hp.array(name, dt, shape)), name
        if t < steps:
            kn = bf(wl.to_bf16(rng.standard_normal((2, 2, D))))
            vn = bf(wl.to_bf16(rng.standard_normal((2, 2, D))))
            hc.append(kn, vn)
            hp.append(kn, vn)
    ld = torch.tensor(lens + steps, dtype=torch.int32, device=DEV)
    dc = mog.dense_decode(Kd, Vd, ld, int(lens.max()) + steps, qd)
    dp = mog.dense_decode(pk, None, ld, int(lens.max()) + steps, qd)
    assert torch.equal(dc, dp)
    assert hc.sync_status() == 0 and hp.sync_status() == 0
    # the appended rows went into the right pages
    Kc = Kd.view(torch.int16).cpu().numpy().view(np.uint16)
    Kp = pk.K.view(torch.int16).cpu().numpy().view(np.uint16)
    for b, n in enumerate(lens):
        for t in range(steps):
            pos = n + t
            pg, r = order[b, pos // page_rows], pos % page_rows
            row = Kp[pg, :, r] if heads_first else Kp[pg, r, :]
            assert np.array_equal(row, Kc[b, :, pos])


@pytest.mark.parametrize("name,heads_per_unit", [("qwen3-14b-128k", (0, 4)), ("ctx-1m", (0, 3))])
def test_full_layer_build_and_decode(name, heads_per_unit):
    """A whole layer at full size, clustered by the library's own build: 4 sequences x 8 KV
    heads at 131072 keys (362 x 17 groups), or 8 KV heads at 1048576 keys (1024 x 20).
    Every head's statistics against the oracle's on the partition the GPU chose; selection
    and decode on two query heads of every KV head."""
    fb = FromBuildBatch(name)
    worst_s = _check_stats(fb)
    G = fb.w.group
    heads = [u * G + g for u in range(fb.w.batch * fb.w.h_kv) for g in heads_per_unit]
    ties, worst = _check_decode(fb, sample_heads=heads)
    print(f"{name} full layer: stats worst {worst_s:.2e}, {ties} near-tie heads, decode worst {worst:.2e}")
