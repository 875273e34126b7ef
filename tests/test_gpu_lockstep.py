"""Lockstep of mog_build's own two Lloyd loops against the fp64 oracle ("Iceberg
Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians", Abstract: the keys
of each head are split into clusters and each cluster into subclusters after prefill).

mog_build_traced records the centroids every step assigned to and the assignment it made,
at both levels.  For every step the tests check, on the GPU's own trajectory:
  (i)   the seeds are the member rows at floor(j n / k), bit for bit (with k-means++ seeding
        of the first level: the rows the oracle's k-means++ draws pick with the same
        uniforms, every round or sampled rounds);
  (ii)  the GPU's assignment equals the oracle's assignment to the GPU's centroids of that
        step, bit for bit (all rows, or a seeded sample of rows at 128K and 1M keys);
  (iii) the GPU's next centroids are the oracle's mean of the GPU's members within 1e-5
        relative (an empty group keeps its centroid exactly);
  (iv)  the loop stopped at the first step that changed no assignment, or after T steps;
  (v)   the final partition lists each cluster's members by (subcluster, position), as
        the oracle orders them from the GPU's last second-level labels.
"""
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
UPD_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    buildlib.build()
    ora.build()
    mog.lib()


def bf(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)


def traced_head(name, b=0, h=0, kpp=False):
    """One KV head of a workload, built by mog_build_traced (with kpp: k-means++ seeds from
    the input generator's draws, returned as the last item)."""
    w = wl.WORKLOADS[name]
    n = int(wl.lengths(w)[b])
    u = wl.UnitDraw(w, b, h, n)
    K = np.zeros((1, 1, n, D), np.uint16)
    V = np.zeros_like(K)
    u.keys_values(K[0, 0], V[0, 0])
    Cn, L = wl.clusters_for(w, n)
    prm = mog.make_params(1, 1, w.group, n, n_clusters=Cn, n_sub=L, top_c=w.top_c, top_s=w.top_s,
                          n_sink=w.n_sink, n_recent=w.n_recent, kmeanspp=int(kpp))
    draws = wl.seed_draws(1, Cn, w.seed + 100) if kpp else None
    hd, tr = mog.build(bf(K), bf(V), [n], prm, trace=True, draws=draws)
    torch.cuda.synchronize()
    assert hd.sync_status() == 0
    return w, K[0, 0], n, Cn, L, hd, tr, draws


def _updates_close(gpu_next, ref, prev, counts):
    """GPU centroids after an update against the oracle's means: relative L2 per centroid
    within UPD_TOL; a centroid with no members is unchanged bit for bit."""
    worst = 0.0
    for c in range(ref.shape[0]):
        if counts[c] == 0:
            assert np.array_equal(gpu_next[c], prev[c]), c
            continue
        nr = np.linalg.norm(ref[c])
        err = np.linalg.norm(gpu_next[c] - ref[c]) / nr if nr > 0 else np.abs(gpu_next[c]).max()
        worst = max(worst, err)
        assert err <= UPD_TOL, (c, err)
    return worst


def _expected_steps(labels, T):
    """(iv): the loop takes T steps unless some step t >= 1 repeats step t - 1's labels,
    in which case it stops after that step."""
    for t in range(1, len(labels)):
        if np.array_equal(labels[t], labels[t - 1]):
            return t + 1
    return T


def lockstep(name, l1_sample=None, l2_clusters=None, seed=0, kpp=False, pp_rounds=None):
    """pp_rounds (with kpp): the k-means++ rounds checked one by one against the oracle's
    step given the GPU's earlier seeds; None checks the whole seed sequence at once."""
    w, K, n, Cn, L, hd, tr, draws = traced_head(name, kpp=kpp)
    S, R = w.n_sink, w.n_recent
    nm = n - S - R
    T1, T2 = tr.layout.iters_l1, tr.layout.iters_l2
    Kmid = np.ascontiguousarray(K[S:S + nm])
    X = wl.from_bf16(Kmid)
    lay = hd.layout()
    steps1 = int(hd.array("l1_steps", torch.int32, (1,)).cpu().numpy()[0])
    l1c = tr.l1_cent[0].cpu().numpy()[:, :Cn]
    l1a = tr.l1_assign[0].cpu().numpy()[:, :nm]
    rng = np.random.default_rng(seed)
    rows = (np.arange(nm) if l1_sample is None or l1_sample >= nm
            else np.sort(rng.choice(nm, size=l1_sample, replace=False)))
    # ------------------------------------------------------------ first level
    if kpp:
        pp = hd.array("pp_idx", torch.int32, (1, lay.c_max)).cpu().numpy()[0, :Cn].astype(np.int64)
        if pp_rounds is None:
            assert np.array_equal(pp, ora.kmeanspp(Kmid, Cn, draws[0])), "k-means++ seeds"
        else:
            for r in pp_rounds:
                assert ora.pp_pick(Kmid, pp[:r], draws[0, r]) == pp[r], ("k-means++ round", r)
        nd = len(set(pp.tolist()))   # distinct, unless every key already sits on a seed
        assert nd == Cn or nd == len(np.unique(Kmid, axis=0)), nd
        assert np.array_equal(l1c[0], X[pp])                                             # (i)
    else:
        assert np.array_equal(l1c[0], X[(np.arange(Cn) * nm) // Cn])                  # (i)
    worst1 = 0.0
    for t in range(steps1):
        cent = l1c[t].astype(np.float64)
        assert np.array_equal(l1a[t, rows], ora.assign(Kmid, cent, rows=rows)), ("L1 step", t)  # (ii)
        if t + 1 < steps1:
            ref = ora.update(Kmid, l1a[t], cent)
            cnt = np.bincount(l1a[t], minlength=Cn)
            worst1 = max(worst1, _updates_close(l1c[t + 1], ref, l1c[t], cnt))          # (iii)
    assert steps1 == _expected_steps(l1a[:steps1], T1)                                  # (iv)
    for t in range(1, steps1 - 1):
        assert not np.array_equal(l1a[t], l1a[t - 1]), t
    for t in range(steps1, T1):          # steps after the stop repeat the last one
        assert np.array_equal(l1a[t], l1a[steps1 - 1]) and np.array_equal(l1c[t], l1c[steps1 - 1])
    final = l1a[steps1 - 1]
    assert np.array_equal(hd.array("l1_assign", torch.int32, (1, lay.n_cap)).cpu().numpy()[0, :nm], final)
    # ----------------------------------------------------------- second level
    order = np.argsort(final, kind="stable")               # members by (cluster, position)
    starts = np.searchsorted(final[order], np.arange(Cn + 1))
    l2c = tr.l2_cent[0].cpu().numpy()
    l2a = tr.l2_assign[0].cpu().numpy()[:, :nm]
    l2s = tr.l2_steps[0].cpu().numpy()
    perm = hd.array("perm", torch.int32, (1, lay.n_cap)).cpu().numpy()[0, :nm]
    off = hd.array("sub_off", torch.int32, (1, lay.sub_off_stride)).cpu().numpy()[0, :Cn * L + 1]
    clusters = range(Cn) if l2_clusters is None else l2_clusters
    worst2, stepped = 0.0, 0
    for c in clusters:
        a, e = starts[c], starts[c + 1]
        mem = order[a:e]
        nc = e - a
        st = int(l2s[c])
        if nc == 0:
            assert st == 0 and off[c * L] == off[(c + 1) * L]
            continue
        assert 1 <= st <= T2
        cc = l2c[c, :, :L]
        assert np.array_equal(cc[0], X[mem[(np.arange(L) * nc) // L]]), c                 # (i)
        labs = []
        for t in range(st):
            cent = cc[t].astype(np.float64)
            lab = l2a[t, a:e]
            assert np.array_equal(lab, ora.assign(Kmid, cent, rows=mem)), ("L2", c, t)    # (ii)
            labs.append(lab)
            if t + 1 < st:
                ref = ora.update(Kmid, lab, cent, rows=mem)
                worst2 = max(worst2, _updates_close(cc[t + 1], ref, cc[t], np.bincount(lab, minlength=L)))  # (iii)
        assert st == _expected_steps(labs, T2), (c, st)                                  # (iv)
        for t in range(1, st - 1):
            assert not np.array_equal(labs[t], labs[t - 1]), (c, t)
        last = labs[-1]                                                                   # (v)
        assert np.array_equal(perm[off[c * L]:off[(c + 1) * L]], S + mem[np.argsort(last, kind="stable")]), c
        assert np.array_equal(np.diff(off[c * L:(c + 1) * L + 1]), np.bincount(last, minlength=L)), c
        stepped += st
    return dict(steps1=steps1, worst_l1_update=worst1, worst_l2_update=worst2, l2_steps=stepped,
                rows_checked=int(rows.size))


def test_lockstep_tiny():
    r = lockstep("tiny-4k")
    print("tiny lockstep", r)
    assert r["steps1"] >= 3


def test_lockstep_qwen3_4b_full_head():
    """A full 32K-key head (181 clusters x 15 subclusters), every row at every step."""
    print("32K lockstep", lockstep("qwen3-4b-32k"))


def test_lockstep_qwen3_14b_head_362_clusters():
    """A 131072-key head with 0.1% outliers (362 clusters, several tensor-core centroid
    groups); first-level assignments on 16384 sampled rows per step, every cluster's
    second level in full."""
    print("128K lockstep", lockstep("qwen3-14b-128k", l1_sample=16384, seed=3))


def test_lockstep_1m_head_1024_clusters():
    """A 1M-key head (1024 clusters x 20 subclusters): first-level assignments on 16384
    sampled rows per step, every first-level update in full, every cluster's second level
    in full."""
    print("1M lockstep", lockstep("ctx-1m", l1_sample=16384, seed=4))


# ------------------------------------------------------------- k-means++ seeding (variant)

def test_kmeanspp_lockstep_tiny():
    """k-means++ seeds equal the oracle's for the same draws, then the whole lockstep."""
    r = lockstep("tiny-4k", kpp=True)
    print("tiny k-means++ lockstep", r)


def test_kmeanspp_lockstep_qwen3_4b_full_head():
    """A full 32K-key head: all 181 seeds against the oracle, every row at every step."""
    print("32K k-means++ lockstep", lockstep("qwen3-4b-32k", kpp=True))


def test_kmeanspp_lockstep_qwen3_14b_head():
    """A 131072-key head: all 362 seeds against the oracle; the Lloyd steps on 16384 sampled
    rows, every cluster's second level in full."""
    print("128K k-means++ lockstep", lockstep("qwen3-14b-128k", l1_sample=16384, seed=5, kpp=True))


def test_kmeanspp_lockstep_1m_head_sampled_rounds():
    """A 1M-key head: rounds 0-3, 17, 64 and 255 of the seeding, each against the oracle's
    step from the GPU's earlier seeds; the Lloyd steps on 16384 sampled rows."""
    print("1M k-means++ lockstep", lockstep("ctx-1m", l1_sample=16384, seed=6, kpp=True,
                                            pp_rounds=[0, 1, 2, 3, 17, 64, 255]))
