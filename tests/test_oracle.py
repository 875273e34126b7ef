"""Pins of the fp64 CPU oracle against facts that do not come from the oracle itself:
library routines (scipy's k-means and distances, numpy statistics, scipy's softmax),
closed forms (the Gaussian moment generating function), exactness cases the method
guarantees, and invariants.  No GPU is used.
"""
import math

import numpy as np
import pytest
from scipy.cluster.vq import kmeans2
from scipy.spatial.distance import cdist
from scipy.special import logsumexp, softmax

from serving_mog_decode_gb300 import workloads as wl

D = 128
TAU = 1.0 / math.sqrt(D)


def f64(h):
    return wl.from_bf16(h).astype(np.float64)


def dense_ref(K, V, n, q):
    """Softmax attention written with scipy/numpy, independent of the oracle."""
    logits = TAU * (f64(K[:n]) @ f64(q))
    return softmax(logits) @ f64(V[:n])


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def planted(n, M=16, sigma=0.5, seed=0, d=D):
    g = np.random.default_rng(seed)
    c = g.standard_normal((M, d))
    z = g.integers(0, M, n)
    K = wl.to_bf16(c[z] + sigma * g.standard_normal((n, d)))
    V = wl.to_bf16(g.standard_normal((n, d)))
    q = wl.to_bf16(0.5 * c[0] + 0.5 * g.standard_normal(d))
    return K, V, q


# ----------------------------------------------------------------------------- inputs

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(3).standard_normal(100000) * 10.0 ** np.random.default_rng(4).integers(-8, 8, 100000)
    ours = wl.to_bf16(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_generator_is_deterministic_and_planted():
    w = wl.WORKLOADS["tiny-4k"]
    K1, V1, q1 = wl.make_unit(w)
    K2, V2, q2 = wl.make_unit(w)
    assert np.array_equal(K1, K2) and np.array_equal(V1, V2) and np.array_equal(q1, q2)
    k = f64(K1)
    assert np.allclose(np.linalg.norm(k[:4], axis=1), 8.0, rtol=1e-2)  # sinks 8*u
    u = wl.UnitDraw(w, 0, 0, w.n)
    resid = k[4:] - u.centres[u.z[4:]]
    assert abs(resid.std() - 0.5) < 0.01                       # sigma 0.5 around centres
    assert abs(f64(V1).std() - 1.0) < 0.01


# ----------------------------------------------------------------------------- k-means

def test_assign_matches_scipy_cdist():
    g = np.random.default_rng(1)
    X = wl.to_bf16(g.standard_normal((3000, D)))
    cent = g.standard_normal((37, D))
    ref = np.argmin(cdist(f64(X), cent, "sqeuclidean"), axis=1)
    from oracle import assign
    assert np.array_equal(assign(X, cent), ref)


def test_assign_ties_take_lowest_index(ora):
    g = np.random.default_rng(2)
    X = wl.to_bf16(g.standard_normal((200, D)))
    base = g.standard_normal((5, D))
    cent = np.concatenate([base, base[::-1]])       # every centroid duplicated
    a = ora.assign(X, cent)
    assert a.max() < 5                              # the lower copy always wins
    assert np.array_equal(a, np.argmin(cdist(f64(X), base, "sqeuclidean"), axis=1))
    # a key equidistant from two centroids goes to the lower index
    c2 = np.stack([np.full(D, 1.0), np.full(D, -1.0)])
    assert ora.assign(wl.to_bf16(np.zeros((1, D))), c2)[0] == 0
    assert ora.assign(wl.to_bf16(np.zeros((1, D))), c2[::-1].copy())[0] == 0


@pytest.mark.parametrize("T", [1, 2, 5, 10])
def test_lloyd_matches_scipy_kmeans2(ora, T):
    K, _, _ = planted(2000, M=24, sigma=0.8, seed=5)
    k = 12
    cent, asg, steps, hist = ora.lloyd(K, k, T, history=True)
    X = f64(K)
    init = X[(np.arange(k) * X.shape[0]) // k]                 # strided seeding
    assert np.array_equal(hist[0], init)
    # scipy runs `iter` assign+update rounds; our label after `steps` assignment steps is
    # scipy's label with iter=steps (same centroid history), and the centroids used by
    # our last step are scipy's code book after steps-1 updates.
    cb, lab = kmeans2(X, init.copy(), iter=steps, minit="matrix", missing="warn")
    assert np.array_equal(asg, lab)
    if steps >= 2:
        cb_prev, _ = kmeans2(X, init.copy(), iter=steps - 1, minit="matrix", missing="warn")
        assert np.allclose(cent, cb_prev, rtol=0, atol=1e-12)
    if steps < T:   # early stop only at a fixed point
        assert np.array_equal(ora.assign(K, cb), asg)


def test_lloyd_objective_never_increases(ora):
    K, _, _ = planted(3000, M=40, sigma=0.7, seed=6)
    _, _, steps, hist = ora.lloyd(K, 20, 10, history=True)
    X = f64(K)
    obj = [cdist(X, h, "sqeuclidean").min(axis=1).sum() for h in hist]
    assert steps >= 3
    assert all(b <= a * (1 + 1e-12) for a, b in zip(obj, obj[1:]))


def test_update_is_the_member_mean_and_empty_keeps(ora):
    """The oracle's update step on its own: numpy's mean of each centroid's rows; a
    centroid with no rows keeps its value (R6); rows may be a subset, in any order."""
    K, _, _ = planted(700, M=9, seed=8)
    g = np.random.default_rng(8)
    cent = g.standard_normal((6, D))
    a = g.integers(0, 5, size=400).astype(np.int32)      # centroid 5 gets no rows
    rows = g.choice(700, size=400, replace=False)
    new = ora.update(K, a, cent, rows=rows)
    X = f64(K)
    for c in range(5):
        np.testing.assert_allclose(new[c], X[rows[a == c]].mean(0), rtol=1e-13, atol=1e-14)
    assert np.array_equal(new[5], cent[5])
    # with the full row set it is one step of the oracle's own Lloyd loop
    _, _, steps, hist = ora.lloyd(K, 6, 4, history=True)
    for t in range(steps - 1):
        assert np.array_equal(ora.update(K, ora.assign(K, hist[t]), hist[t]), hist[t + 1])
    with pytest.raises(RuntimeError):
        ora.update(K, np.full(700, 6, np.int32), cent)   # label out of range


def test_lloyd_more_centroids_than_points(ora):
    K, _, _ = planted(5, M=5, seed=7)
    cent, asg, steps, _ = ora.lloyd(K, 8, 3)
    # seeds repeat members; duplicates tie and the lower index keeps the member
    assert sorted(asg.tolist()) == sorted(set(asg.tolist()))   # each member its own cluster
    assert np.array_equal(f64(K)[:, :], cent[asg])


# ----------------------------------------------------------------------------- statistics

def test_stats_match_numpy_and_identities(ora):
    g = np.random.default_rng(8)
    n, Cn, L = 1500, 7, 5
    K = wl.to_bf16(g.standard_normal((n, D)) * 2 + 1)
    V = wl.to_bf16(g.standard_normal((n, D)))
    lab = g.integers(0, Cn * L, n)
    lab[lab == 3] = 4                                     # group 3 stays empty
    perm = np.argsort(lab, kind="stable").astype(np.int32)
    sub_off = np.searchsorted(lab[perm], np.arange(Cn * L + 1)).astype(np.int32)
    s = ora.stats(K, V, perm, sub_off, Cn, L)
    X, Y = f64(K), f64(V)
    for grp in range(Cn * L):
        m = lab == grp
        assert s["sub_n"][grp] == m.sum()
        if m.sum() == 0:
            assert not s["sub_mu"][grp].any() and not s["sub_var"][grp].any()
            continue
        np.testing.assert_allclose(s["sub_mu"][grp], X[m].mean(0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(s["sub_var"][grp], X[m].var(0), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s["sub_vbar"][grp], Y[m].mean(0), rtol=1e-12, atol=1e-12)
    for c in range(Cn):
        m = (lab // L) == c
        sl = slice(c * L, (c + 1) * L)
        ns = s["sub_n"][sl].astype(np.float64)
        assert s["cl_n"][c] == m.sum() == ns.sum()
        np.testing.assert_allclose(s["cl_mu"][c], X[m].mean(0), rtol=1e-12, atol=1e-12)
        # count-weighted sub means give the cluster mean; law of total variance
        np.testing.assert_allclose((ns[:, None] * s["sub_mu"][sl]).sum(0) / ns.sum(), s["cl_mu"][c],
                                   atol=1e-12)
        within = (ns[:, None] * s["sub_var"][sl]).sum(0) / ns.sum()
        between = (ns[:, None] * (s["sub_mu"][sl] - s["cl_mu"][c]) ** 2).sum(0) / ns.sum()
        np.testing.assert_allclose(s["cl_var"][c], within + between, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s["cl_vbar"][c], Y[m].mean(0), rtol=1e-12, atol=1e-12)


def test_build_partition_is_consistent(ora):
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    S, R, Cn, L = w.n_sink, w.n_recent, w.n_clusters, w.n_sub
    b = ora.build_unit(K, V, w.n, S, R, Cn, L)
    nm = w.n - S - R
    perm, off, a1 = b["perm"], b["sub_off"], b["l1_assign"]
    assert np.array_equal(np.sort(perm), np.arange(S, S + nm))           # mid region only
    assert off[0] == 0 and off[-1] == nm and np.all(np.diff(off) >= 0)
    # clusters are the first-level labels; positions ascend inside every subcluster
    for c in range(Cn):
        seg = perm[off[c * L]:off[(c + 1) * L]]
        assert np.all(a1[seg - S] == c)
        for l in range(L):
            sub = perm[off[c * L + l]:off[c * L + l + 1]]
            assert np.all(np.diff(sub) > 0)
    # the first level is scipy's k-means from the same strided seeds
    X = f64(K[S:S + nm])
    init = X[(np.arange(Cn) * nm) // Cn]
    s1 = b["steps"][0]
    _, lab = kmeans2(X, init, iter=s1, minit="matrix", missing="warn")
    assert np.array_equal(a1, lab)
    # the second level of every cluster is scipy's k-means on its members, run for
    # exactly the number of steps the oracle's loop took on that cluster
    checked = 0
    for c in range(Cn):
        seg = np.sort(perm[off[c * L]:off[(c + 1) * L]])
        if seg.size == 0:
            continue
        Xc = f64(K[seg])
        init2 = Xc[(np.arange(L) * seg.size) // L]
        sub_of = np.empty(seg.size, np.int64)
        for l in range(L):
            sub_of[np.isin(seg, perm[off[c * L + l]:off[c * L + l + 1]])] = l
        _, own, st2, _ = ora.lloyd(K, L, 10, rows=seg)
        assert np.array_equal(own, sub_of), c
        lab2 = kmeans2(Xc, init2.copy(), iter=st2, minit="matrix", missing="warn")[1]
        assert np.array_equal(lab2, sub_of), (c, st2)
        checked += 1
    assert checked == int((b["cl_n"] > 0).sum())


# ------------------------------------------------------------------ k-means++ seeding

def _pp_set(n, seed, dup=None):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((n, D)) * rng.uniform(0.2, 3.0, (n, 1))
    if dup is not None:
        X = X[np.arange(n) % dup]
    return wl.to_bf16(X)


def _d2(X, seeds):
    """Squared distance of every row to its nearest seed, by scipy (fp64)."""
    return cdist(f64(X), f64(X[np.asarray(seeds)]), "sqeuclidean").min(axis=1)


def test_pp_pick_hits_constructed_intervals(ora):
    """A draw in the middle of member i's interval of the D2-weighted line picks i: the
    inversion rule of k-means++ sampling, with D2 from scipy."""
    X = _pp_set(40, 1)
    for r in range(1, 6):
        seeds = [7, 31, 2, 19, 25][:r]
        d2 = _d2(X, seeds)
        cum = np.concatenate([[0.0], np.cumsum(d2)])
        for i in range(40):
            if d2[i] == 0:
                assert i in seeds
                continue
            u = (cum[i] + 0.5 * d2[i]) / cum[-1]
            assert ora.pp_pick(X, seeds, u) == i, (r, i)
    # the first seed: member floor(u n)
    for i in range(40):
        assert ora.pp_pick(X, [], (i + 0.5) / 40) == i
    assert ora.pp_pick(X, [], 0.0) == 0


def test_pp_pick_frequencies_follow_squared_distance(ora):
    """Over uniform draws, member i is picked with probability D2_i / sum D2 (scipy D2);
    every frequency lies within 5 binomial standard deviations."""
    X = _pp_set(12, 2)
    seeds = [3, 8]
    p = _d2(X, seeds)
    p = p / p.sum()
    rng = np.random.default_rng(5)
    m = 20000
    picks = np.array([ora.pp_pick(X, seeds, u) for u in rng.random(m)])
    f = np.bincount(picks, minlength=12) / m
    assert f[3] == 0 and f[8] == 0
    assert np.all(np.abs(f - p) <= 5 * np.sqrt(p * (1 - p) / m) + 1e-12), (f, p)


def test_kmeanspp_special_cases(ora):
    rng = np.random.default_rng(3)
    # k = n distinct members: every member becomes a seed exactly once
    X = _pp_set(30, 4)
    s = ora.kmeanspp(X, 30, rng.random(30))
    assert sorted(s.tolist()) == list(range(30))
    # all members equal: sum D2 = 0 after the first seed, so every pick is floor(u n)
    Xe = np.repeat(_pp_set(1, 5), 25, axis=0)
    u = rng.random(6)
    assert ora.kmeanspp(Xe, 6, u).tolist() == np.floor(u * 25).astype(int).tolist()
    # two distinct points repeated: the second seed is always of the other point
    X2 = _pp_set(40, 6, dup=2)
    for _ in range(20):
        s = ora.kmeanspp(X2, 2, rng.random(2))
        assert s[0] % 2 != s[1] % 2
    # the seeds of the full sequence are the one-step picks given the seeds before them
    u = rng.random(12)
    s = ora.kmeanspp(X, 12, u)
    assert all(ora.pp_pick(X, s[:r], u[r]) == s[r] for r in range(12))
    # a member already chosen is never drawn again while some distance is positive
    assert len(set(s.tolist())) == 12
    with pytest.raises(RuntimeError):
        ora.kmeanspp(X, 3, [0.5, 1.0, 0.2])      # draws must lie in [0, 1)


def test_build_with_kmeanspp_seeds_is_lloyd_from_them(ora):
    """With draws, the first level is scipy's k-means started from the k-means++ seeds
    (the rows the pick rule chooses), for the number of steps the oracle took; the rest of
    the build is unchanged."""
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    S, R, Cn, L = w.n_sink, w.n_recent, w.n_clusters, w.n_sub
    nm = w.n - S - R
    u = np.random.default_rng(8).random(Cn)
    b = ora.build_unit(K, V, w.n, S, R, Cn, L, draws=u)
    seeds = ora.kmeanspp(K[S:S + nm], Cn, u)
    X = f64(K[S:S + nm])
    _, lab = kmeans2(X, X[seeds], iter=b["steps"][0], minit="matrix", missing="warn")
    assert np.array_equal(b["l1_assign"], lab)
    assert np.array_equal(np.sort(b["perm"]), np.arange(S, S + nm))
    # strided seeds give a different partition on these inputs
    assert not np.array_equal(ora.build_unit(K, V, w.n, S, R, Cn, L)["l1_assign"], b["l1_assign"])


# -------------------------------------------------------- feature-map residual (R29)

def _fm_case(n=300, scale=1.0, seed=9):
    rng = np.random.default_rng(seed)
    K = wl.to_bf16(rng.standard_normal((n, D)) * scale)
    V = wl.to_bf16(rng.standard_normal((n, D)))
    q = wl.to_bf16(rng.standard_normal(D) * scale)
    return K, V, q


def _np_feature_weights(K, q, omega):
    """phi(q~).phi(k~) for every row of K, written with numpy matrix products (fp64)."""
    st = math.sqrt(TAU)
    qt, kt = st * f64(q), st * f64(K)
    a = omega @ qt - 0.5 * qt @ qt                      # [m]
    b = kt @ omega.T - 0.5 * np.sum(kt * kt, axis=1)[:, None]   # [n, m]
    return np.exp(a[None, :] + b).mean(axis=1)


def test_fm_identity_random_features_estimate_the_softmax_kernel():
    """E over w ~ N(0, I) of exp(w.x - |x|^2/2) exp(w.y - |y|^2/2) = exp(x.y): the sample
    mean over 400,000 draws lies within 5 standard errors (the identity R29 rests on)."""
    rng = np.random.default_rng(1)
    x, y = rng.standard_normal(D) * 0.06, rng.standard_normal(D) * 0.06
    w = rng.standard_normal((400000, D))
    f = np.exp(w @ x - 0.5 * x @ x + w @ y - 0.5 * y @ y)
    assert abs(f.mean() - math.exp(x @ y)) <= 5 * f.std() / math.sqrt(f.size)


def test_fm_decode_matches_brute_force_and_special_cases(ora):
    K, V, q = _fm_case()
    S, R, Cn, L = 4, 16, 4, 3
    n = K.shape[0]
    b = ora.build_unit(K, V, n, S, R, Cn, L)
    omega = np.random.default_rng(2).standard_normal((64, D))
    # nothing selected: anchors exact, every mid key estimated
    sc = np.full(2, -1, np.int32)
    ss = np.full((2, 2), -1, np.int32)
    out, diag = ora.decode_fm(K, V, n, q, b, sc, ss, omega)
    w_exact = np.exp(TAU * (f64(K) @ f64(q)))
    anchors = np.r_[0:S, n - R:n]
    mid = np.arange(S, n - R)
    w = np.zeros(n)
    w[anchors] = w_exact[anchors]
    w[mid] = _np_feature_weights(K[mid], q, omega)
    ref = w @ f64(V) / w.sum()
    assert rel_l2(out, ref) < 1e-12 and diag[2] == S + R and diag[3] == n - S - R
    # two subclusters selected: their members move to the exact part
    sc = np.array([1, 3], np.int32)
    ss = np.array([[0, 2], [1, -1]], np.int32)
    out, diag = ora.decode_fm(K, V, n, q, b, sc, ss, omega)
    off, perm = b["sub_off"], b["perm"]
    chosen = np.concatenate([perm[off[c * L + l]:off[c * L + l + 1]] for c, l in ((1, 0), (1, 2), (3, 1))])
    w2 = w.copy()
    w2[chosen] = w_exact[chosen]
    assert rel_l2(out, w2 @ f64(V) / w2.sum()) < 1e-12 and diag[2] == S + R + chosen.size
    # everything selected: the dense softmax, no key estimated
    sc = np.arange(Cn, dtype=np.int32)
    ss = np.tile(np.arange(L, dtype=np.int32), (Cn, 1))
    out, diag = ora.decode_fm(K, V, n, q, b, sc, ss, omega)
    assert rel_l2(out, dense_ref(K, V, n, q)) < 1e-12 and diag[3] == 0


def test_fm_decode_converges_to_dense_with_more_features(ora):
    """Nothing selected, small keys (the estimator's variance is then small) and values
    with mean 1: the output approaches the dense softmax as the number of features grows,
    the error falling about as 1 / sqrt(m)."""
    rng = np.random.default_rng(10)
    n = 300
    K = wl.to_bf16(rng.standard_normal((n, D)) * 0.3)
    V = wl.to_bf16(rng.standard_normal((n, D)) + 1.0)
    q = wl.to_bf16(rng.standard_normal(D) * 0.3)
    b = ora.build_unit(K, V, n, 4, 16, 4, 3)
    sc = np.full(1, -1, np.int32)
    ss = np.full((1, 1), -1, np.int32)
    ref = dense_ref(K, V, n, q)
    rng = np.random.default_rng(3)
    errs = [rel_l2(ora.decode_fm(K, V, n, q, b, sc, ss, rng.standard_normal((m, D)))[0], ref)
            for m in (64, 1024, 16384)]
    assert errs[2] < 0.003 and errs[2] < errs[1] / 2 < errs[0] / 4, errs


def test_fm_sums_are_the_per_subcluster_feature_sums(ora):
    K, V, q = _fm_case(seed=11)
    S, R, Cn, L = 4, 16, 4, 3
    n = K.shape[0]
    b = ora.build_unit(K, V, n, S, R, Cn, L)
    omega = np.random.default_rng(4).standard_normal((16, D))
    z = ora.fm_sums(K, V, b, omega)
    st = math.sqrt(TAU)
    off, perm = b["sub_off"], b["perm"]
    for g in range(Cn * L):
        rows = perm[off[g]:off[g + 1]]
        kt = st * f64(K[rows])
        e = np.exp(kt @ omega.T - 0.5 * np.sum(kt * kt, axis=1)[:, None])   # [rows, m]
        assert np.allclose(z[g, :, D], e.sum(axis=0), rtol=1e-12, atol=0)
        assert np.allclose(z[g, :, :D], e.T @ f64(V[rows]), rtol=1e-10, atol=1e-300)


# ----------------------------------------------------------------------------- estimator

def _single_group(ora, K, V):
    """Everything in one cluster / one subcluster, no anchors."""
    n = K.shape[0]
    return ora.build_unit(K, V, n, 0, 0, 1, 1, 1, 1)


def test_log_mass_is_gaussian_mgf(ora):
    """For keys drawn from N(mu, diag s^2), sum_i exp(tau q.k_i) -> n exp(tau q.mu +
    tau^2 sum q_j^2 s_j^2 / 2): the residual exponent must match the empirical log-sum."""
    g = np.random.default_rng(11)
    n = 200000
    mu = g.standard_normal(D)
    s = g.uniform(0.2, 1.2, D)
    K = wl.to_bf16(mu + s * g.standard_normal((n, D)))
    V = wl.to_bf16(g.standard_normal((n, D)))
    q = wl.to_bf16(0.6 * g.standard_normal(D) / s)
    summ = _single_group(ora, K, V)
    out, diag = ora.decode(K, V, n, q, summ, np.array([-1], np.int32), np.array([[-1]], np.int32))
    e_s = diag[0]                       # no exact keys: m is the residual exponent itself
    emp = logsumexp(TAU * (f64(K) @ f64(q)))
    qq = f64(q)
    half = 0.5 * TAU ** 2 * np.sum(qq ** 2 * summ["cl_var"][0])
    assert half > 0.1                   # the variance term matters at this scale
    assert abs(e_s - emp) < 0.02 * half + 5e-3   # sampling error ~1.5e-3
    np.testing.assert_allclose(out, summ["cl_vbar"][0], atol=1e-12)   # lone group: out = vbar


def test_log_mass_two_point_group(ora):
    """Two keys mu +- delta e_j: population variance delta^2 in dimension j only; the
    exact log-sum is ln(2 cosh(tau q_j delta)) + tau q.mu; the Gaussian exponent replaces
    ln cosh(x) by x^2/2, so the gap is ln cosh(x) - x^2/2 = -x^4/12 + x^6/45 - ..."""
    mu = np.zeros(D)
    mu[:4] = [1.0, -2.0, 0.5, 3.0]
    K = np.stack([mu, mu]).copy()
    K[0, 5] += 0.25
    K[1, 5] -= 0.25
    Kb = wl.to_bf16(K)
    V = wl.to_bf16(np.random.default_rng(0).standard_normal((2, D)))
    q = np.zeros(D)
    q[:4] = [0.5, 0.25, -1.0, 2.0]
    q[5] = 2.0
    qb = wl.to_bf16(q)
    summ = _single_group(ora, Kb, V)
    _, diag = ora.decode(Kb, V, 2, qb, summ, np.array([-1], np.int32), np.array([[-1]], np.int32))
    x = TAU * 2.0 * 0.25
    exact = math.log(2 * math.cosh(x)) + TAU * float(f64(qb) @ mu)
    assert abs((exact - diag[0]) - (math.log(math.cosh(x)) - x * x / 2)) < 1e-14
    assert abs(math.log(math.cosh(x)) - x * x / 2 + x ** 4 / 12) < x ** 6 / 40


def test_all_selected_equals_dense(ora):
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    b = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    out, sel_c, sel_s, diag = ora.mog_head(K, V, w.n, q[0], b, w.n_clusters, w.n_sub)
    nonempty = int((b["cl_n"] > 0).sum())
    assert (sel_c >= 0).sum() == nonempty
    assert diag[2] == w.n
    ref = dense_ref(K, V, w.n, q[0])
    assert rel_l2(out, ref) < 1e-12
    assert rel_l2(ora.dense(K, V, w.n, q[0]), ref) < 1e-12


def test_singleton_subclusters_make_residual_exact(ora):
    K, V, q = planted(300, M=6, seed=12)
    Cn, L = 4, 300            # L >= any cluster size: every member becomes its own subcluster
    b = ora.build_unit(K, V, 300, 2, 10, Cn, L, 10, 3)
    assert b["sub_n"].max() == 1
    assert np.all(b["sub_var"] == 0)
    out, _, _, diag = ora.mog_head(K, V, 300, q, b, Cn, 0)   # all clusters, no subclusters
    assert diag[2] == 12                                      # only the anchors are exact
    assert rel_l2(out, dense_ref(K, V, 300, q)) < 1e-12


def test_duplicate_keys_make_residual_exact(ora):
    g = np.random.default_rng(13)
    distinct = g.standard_normal((16, D)) * 2
    Kd = np.repeat(distinct, 8, axis=0)              # position p holds vector p // 8
    K = wl.to_bf16(Kd)
    V = wl.to_bf16(g.standard_normal((128, D)))
    q = wl.to_bf16(0.3 * distinct[3] + 0.3 * g.standard_normal(D))
    b = ora.build_unit(K, V, 128, 0, 0, 16, 3)
    assert np.all(b["cl_n"] == 8) and np.all(b["cl_var"] == 0)
    out, _, _, diag = ora.mog_head(K, V, 128, q, b, 0, 0)    # nothing selected
    assert diag[2] == 0
    assert rel_l2(out, dense_ref(K, V, 128, q)) < 1e-12


def test_short_context_is_all_anchors(ora):
    K, V, q = planted(200, seed=14)
    b = ora.build_unit(K, V, 200, 4, 196, 3, 2)
    assert b["perm"].size == 0 and np.all(b["cl_n"] == 0)
    out, _, _, diag = ora.mog_head(K, V, 200, q, b, 3, 2)
    assert diag[2] == 200
    assert rel_l2(out, dense_ref(K, V, 200, q)) < 1e-12


def test_appended_keys_join_recent_anchors(ora):
    K, V, q = planted(600, seed=15)
    b = ora.build_unit(K, V, 500, 4, 32, 8, 4)
    out, _, _, diag = ora.mog_head(K, V, 600, q, b, 8, 4)   # all selected
    assert diag[2] == 600
    assert rel_l2(out, dense_ref(K, V, 600, q)) < 1e-12


def test_tiny_sweep_brute_force(ora):
    """Tiny N (64 keys, 8 clusters x 4 subclusters): every (top_c, top_s) case against a
    direct restatement in numpy -- scores of every group from numpy statistics of the
    partition, the ranking by brute force, the exact set and the residual groups listed
    by hand, and the whole mixture as one softmax."""
    K, V, q = planted(64, M=5, seed=16)
    S, R, Cn, L = 2, 6, 8, 4
    b = ora.build_unit(K, V, 64, S, R, Cn, L)
    perm, off = b["perm"], b["sub_off"]
    Kf, qf = f64(K), f64(q)

    def score(mem):
        X = Kf[mem]
        return math.log(len(mem)) + TAU * (qf @ X.mean(0)) + 0.5 * TAU ** 2 * float(qf ** 2 @ X.var(0))

    def ranked(scores):   # (score desc, index asc) over the non-empty groups
        return [i for _, i in sorted((-sc, i) for i, sc in scores.items())]

    cl_mem = {c: perm[off[c * L]:off[(c + 1) * L]] for c in range(Cn)}
    sub_mem = {(c, l): perm[off[c * L + l]:off[c * L + l + 1]] for c in range(Cn) for l in range(L)}
    cl_rank = ranked({c: score(m) for c, m in cl_mem.items() if m.size})
    anchors = list(range(S)) + list(range(64 - R, 64))
    cases = 0
    for tc in range(0, Cn + 1):
        for ts in range(0, L + 1):
            out, sel_c, sel_s, _ = ora.mog_head(K, V, 64, q, b, tc, ts)
            chosen = cl_rank[:tc]
            assert [int(c) for c in sel_c if c >= 0] == chosen
            exact, groups = list(anchors), []
            for c in range(Cn):
                if c not in chosen:
                    if cl_mem[c].size:
                        groups.append(cl_mem[c])
                    continue
                i = chosen.index(c)
                sub_rank = ranked({l: score(sub_mem[(c, l)]) for l in range(L) if sub_mem[(c, l)].size})
                assert [int(l) for l in sel_s[i] if l >= 0] == sub_rank[:ts]
                for l in range(L):
                    if l in sub_rank[:ts]:
                        exact += sub_mem[(c, l)].tolist()
                    elif sub_mem[(c, l)].size:
                        groups.append(sub_mem[(c, l)])
            assert rel_l2(out, mixture_ref(K, V, 64, q, exact, groups)) < 1e-12, (tc, ts)
            if tc == Cn and ts == L:
                assert rel_l2(out, dense_ref(K, V, 64, q)) < 1e-12
            cases += 1
    assert cases == (Cn + 1) * (L + 1)


def test_selection_order_and_variance_term(ora):
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    b = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    sel_c, sel_s, cs, ss = ora.select(q[0], b, 10, 6)
    order = np.lexsort((np.arange(cs.size), -cs))
    order = [i for i in order if b["cl_n"][i] > 0]
    assert np.array_equal(sel_c, order[:10])
    for i, c in enumerate(sel_c):
        sc = ss[i]
        o = [l for l in np.lexsort((np.arange(sc.size), -sc)) if b["sub_n"][c * w.n_sub + l] > 0]
        assert np.array_equal(sel_s[i][:len(o[:6])], o[:6])
    # two groups that differ only in spread along q: the wider one carries more mass
    g = np.random.default_rng(17)
    base = np.zeros((64, D))
    narrow = base + 0.05 * g.standard_normal((64, D))
    wide = base + 1.0 * g.standard_normal((64, D))
    Kx = wl.to_bf16(np.concatenate([narrow, wide]))
    Vx = wl.to_bf16(g.standard_normal((128, D)))
    bx = ora.build_unit(Kx, Vx, 128, 0, 0, 2, 1)
    if bx["cl_n"][0] == 64 and bx["cl_n"][1] == 64:
        qx = wl.to_bf16(np.full(D, 1.0))
        sc, _, cs2, _ = ora.select(qx, bx, 1, 0)
        wide_id = int(np.argmax(bx["cl_var"].sum(1)))
        assert sc[0] == wide_id
        _, _, cs1, _ = ora.select(qx, bx, 1, 0, score_mode=1)
        assert abs((cs2 - cs1)[wide_id] - (math.log(64) + 0.5 * TAU ** 2 * bx["cl_var"][wide_id].sum())) < 1e-9


def test_residual_reduces_error_on_planted_data(ora):
    """The page reports that adding the residual cuts the error of top-cluster-only
    attention; on planted-centre data it must at least reduce it."""
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    b = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    ref = dense_ref(K, V, w.n, q[0])
    mog, _, _, _ = ora.mog_head(K, V, w.n, q[0], b, w.top_c, w.top_s)
    top, _, _, _ = ora.mog_head(K, V, w.n, q[0], b, w.top_c, w.top_s, residual=False)
    assert rel_l2(mog, ref) < rel_l2(top, ref)


# ------------------------------------------------------- GQA union-exact (library variant)

def mixture_ref(K, V, n_now, q, exact, groups):
    """Exact attention over the positions `exact` plus one Gaussian term per member list
    in `groups` (count, mean, population variance and value mean taken with numpy), all
    in one softmax: an independent restatement of the residual mixture."""
    Kf, Vf, qf = f64(K), f64(V), f64(q)
    logits = [TAU * (Kf[p] @ qf) for p in exact]
    rows = [Vf[p] for p in exact]
    for mem in groups:
        X = Kf[mem]
        mu, var = X.mean(0), X.var(0)
        logits.append(math.log(len(mem)) + TAU * (qf @ mu) + 0.5 * TAU ** 2 * float(qf ** 2 @ var))
        rows.append(Vf[mem].mean(0))
    wgt = softmax(np.array(logits))
    return wgt @ np.array(rows)


def _union_case(ora, G=4, seed=0):
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    b = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    g = np.random.default_rng(seed)
    centres = f64(K[g.integers(w.n_sink, w.n - w.n_recent, G)])
    qs = wl.to_bf16(0.5 * centres + 0.5 * g.standard_normal((G, D)))
    return w, K, V, qs, b


def test_union_selection_is_the_union_of_the_heads(ora):
    w, K, V, qs, b = _union_case(ora)
    out, uc, us, sels = ora.mog_group_union(K, V, w.n, qs, b, w.top_c, w.top_s)
    want = set()
    for sel_c, sel_s in sels:
        for i, c in enumerate(sel_c):
            want |= {(int(c), int(l)) for l in sel_s[i] if c >= 0 and l >= 0}
    got = {(int(c), int(l)) for i, c in enumerate(uc) for l in us[i] if l >= 0}
    assert got == want
    assert list(uc) == sorted(set(uc.tolist())) and len(uc) > w.top_c   # heads differ


def test_union_exact_matches_independent_mixture(ora):
    """Every head attends the anchors and the union's rows exactly; the groups no head
    chose are Gaussians, checked against numpy statistics of the partition."""
    w, K, V, qs, b = _union_case(ora, seed=1)
    out, uc, us, _ = ora.mog_group_union(K, V, w.n, qs, b, w.top_c, w.top_s)
    perm, off, L = b["perm"], b["sub_off"], b["L"]
    chosen = {(int(c), int(l)) for i, c in enumerate(uc) for l in us[i] if l >= 0}
    exact = list(range(w.n_sink)) + list(range(w.n - w.n_recent, w.n))
    groups = []
    for c in range(b["C"]):
        if c in set(uc.tolist()):
            for l in range(L):
                mem = perm[off[c * L + l]:off[c * L + l + 1]]
                if (c, l) in chosen:
                    exact += mem.tolist()
                elif mem.size:
                    groups.append(mem)
        else:
            mem = perm[off[c * L]:off[(c + 1) * L]]
            if mem.size:
                groups.append(mem)
    for gq in range(len(qs)):
        assert rel_l2(out[gq], mixture_ref(K, V, w.n, qs[gq], exact, groups)) < 1e-12


def test_union_exact_with_one_head_is_the_standard_decode(ora):
    w, K, V, qs, b = _union_case(ora, G=1, seed=2)
    out, _, _, _ = ora.mog_group_union(K, V, w.n, qs, b, w.top_c, w.top_s)
    ref, _, _, _ = ora.mog_head(K, V, w.n, qs[0], b, w.top_c, w.top_s)
    assert rel_l2(out[0], ref) < 1e-14


def test_union_exact_of_identical_heads_is_the_standard_decode(ora):
    w, K, V, qs, b = _union_case(ora, G=1, seed=3)
    same = np.repeat(qs, 3, axis=0)
    out, _, _, _ = ora.mog_group_union(K, V, w.n, same, b, w.top_c, w.top_s)
    ref, _, _, _ = ora.mog_head(K, V, w.n, qs[0], b, w.top_c, w.top_s)
    for g in range(3):
        assert rel_l2(out[g], ref) < 1e-14


def test_union_exact_never_attends_fewer_rows(ora):
    """Each head's exact set grows from its own selection to the union; the error against
    dense attention is reported, and with everything chosen both are dense."""
    w, K, V, qs, b = _union_case(ora, seed=4)
    out, uc, us, sels = ora.mog_group_union(K, V, w.n, qs, b, w.top_c, w.top_s)
    n_union = ora.decode(K, V, w.n, qs[0], b, uc, us)[1][2]
    for g, (sel_c, sel_s) in enumerate(sels):
        assert ora.decode(K, V, w.n, qs[g], b, sel_c, sel_s)[1][2] <= n_union
    full, _, _, _ = ora.mog_group_union(K, V, w.n, qs, b, w.n_clusters, w.n_sub)
    for g in range(len(qs)):
        assert rel_l2(full[g], dense_ref(K, V, w.n, qs[g])) < 1e-12


# ------------------------------------------------------ sliding recent window (variant)

def _slid(ora, steps, seed=5):
    """tiny-4k built on its first 4096 - steps keys, then `steps` appends, each pushing the
    oldest recent key into the clusters."""
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    nb = w.n - steps
    b = ora.build_unit(K, V, nb, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    s, moves = b, []
    for t in range(steps):
        s, cl = ora.slide(K, V, s)
        moves.append(cl)
    return w, K, V, q, b, s, moves


def test_slide_welford_equals_two_pass_statistics(ora):
    w, K, V, q, b, s, moves = _slid(ora, 40)
    ref = ora.stats(K, V, s["perm"], s["sub_off"], s["C"], s["L"])
    for key in ("cl_n", "sub_n"):
        assert np.array_equal(s[key], ref[key])
    for key in ("cl_mu", "cl_var", "cl_vbar", "sub_mu", "sub_var", "sub_vbar"):
        err = np.abs(s[key] - ref[key]).max() / max(np.abs(ref[key]).max(), 1e-300)
        assert err < 1e-12, (key, err)
    assert s["n_build"] == b["n_build"] + 40 and s["perm"].size == b["perm"].size + 40


def test_slide_joins_the_nearest_nonempty_groups(ora):
    w, K, V, q, b, _, _ = _slid(ora, 0)
    s = b
    for t in range(12):
        p = max(s["S"], s["n_build"] - s["R"])
        x = f64(K[p:p + 1])
        full = np.nonzero(s["cl_n"] > 0)[0]
        dc = cdist(x, s["cl_mu"][full], "sqeuclidean")[0]
        c_ref = int(full[np.argmin(dc)])
        L = s["L"]
        subs = np.nonzero(s["sub_n"][c_ref * L:(c_ref + 1) * L] > 0)[0]
        ds = cdist(x, s["sub_mu"][c_ref * L + subs], "sqeuclidean")[0]
        s, (c, l) = ora.slide(K, V, s)
        assert (c, l) == (c_ref, int(subs[np.argmin(ds)]))
        g = c * L + l
        assert p in s["perm"][s["sub_off"][g]:s["sub_off"][g + 1]]
        assert p == s["perm"][s["sub_off"][g + 1] - 1]   # at the end of its subcluster's run


def test_slide_keeps_r_anchors_and_all_selected_is_dense(ora):
    w, K, V, q, b, s, _ = _slid(ora, 30)
    out, _, _, diag = ora.mog_head(K, V, w.n, q[0], s, 0, 0)       # nothing selected
    assert diag[2] == w.n_sink + w.n_recent
    full, _, _, diag = ora.mog_head(K, V, w.n, q[0], s, w.n_clusters, w.n_sub)
    assert diag[2] == w.n
    assert rel_l2(full, dense_ref(K, V, w.n, q[0])) < 1e-12


def test_slide_with_no_nonempty_cluster_is_a_no_op(ora):
    K, V, q = planted(200, seed=14)
    b = ora.build_unit(K, V, 200, 4, 196, 3, 2)       # everything is an anchor
    s, cl = ora.slide(K, V, b)
    assert cl is None and s["n_build"] == b["n_build"] and s["perm"].size == 0


# -------------------------------------------------- group-shared selection (variant)

def _log_mass_np(q, n, mu, var):
    """ln n + tau q.mu + tau^2/2 sum_j q_j^2 var_j, restated with numpy (-inf if empty)."""
    qf = f64(q)
    with np.errstate(divide="ignore"):
        return np.where(n > 0, np.log(np.maximum(n, 1)) + TAU * (mu @ qf) + 0.5 * TAU ** 2 * (var @ qf ** 2),
                        -np.inf)


def test_group_selection_matches_numpy_log_sum_exp(ora):
    w, K, V, qs, b = _union_case(ora, G=4, seed=6)
    sel_c, sel_s, gc, gs = ora.group_selection(qs, b, w.top_c, w.top_s)
    Cn, L = b["C"], b["L"]
    cl = np.stack([_log_mass_np(q, b["cl_n"], b["cl_mu"], b["cl_var"]) for q in qs])
    sub = np.stack([_log_mass_np(q, b["sub_n"], b["sub_mu"], b["sub_var"]) for q in qs])
    gc_ref = np.log(np.exp(cl - cl.max(0)).sum(0)) + cl.max(0)
    order = [c for c in np.lexsort((np.arange(Cn), -gc_ref)) if b["cl_n"][c] > 0][:w.top_c]
    assert list(sel_c) == order
    np.testing.assert_allclose(gc[b["cl_n"] > 0], gc_ref[b["cl_n"] > 0], rtol=1e-12, atol=1e-9)
    for r, c in enumerate(order):
        s = sub[:, c * L:(c + 1) * L]
        gsc = np.log(np.exp(s - s.max(0)).sum(0)) + s.max(0)
        so = [l for l in np.lexsort((np.arange(L), -gsc)) if b["sub_n"][c * L + l] > 0][:w.top_s]
        assert list(sel_s[r][:len(so)]) == so and np.all(sel_s[r][len(so):] == -1)


def test_group_shared_with_one_head_or_identical_heads_is_the_standard_decode(ora):
    w, K, V, qs, b = _union_case(ora, G=1, seed=7)
    ref, _, _, _ = ora.mog_head(K, V, w.n, qs[0], b, w.top_c, w.top_s)
    out, _, _ = ora.mog_group_shared(K, V, w.n, qs, b, w.top_c, w.top_s)
    assert rel_l2(out[0], ref) < 1e-14
    out3, _, _ = ora.mog_group_shared(K, V, w.n, np.repeat(qs, 3, axis=0), b, w.top_c, w.top_s)
    for g in range(3):
        assert rel_l2(out3[g], ref) < 1e-14


def test_group_shared_all_selected_is_dense_and_rows_are_shared(ora):
    w, K, V, qs, b = _union_case(ora, G=4, seed=8)
    out, sel_c, sel_s = ora.mog_group_shared(K, V, w.n, qs, b, w.n_clusters, w.n_sub)
    for g in range(len(qs)):
        assert rel_l2(out[g], dense_ref(K, V, w.n, qs[g])) < 1e-12
    _, sel_c, sel_s = ora.mog_group_shared(K, V, w.n, qs, b, w.top_c, w.top_s)
    n_rows = [ora.decode(K, V, w.n, q, b, sel_c, sel_s)[1][2] for q in qs]
    assert len(set(n_rows)) == 1      # every head attends the same rows


# ------------------------------------------------------------- bf16 summaries (variant)

def test_bf16_round_matches_torch_and_ties_go_to_even(ora):
    """The summaries' rounding: to float32, then to bfloat16, nearest with ties to even --
    torch's float32 -> bfloat16 conversion on the float32 value."""
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(40)
    x = np.concatenate([g.standard_normal(5000) * 10.0 ** g.integers(-6, 6, 5000), [0.0, -0.0, 1.0, -2.5]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ora.bf16_round(x), ref)
    # exact halfway cases: 1 + 2^-8 lies between 1 and 1 + 2^-7 -> even (1); 1 + 3*2^-8 -> 1 + 2^-6
    assert ora.bf16_round(1.0 + 2.0 ** -8) == 1.0
    assert ora.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6


def test_bf16_summaries_exact_when_statistics_are_representable(ora):
    """Groups of identical bf16 keys and values: every mean is a bf16 value and every
    variance is zero, so rounding changes nothing and the decode is unchanged."""
    g = np.random.default_rng(41)
    base_k = wl.to_bf16(g.standard_normal((6, D)))
    base_v = wl.to_bf16(g.standard_normal((6, D)))
    K = np.repeat(base_k, 40, axis=0)
    V = np.repeat(base_v, 40, axis=0)
    q = wl.to_bf16(g.standard_normal(D))
    b = ora.build_unit(K, V, 240, 0, 0, 6, 2)
    r = ora.summaries_bf16(b)
    for k in ("cl_mu", "cl_var", "cl_vbar", "sub_mu", "sub_var", "sub_vbar"):
        assert np.array_equal(r[k], b[k]), k
    o1, _, _, _ = ora.mog_head(K, V, 240, q, b, 2, 1)
    o2, _, _, _ = ora.mog_head(K, V, 240, q, r, 2, 1)
    assert np.array_equal(o1, o2)


def test_bf16_summaries_decode_matches_independent_mixture(ora):
    """Decode on the rounded summaries, against a numpy restatement of the mixture whose
    group statistics are rounded by torch (float32 -> bfloat16), with selection by brute
    force on the rounded scores."""
    torch = pytest.importorskip("torch")
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    b = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    r = ora.summaries_bf16(b)
    out, sel_c, sel_s, _ = ora.mog_head(K, V, w.n, q[0], r, w.top_c, w.top_s)
    tq = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    Kf, Vf, qf = f64(K), f64(V), f64(q[0])
    perm, off, L = b["perm"], b["sub_off"], w.n_sub

    def gstats(mem):
        X = Kf[mem]
        return tq(X.mean(0)), tq(X.var(0)), tq(Vf[mem].mean(0))

    def score(mu, var, n):
        return math.log(n) + TAU * (qf @ mu) + 0.5 * TAU ** 2 * float(qf ** 2 @ var)

    cl = {c: perm[off[c * L]:off[(c + 1) * L]] for c in range(w.n_clusters)}
    cs = {c: score(*gstats(m)[:2], m.size) for c, m in cl.items() if m.size}
    chosen = [c for _, c in sorted((-v, c) for c, v in cs.items())][:w.top_c]
    assert [int(c) for c in sel_c if c >= 0] == chosen
    logits = [TAU * (Kf[p] @ qf) for p in list(range(w.n_sink)) + list(range(w.n - w.n_recent, w.n))]
    rows = [Vf[p] for p in list(range(w.n_sink)) + list(range(w.n - w.n_recent, w.n))]
    for c in range(w.n_clusters):
        if c not in chosen:
            if cl[c].size:
                mu, var, vb = gstats(cl[c])
                logits.append(score(mu, var, cl[c].size))
                rows.append(vb)
            continue
        subs = {l: perm[off[c * L + l]:off[c * L + l + 1]] for l in range(L)}
        ss = {l: score(*gstats(m)[:2], m.size) for l, m in subs.items() if m.size}
        top = [l for _, l in sorted((-v, l) for l, v in ss.items())][:w.top_s]
        assert [int(l) for l in sel_s[chosen.index(c)] if l >= 0] == top
        for l, m in subs.items():
            if l in top:
                logits += [TAU * (Kf[p] @ qf) for p in m]
                rows += [Vf[p] for p in m]
            elif m.size:
                mu, var, vb = gstats(m)
                logits.append(score(mu, var, m.size))
                rows.append(vb)
    ref = softmax(np.array(logits)) @ np.array(rows)
    assert rel_l2(out, ref) < 1e-12
    full, _, _, _ = ora.mog_head(K, V, w.n, q[0], b, w.top_c, w.top_s)
    print("bf16 summaries vs fp64 summaries, rel-L2", rel_l2(out, full))


# -------------------------------------------------------------- fp8 summaries (variant)

def test_fp8_round_matches_torch_e4m3_and_saturates(ora):
    """The fp8 summaries' rounding: float32, then e4m3 to nearest with ties to even --
    torch's float32 -> float8_e4m3fn conversion on in-range values, subnormals included --
    and saturation at +-448 beyond the range."""
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(42)
    x = np.concatenate([g.standard_normal(4000) * 2.0 ** g.integers(-11, 8, 4000), [0.0, 1.0, -3.3]])
    x = x[np.abs(x) <= 440.0]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ora.fp8_round(x), ref)
    assert ora.fp8_round(1.0625) == 1.0 and ora.fp8_round(1.1875) == 1.25       # ties to even
    assert ora.fp8_round(2.0 ** -10) == 0.0 and ora.fp8_round(3 * 2.0 ** -10) == 2.0 ** -8
    assert ora.fp8_round(1000.0) == 448.0 and ora.fp8_round(-470.0) == -448.0


def test_fp8_summaries_decode_matches_independent_mixture(ora):
    """Decode on the fp8-rounded summaries against the numpy mixture with statistics rounded
    by torch's e4m3 conversion, and a brute-force selection on the rounded scores."""
    torch = pytest.importorskip("torch")
    w = wl.WORKLOADS["tiny-4k"]
    K, V, q = wl.make_unit(w)
    b = ora.build_unit(K, V, w.n, w.n_sink, w.n_recent, w.n_clusters, w.n_sub)
    r = ora.summaries_fp8(b)
    out, sel_c, sel_s, _ = ora.mog_head(K, V, w.n, q[0], r, w.top_c, w.top_s)
    tq = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    Kf, Vf, qf = f64(K), f64(V), f64(q[0])
    perm, off, L = b["perm"], b["sub_off"], w.n_sub

    def gstats(mem):
        X = Kf[mem]
        return tq(X.mean(0)), tq(X.var(0)), tq(Vf[mem].mean(0))

    def score(mu, var, n):
        return math.log(n) + TAU * (qf @ mu) + 0.5 * TAU ** 2 * float(qf ** 2 @ var)

    cl = {c: perm[off[c * L]:off[(c + 1) * L]] for c in range(w.n_clusters)}
    cs = {c: score(*gstats(m)[:2], m.size) for c, m in cl.items() if m.size}
    chosen = [c for _, c in sorted((-v, c) for c, v in cs.items())][:w.top_c]
    assert [int(c) for c in sel_c if c >= 0] == chosen
    anchors = list(range(w.n_sink)) + list(range(w.n - w.n_recent, w.n))
    logits = [TAU * (Kf[p] @ qf) for p in anchors]
    rows = [Vf[p] for p in anchors]
    for c in range(w.n_clusters):
        if c not in chosen:
            if cl[c].size:
                mu, var, vb = gstats(cl[c])
                logits.append(score(mu, var, cl[c].size))
                rows.append(vb)
            continue
        subs = {l: perm[off[c * L + l]:off[c * L + l + 1]] for l in range(L)}
        ss = {l: score(*gstats(m)[:2], m.size) for l, m in subs.items() if m.size}
        top = [l for _, l in sorted((-v, l) for l, v in ss.items())][:w.top_s]
        assert [int(l) for l in sel_s[chosen.index(c)] if l >= 0] == top
        for l, m in subs.items():
            if l in top:
                logits += [TAU * (Kf[p] @ qf) for p in m]
                rows += [Vf[p] for p in m]
            elif m.size:
                mu, var, vb = gstats(m)
                logits.append(score(mu, var, m.size))
                rows.append(vb)
    assert rel_l2(out, softmax(np.array(logits)) @ np.array(rows)) < 1e-12
