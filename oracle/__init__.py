"""ctypes front end of the fp64 CPU oracle (``mog_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It never touches the CUDA
library and the CUDA library never touches it.

Every function takes bf16 data as ``uint16`` bit patterns and returns numpy arrays.
Summaries are returned as a dict with keys ``cl_n, cl_mu, cl_var, cl_vbar, sub_n,
sub_mu, sub_var, sub_vbar`` (counts int32, the rest float64, shapes ``[C]``,
``[C, d]``, ``[C*L]``, ``[C*L, d]``).
"""
from __future__ import annotations

import ctypes as C
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mog_oracle.c")
_LIB = os.path.join(_HERE, "libmog_oracle.so")

_i64 = C.c_int64
_dbl = C.c_double
_p = C.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off, OpenMP on)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
            "-o", tmp, _SRC, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        l = C.CDLL(_LIB)
        for name in ("ora_assign", "ora_update", "ora_lloyd", "ora_stats", "ora_build",
                     "ora_select", "ora_decode", "ora_dense", "ora_pp_pick", "ora_kmeanspp",
                     "ora_decode_fm", "ora_fm_sums"):
            getattr(l, name).restype = C.c_int
        _lib = l
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are uint16 bit patterns")
    return a


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"oracle {name} failed with code {rc}")


def tau_of(d: int) -> float:
    return 1.0 / math.sqrt(d)


def assign(x: np.ndarray, cent: np.ndarray, rows=None) -> np.ndarray:
    """Nearest centroid (canonical fp64 distance, lowest index on ties) of x[rows]."""
    x = _u16(x)
    d = x.shape[1]
    rows = np.arange(x.shape[0], dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cent = np.ascontiguousarray(cent, np.float64)
    out = np.empty(rows.shape[0], np.int32)
    _check(lib().ora_assign(_ptr(x), _i64(d), _ptr(rows), _i64(rows.shape[0]), _ptr(cent),
                            _i64(cent.shape[0]), _i64(d), _ptr(out)), "assign")
    return out


def update(x: np.ndarray, a: np.ndarray, cent: np.ndarray, rows=None) -> np.ndarray:
    """One centroid update (R6): the fp64 mean of the rows x[rows] assigned to each
    centroid by `a`; a centroid with no rows keeps its value from `cent`."""
    x = _u16(x)
    d = x.shape[1]
    rows = np.arange(x.shape[0], dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    a = np.ascontiguousarray(a, np.int32)
    if a.shape[0] != rows.shape[0]:
        raise ValueError("one assignment per row")
    out = np.array(cent, np.float64, copy=True, order="C")
    _check(lib().ora_update(_ptr(x), _i64(d), _ptr(rows), _i64(rows.shape[0]), _ptr(a),
                            _i64(out.shape[0]), _i64(d), _ptr(out)), "update")
    return out


def lloyd(x: np.ndarray, k: int, iters: int, rows=None, history: bool = False):
    """Lloyd's algorithm with strided seeding.  Returns (cent, assign, steps, hist)."""
    x = _u16(x)
    d = x.shape[1]
    rows = np.arange(x.shape[0], dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cent = np.empty((k, d), np.float64)
    asg = np.empty(rows.shape[0], np.int32)
    hist = np.zeros((iters, k, d), np.float64) if history else None
    steps = np.zeros(1, np.int64)
    _check(lib().ora_lloyd(_ptr(x), _i64(d), _ptr(rows), _i64(rows.shape[0]), _i64(k), _i64(d),
                           _i64(iters), _ptr(cent), _ptr(asg), _ptr(hist), _ptr(steps)), "lloyd")
    s = int(steps[0])
    return cent, asg, s, (hist[:s] if history else None)


def _draws(draws, k):
    u = np.ascontiguousarray(draws, np.float64).reshape(-1)
    if u.shape[0] < k:
        raise ValueError("one draw per seed")
    return u


def pp_pick(x: np.ndarray, seeds, u: float, rows=None) -> int:
    """One k-means++ step (R28): the member index of the next seed after `seeds` (member
    indices into x[rows]) for the uniform draw u."""
    x = _u16(x)
    d = x.shape[1]
    rows = np.arange(x.shape[0], dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    sd = np.ascontiguousarray(seeds, np.int64).reshape(-1)
    out = np.zeros(1, np.int64)
    _check(lib().ora_pp_pick(_ptr(x), _i64(d), _ptr(rows), _i64(rows.shape[0]), _i64(d),
                             _ptr(sd if sd.size else np.zeros(1, np.int64)), _i64(sd.size),
                             C.c_double(float(u)), _ptr(out)), "pp_pick")
    return int(out[0])


def kmeanspp(x: np.ndarray, k: int, draws, rows=None) -> np.ndarray:
    """k-means++ seeding (R28) of x[rows]: the k seeds' member indices, seed r drawn with
    draws[r]."""
    x = _u16(x)
    d = x.shape[1]
    rows = np.arange(x.shape[0], dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    u = _draws(draws, k)
    out = np.zeros(k, np.int64)
    _check(lib().ora_kmeanspp(_ptr(x), _i64(d), _ptr(rows), _i64(rows.shape[0]), _i64(k), _i64(d),
                              _ptr(u), _ptr(out)), "kmeanspp")
    return out


def _summ_buffers(Cn: int, L: int, d: int):
    return dict(
        cl_n=np.zeros(Cn, np.int32), cl_mu=np.zeros((Cn, d)), cl_var=np.zeros((Cn, d)),
        cl_vbar=np.zeros((Cn, d)), sub_n=np.zeros(Cn * L, np.int32),
        sub_mu=np.zeros((Cn * L, d)), sub_var=np.zeros((Cn * L, d)), sub_vbar=np.zeros((Cn * L, d)),
    )


def _summ_args(s):
    return [_ptr(s[k]) for k in ("cl_n", "cl_mu", "cl_var", "cl_vbar", "sub_n", "sub_mu",
                                 "sub_var", "sub_vbar")]


def stats(K: np.ndarray, V: np.ndarray, perm: np.ndarray, sub_off: np.ndarray, Cn: int, L: int):
    """Gaussian summaries of a given (cluster, subcluster) partition."""
    K, V = _u16(K), _u16(V)
    d = K.shape[1]
    perm = np.ascontiguousarray(perm, np.int32)
    sub_off = np.ascontiguousarray(sub_off, np.int32)
    s = _summ_buffers(Cn, L, d)
    _check(lib().ora_stats(_ptr(K), _ptr(V), _i64(d), _i64(d), _ptr(perm), _ptr(sub_off),
                           _i64(Cn), _i64(L), *_summ_args(s)), "stats")
    return s


def build_unit(K: np.ndarray, V: np.ndarray, n_build: int, S: int, R: int, Cn: int, L: int,
               T1: int = 10, T2: int = 10, draws=None):
    """The full two-level build of one KV head.  Returns a dict with ``perm``,
    ``sub_off``, ``l1_assign``, ``steps`` and the summaries.  draws (Cn uniforms in
    [0, 1)): k-means++ seeds for the first level (R28) instead of strided ones."""
    K, V = _u16(K), _u16(V)
    d = K.shape[1]
    nm = max(0, n_build - R - S)
    s = _summ_buffers(Cn, L, d)
    perm = np.zeros(max(nm, 1), np.int32)
    sub_off = np.zeros(Cn * L + 1, np.int32)
    l1 = np.zeros(max(nm, 1), np.int32)
    steps = np.zeros(2, np.int64)
    u = None if draws is None else _draws(draws, Cn)
    _check(lib().ora_build(_ptr(K), _ptr(V), _i64(d), _i64(n_build), _i64(d), _i64(S), _i64(R),
                           _i64(Cn), _i64(L), _i64(T1), _i64(T2), _ptr(u), _ptr(perm), _ptr(sub_off),
                           *_summ_args(s), _ptr(l1), _ptr(steps)), "build")
    s.update(perm=perm[:nm], sub_off=sub_off, l1_assign=l1[:nm], steps=(int(steps[0]), int(steps[1])),
             C=Cn, L=L, n_build=n_build, S=S, R=R)
    return s


def select(q: np.ndarray, summ: dict, top_c: int, top_s: int, score_mode: int = 0):
    """Cluster and subcluster selection of one query head.
    Returns (sel_c[top_c], sel_s[top_c, top_s], cscore[C], sscore[top_c, L])."""
    q = _u16(q)
    d = q.shape[0]
    Cn, L = summ["C"], summ["L"]
    sel_c = np.zeros(max(top_c, 1), np.int32)
    sel_s = np.zeros(max(top_c * top_s, 1), np.int32)
    cs = np.zeros(max(Cn, 1))
    ss = np.zeros(max(top_c * L, 1))
    _check(lib().ora_select(_ptr(q), _i64(d), _dbl(tau_of(d)), _i64(Cn), _i64(L),
                            _ptr(summ["cl_n"]), _ptr(summ["cl_mu"]), _ptr(summ["cl_var"]),
                            _ptr(summ["sub_n"]), _ptr(summ["sub_mu"]), _ptr(summ["sub_var"]),
                            _i64(top_c), _i64(top_s), C.c_int(score_mode), _ptr(sel_c),
                            _ptr(sel_s), _ptr(cs), _ptr(ss)), "select")
    return (sel_c[:top_c], sel_s[:top_c * top_s].reshape(top_c, top_s), cs[:Cn],
            ss[:top_c * L].reshape(top_c, L))


def decode(K: np.ndarray, V: np.ndarray, n_now: int, q: np.ndarray, summ: dict,
           sel_c: np.ndarray, sel_s: np.ndarray, residual: bool = True):
    """Exact + residual output of one query head for a given selection.
    Returns (out[d], diag = (m, den, n_exact))."""
    K, V, q = _u16(K), _u16(V), _u16(q)
    d = K.shape[1]
    sel_c = np.ascontiguousarray(sel_c, np.int32).reshape(-1)
    tc = sel_c.shape[0]
    sel_s = np.ascontiguousarray(sel_s, np.int32).reshape(-1)
    ts = sel_s.shape[0] // tc if tc else 0
    out = np.zeros(d)
    diag = np.zeros(3)
    perm = np.ascontiguousarray(summ["perm"], np.int32)
    if perm.size == 0:
        perm = np.zeros(1, np.int32)
    _check(lib().ora_decode(_ptr(K), _ptr(V), _i64(d), _i64(d), _i64(n_now), _i64(summ["n_build"]),
                            _i64(summ["S"]), _i64(summ["R"]), _ptr(q), _dbl(tau_of(d)),
                            _i64(summ["C"]), _i64(summ["L"]), _ptr(perm), _ptr(summ["sub_off"]),
                            *_summ_args(summ), _ptr(sel_c if tc else np.zeros(1, np.int32)),
                            _ptr(sel_s if sel_s.size else np.zeros(1, np.int32)), _i64(tc),
                            _i64(ts), C.c_int(1 if residual else 0), _ptr(out), _ptr(diag)),
           "decode")
    return out, diag


def decode_fm(K: np.ndarray, V: np.ndarray, n_now: int, q: np.ndarray, summ: dict,
              sel_c: np.ndarray, sel_s: np.ndarray, omega: np.ndarray):
    """Decode of one query head with the feature-map residual (R29): exact attention over
    the anchors and the selected subclusters' members, the random-feature estimate with
    the rows of `omega` [m, d] for every other mid key.  Returns (out[d], diag[4])."""
    K, V, q = _u16(K), _u16(V), _u16(q)
    d = K.shape[1]
    om = np.ascontiguousarray(omega, np.float64)
    tc = int(np.asarray(sel_c).shape[0])
    ts = int(np.asarray(sel_s).reshape(tc, -1).shape[1]) if tc else 0
    sc = np.ascontiguousarray(sel_c, np.int32).reshape(-1)
    ss = np.ascontiguousarray(sel_s, np.int32).reshape(-1)
    out = np.zeros(d)
    diag = np.zeros(4)
    _check(lib().ora_decode_fm(_ptr(K), _ptr(V), _i64(d), _i64(d), _i64(n_now), _i64(summ["n_build"]),
                               _i64(summ["S"]), _i64(summ["R"]), _ptr(q), _dbl(tau_of(d)),
                               _i64(summ["C"]), _i64(summ["L"]), _ptr(summ["perm"]),
                               _ptr(summ["sub_off"]), _ptr(sc if sc.size else np.zeros(1, np.int32)),
                               _ptr(ss if ss.size else np.zeros(1, np.int32)), _i64(tc), _i64(ts),
                               _ptr(om), _i64(om.shape[0]), _ptr(out), _ptr(diag)), "decode_fm")
    return out, diag


def fm_sums(K: np.ndarray, V: np.ndarray, summ: dict, omega: np.ndarray) -> np.ndarray:
    """Unscaled feature sums of every subcluster (R29): [C*L, m, d+1], the value-weighted
    sums in [..., :d] and the plain sums in [..., d]."""
    K, V = _u16(K), _u16(V)
    d = K.shape[1]
    om = np.ascontiguousarray(omega, np.float64)
    m = om.shape[0]
    Cn, L = summ["C"], summ["L"]
    z = np.zeros((Cn * L, m, d + 1))
    _check(lib().ora_fm_sums(_ptr(K), _ptr(V), _i64(d), _i64(d), _ptr(summ["perm"]),
                             _ptr(summ["sub_off"]), _i64(Cn), _i64(L), _dbl(tau_of(d)), _ptr(om),
                             _i64(m), _ptr(z)), "fm_sums")
    return z


def dense(K: np.ndarray, V: np.ndarray, n: int, q: np.ndarray) -> np.ndarray:
    """Exact softmax attention of one query head over keys [0, n)."""
    K, V, q = _u16(K), _u16(V), _u16(q)
    d = K.shape[1]
    out = np.zeros(d)
    _check(lib().ora_dense(_ptr(K), _ptr(V), _i64(d), _i64(d), _i64(n), _ptr(q), _dbl(tau_of(d)),
                           _ptr(out)), "dense")
    return out


def mog_head(K, V, n_now, q, summ, top_c, top_s, score_mode=0, residual=True):
    """Selection then decode for one query head (the oracle's whole decode step)."""
    sel_c, sel_s, _, _ = select(q, summ, top_c, top_s, score_mode)
    out, diag = decode(K, V, n_now, q, summ, sel_c, sel_s, residual)
    return out, sel_c, sel_s, diag


def union_selection(sels, L: int):
    """Union of the choices of the query heads that share one KV head (the GQA union-exact
    variant of this library; the pages select per query head and do not define it).
    sels: (sel_c[tc], sel_s[tc, ts]) per head, as select() returns them.
    Returns (uc[U], us[U, L]): every cluster some head chose, ascending, and inside each
    every subcluster some head chose for it, ascending, -1 padded."""
    chosen = {}
    for sel_c, sel_s in sels:
        sel_s = np.asarray(sel_s).reshape(len(sel_c), -1)
        for i, c in enumerate(np.asarray(sel_c).tolist()):
            if c < 0:
                continue
            subs = chosen.setdefault(int(c), set())
            subs.update(int(l) for l in sel_s[i].tolist() if l >= 0)
    uc = np.array(sorted(chosen), np.int32)
    us = np.full((len(uc), L), -1, np.int32)
    for i, c in enumerate(uc.tolist()):
        sub = sorted(chosen[c])
        us[i, :len(sub)] = sub
    return uc, us


def mog_group_union(K, V, n_now, qs, summ, top_c, top_s, score_mode=0, residual=True):
    """GQA union-exact decode of the query heads qs[G][d] of one KV head: each head makes
    its own selection; every head then attends exactly the anchors and the members of
    every subcluster in the union of the heads' choices, and takes the Gaussian residual
    of every other non-empty group (the subclusters of union clusters outside the union,
    the clusters outside the union).  Returns (out[G][d], uc, us, per-head selections)."""
    sels = [select(q, summ, top_c, top_s, score_mode)[:2] for q in qs]
    uc, us = union_selection(sels, summ["L"])
    outs = [decode(K, V, n_now, q, summ, uc, us, residual)[0] for q in qs]
    return np.stack(outs), uc, us, sels


def slide(K: np.ndarray, V: np.ndarray, summ: dict, force=None):
    """One step of the sliding recent window (a reading of this library; the pages keep a
    recent window but do not say what happens to a key that leaves it).  The oldest recent
    key, position max(S, n_build - R), leaves the window: it joins the nearest non-empty
    cluster under the assignment rule R5 against the cluster means, then the nearest
    non-empty subcluster of that cluster against the subcluster means (or `force` =
    (c, l)), and both groups take it with Welford's update of count, mean, population
    variance and value mean.  The key goes to the end of its subcluster's run of `perm`
    and n_build advances by one, so that the recent window [n_build - R, n) keeps R keys.
    Returns (the updated copy of summ, (c, l)); (summ, None) when no cluster is non-empty."""
    s = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in summ.items()}
    S, R, Cn, L = s["S"], s["R"], s["C"], s["L"]
    p = max(S, s["n_build"] - R)
    full = np.nonzero(s["cl_n"][:Cn] > 0)[0]
    if full.size == 0:
        return s, None
    x_bf = np.ascontiguousarray(_u16(K)[p:p + 1])
    if force is None:
        c = int(full[assign(x_bf, s["cl_mu"][full])[0]])
        subs = np.nonzero(s["sub_n"][c * L:(c + 1) * L] > 0)[0]
        l = int(subs[assign(x_bf, s["sub_mu"][c * L + subs])[0]])
    else:
        c, l = int(force[0]), int(force[1])
    x = _u16(K)[p].astype(np.uint32) << 16
    v = _u16(V)[p].astype(np.uint32) << 16
    x = x.view(np.float32).astype(np.float64)
    v = v.view(np.float32).astype(np.float64)
    for cnt, mu, var, vb, i in ((s["cl_n"], s["cl_mu"], s["cl_var"], s["cl_vbar"], c),
                                (s["sub_n"], s["sub_mu"], s["sub_var"], s["sub_vbar"], c * L + l)):
        n = float(cnt[i])
        delta = x - mu[i]
        mu_new = mu[i] + delta / (n + 1.0)
        var[i] = (n * var[i] + delta * (x - mu_new)) / (n + 1.0)
        mu[i] = mu_new
        vb[i] = vb[i] + (v - vb[i]) / (n + 1.0)
        cnt[i] += 1
    g = c * L + l
    s["perm"] = np.insert(s["perm"], int(s["sub_off"][g + 1]), p).astype(np.int32)
    s["sub_off"][g + 1:] += 1
    s["n_build"] += 1
    return s, (c, l)


def bf16_round(x) -> np.ndarray:
    """x (float64) rounded to float32, then to bfloat16, each to nearest with ties to even;
    returned as float64.  (The summaries' storage path: fp32 values rounded to bf16.)"""
    f = np.ascontiguousarray(np.asarray(x, np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def summaries_bf16(summ: dict) -> dict:
    """The bf16-summary variant of this library (MOG_FLAG_BF16_SUMMARIES; the pages do not
    fix the summaries' precision): every group's key mean, per-dimension variance and value
    mean rounded as bf16_round does; counts, partition and everything else unchanged.
    Selection and decode on the returned dict are the method on the rounded summaries."""
    s = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in summ.items()}
    for k in ("cl_mu", "cl_var", "cl_vbar", "sub_mu", "sub_var", "sub_vbar"):
        s[k] = bf16_round(s[k])
    return s


def fp8_round(x) -> np.ndarray:
    """x (float64) rounded to float32, then to fp8 e4m3 (3 mantissa bits, exponents -6..8,
    subnormal steps of 2^-9), to nearest with ties to even, saturating at +-448; returned as
    float64."""
    f = np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
    a = np.minimum(np.abs(f), 448.0)
    e = np.clip(np.floor(np.log2(np.maximum(a, 2.0 ** -9))), -6, 8)
    step = 2.0 ** (e - 3)
    r = np.minimum(np.round(a / step) * step, 448.0)   # np.round: half to even
    return np.copysign(r, f)


def summaries_fp8(summ: dict) -> dict:
    """The fp8-summary variant of this library (MOG_FLAG_FP8_SUMMARIES; the pages do not
    fix the summaries' precision): every group's key mean, per-dimension variance and value
    mean rounded as fp8_round does; counts, partition and everything else unchanged."""
    s = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in summ.items()}
    for k in ("cl_mu", "cl_var", "cl_vbar", "sub_mu", "sub_var", "sub_vbar"):
        s[k] = fp8_round(s[k])
    return s


def group_selection(qs, summ: dict, top_c: int, top_s: int, score_mode: int = 0):
    """Group-shared selection (a variant of this library; the pages select per query head):
    the query heads qs[G][d] of one KV head select once.  A group's score is the log of the
    sum over the heads of exp(its per-head selection score) -- the log of the group's total
    estimated attention mass -- and the top_c clusters, then the top_s subclusters inside
    each, are taken by that score (descending, index ascending, empty groups never).
    Returns (sel_c[top_c], sel_s[top_c, top_s], group cluster scores[C], group subcluster
    scores[C, L]), -1 padded."""
    Cn, L = summ["C"], summ["L"]
    cl = np.full((len(qs), Cn), -np.inf)
    sub = np.full((len(qs), Cn, L), -np.inf)
    for g, q in enumerate(qs):  # every head's scores of every group
        sc_all, _, cs, ss = select(q, summ, Cn, L, score_mode)
        cl[g] = cs
        for i, c in enumerate(sc_all):
            if c >= 0:
                sub[g, c] = ss[i]
    with np.errstate(invalid="ignore"):
        gc = np.logaddexp.reduce(cl, axis=0)
        gs = np.logaddexp.reduce(sub, axis=0)
    sel_c = np.full(max(top_c, 1), -1, np.int32)
    sel_s = np.full((max(top_c, 1), max(top_s, 1)), -1, np.int32)
    order = [int(i) for i in np.lexsort((np.arange(Cn), -gc)) if np.isfinite(gc[i]) and summ["cl_n"][i] > 0]
    for r, c in enumerate(order[:top_c]):
        sel_c[r] = c
        so = [int(l) for l in np.lexsort((np.arange(L), -gs[c])) if np.isfinite(gs[c, l])
              and summ["sub_n"][c * L + l] > 0]
        sel_s[r, :len(so[:top_s])] = so[:top_s]
    return sel_c[:top_c], sel_s[:top_c, :top_s], gc, gs


def mog_group_shared(K, V, n_now, qs, summ, top_c, top_s, score_mode=0, residual=True):
    """Group-shared decode: every head attends exactly the anchors and the rows of the
    group's selection, and takes its own Gaussian residual of every other non-empty group.
    Returns (out[G][d], sel_c, sel_s)."""
    sel_c, sel_s, _, _ = group_selection(qs, summ, top_c, top_s, score_mode)
    outs = [decode(K, V, n_now, q, summ, sel_c, sel_s, residual)[0] for q in qs]
    return np.stack(outs), sel_c, sel_s
