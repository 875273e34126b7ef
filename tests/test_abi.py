"""Host-side checks of the C ABI: the library builds for sm_103a, loads, exports every
function declared in include/mog.h, and rejects bad arguments before touching the GPU."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import serving_mog_decode_gb300 as mog
from serving_mog_decode_gb300 import buildlib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    buildlib.build()
    return mog.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mog.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)
    return sorted({n for n in names if n.startswith(("mog_", "dense_decode"))})


def test_every_declared_symbol_is_exported(lib):
    decl = declared_functions()
    assert len(decl) >= 18
    for name in decl:
        assert hasattr(lib, name), name
    assert set(decl) == set(mog.exported_symbols())


def test_status_strings(lib):
    assert lib.mog_status_string(0) == b"MOG_OK"
    assert lib.mog_status_string(3) == b"MOG_ERR_ARENA_TOO_SMALL"
    assert lib.mog_status_string(99) == b"MOG_UNKNOWN_STATUS"


def test_arena_size_query_and_validation(lib):
    p = mog.make_params(1, 8, 32, 32768, n_clusters=181, n_sub=15, top_c=8, top_s=8)
    n = mog.arena_bytes(p, [32768])
    assert n > 32768 * 8 * 4 * 4       # perm, l1 assignment, rows, ... per unit
    with pytest.raises(mog.MogError, match="SHAPE"):
        mog.arena_bytes(mog.make_params(1, 8, 30, 100), [100])          # 30 % 8 != 0
    with pytest.raises(mog.MogError, match="SHAPE"):
        mog.arena_bytes(mog.make_params(1, 1, 1, 100, d=64), [100])
    with pytest.raises(mog.MogError, match="SHAPE"):
        mog.arena_bytes(mog.make_params(1, 1, 1, 100), [101])            # longer than n_cap
    with pytest.raises(mog.MogError, match="SHAPE"):
        mog.arena_bytes(mog.make_params(1, 1, 1, 100, n_sub=33), [100])  # L > 32
    with pytest.raises(mog.MogError, match="INVALID_ARG"):
        mog.arena_bytes(mog.make_params(1, 1, 1, 100, top_c=-1), [100])
    # flags: the union-exact, sliding, group-select, bf16- and fp8-summary and k-means++ bits are the only ones defined
    u = mog.make_params(1, 8, 32, 32768, n_clusters=181, n_sub=15, top_c=8, top_s=8, union_exact=1)
    assert u.flags == mog.FLAG_UNION_EXACT and mog.arena_bytes(u, [32768]) == n
    assert mog.make_params(1, 1, 1, 100, sliding=1).flags == mog.FLAG_SLIDING
    assert mog.make_params(1, 1, 1, 100, group_select=1).flags == mog.FLAG_GROUP_SELECT
    bf = mog.make_params(1, 8, 32, 32768, n_clusters=181, n_sub=15, top_c=8, top_s=8, bf16_summaries=1)
    assert bf.flags == mog.FLAG_BF16_SUMMARIES and mog.arena_bytes(bf, [32768]) > n  # + the bf16 copies
    f8 = mog.make_params(1, 8, 32, 32768, n_clusters=181, n_sub=15, top_c=8, top_s=8, fp8_summaries=1)
    nb, n8 = mog.arena_bytes(bf, [32768]), mog.arena_bytes(f8, [32768])
    assert f8.flags == mog.FLAG_FP8_SUMMARIES and n < n8 < nb  # + the e4m3 copies, half the bf16 ones
    both = mog.make_params(1, 1, 1, 100, bf16_summaries=1, fp8_summaries=1)  # one rounding at most
    with pytest.raises(mog.MogError, match="INVALID_ARG"):
        mog.arena_bytes(both, [100])
    # the feature-map residual: accepted alone, refused with union-exact or sliding
    assert mog.arena_bytes(mog.make_params(1, 8, 32, 32768, n_clusters=181, n_sub=15, top_c=8, top_s=8,
                                           residual=2), [32768]) > n
    for kw in (dict(union_exact=1), dict(sliding=1)):
        with pytest.raises(mog.MogError, match="INVALID_ARG"):
            mog.arena_bytes(mog.make_params(1, 1, 1, 100, residual=2, **kw), [100])
    with pytest.raises(mog.MogError, match="INVALID_ARG"):
        mog.arena_bytes(mog.make_params(1, 1, 1, 100, residual=3), [100])
    u.flags = 64
    with pytest.raises(mog.MogError, match="INVALID_ARG"):
        mog.arena_bytes(u, [32768])
    # automatic C and L follow round(sqrt N) and ceil(log2 N)
    a = mog.arena_bytes(mog.make_params(2, 1, 1, 70000), [65536, 16384])
    b = mog.arena_bytes(mog.make_params(2, 1, 1, 70000, n_clusters=256, n_sub=16), [65536, 16384])
    assert a == b


def test_null_arguments_are_rejected_before_any_gpu_work(lib):
    p = mog.make_params(1, 1, 1, 128)
    lens = np.array([128], np.int32)
    out = C.c_void_p()
    rc = lib.mog_build(None, None, lens.ctypes.data_as(C.c_void_p), C.byref(p), None, 0, None, C.byref(out))
    assert rc == 1
    assert lib.mog_decode(None, None, None, None) == 1
    assert lib.mog_feature_map(None, None, None) == 1
    assert lib.mog_append(None, None, None, None) == 1
    # k-means++ seeding needs its draws: mog_build and mog_build_traced refuse the flag,
    # mog_build_seeded refuses it missing or the draws missing
    pk = mog.make_params(1, 1, 1, 128, kmeanspp=1)
    assert pk.flags == mog.FLAG_KMEANSPP
    lp = lens.ctypes.data_as(C.c_void_p)
    assert lib.mog_build(None, None, lp, C.byref(pk), None, 0, None, C.byref(out)) == 1
    assert lib.mog_build_traced(None, None, lp, C.byref(pk), None, 0, C.c_void_p(256), 1 << 20, None,
                                C.byref(out)) == 1
    assert lib.mog_build_seeded(None, None, lp, C.byref(pk), None, None, 0, None, 0, None, C.byref(out)) == 1
    assert lib.mog_build_seeded(None, None, lp, C.byref(p), C.c_void_p(256), None, 0, None, 0, None,
                                C.byref(out)) == 1
    sz = C.c_size_t()
    assert lib.dense_decode_scratch_bytes(1, 2, 3, 128, 100, C.byref(sz)) == 2
    assert lib.dense_decode_scratch_bytes(1, 2, 8, 128, 100, C.byref(sz)) == 0 and sz.value > 0
    assert lib.mog_kmeans_assign_scratch_bytes(10, 4, 128, C.byref(sz)) == 0
    lib.mog_destroy(None)


def test_oracle_is_not_imported_by_the_product():
    for dirpath, _, files in os.walk(os.path.join(ROOT, "serving_mog_decode_gb300")):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "mog_oracle" not in text, f
