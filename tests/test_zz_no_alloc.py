"""dense_decode_noalloc: the variant of dense_decode for callers that cannot allocate
device memory (for instance a serving engine that gave its whole device budget to a
preallocated KV pool).  Its scratch is a static device array inside the library.  Checked
against dense_decode (which takes caller-allocated scratch) on two calls in a row, so that
leftover contents of the shared array from the first call cannot leak into the second.
This file is collected last on purpose."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import serving_mog_decode_gb300 as mog
from serving_mog_decode_gb300 import buildlib
from serving_mog_decode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
D = 128
TOL = 1e-3


def _batch(lens, h_kv, G, seed):
    w = wl.Workload("noalloc", batch=len(lens), h_kv=h_kv, h_q=h_kv * G, n=max(lens), centres=64,
                    seed=seed)
    n_cap = max(lens) + 5
    K = np.zeros((len(lens), h_kv, n_cap, D), np.uint16)
    V = np.zeros_like(K)
    q = np.zeros((len(lens), h_kv * G, D), np.uint16)
    for b, n in enumerate(lens):
        for h in range(h_kv):
            u = wl.UnitDraw(w, b, h, n)
            u.keys_values(K[b, h], V[b, h])
            q[b, h * G:(h + 1) * G] = u.q

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    return bf(K), bf(V), bf(q), torch.tensor(lens, dtype=torch.int32, device="cuda")


def test_noalloc_matches_dense_decode_twice():
    buildlib.build()
    calls = [((3000, 1777), 2, 4, 1), ((513, 9000, 64), 3, 5, 2)]   # two different shapes
    for lens, h_kv, G, seed in calls:
        K, V, q, ld = _batch(lens, h_kv, G, seed)
        ref = mog.dense_decode(K, V, ld, max(lens), q)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        mog.dense_decode_noalloc(K, V, ld, max(lens), q, out)
        torch.cuda.synchronize()
        r, o = ref.double().cpu().numpy(), out.double().cpu().numpy()
        for b in range(len(lens)):
            for h in range(q.shape[1]):
                err = np.linalg.norm(o[b, h] - r[b, h]) / np.linalg.norm(r[b, h])
                assert err <= TOL, (lens, b, h, err)


def test_noalloc_rejects_shapes_beyond_its_array():
    buildlib.build()
    K, V, q, ld = _batch((256,), 1, 1, 3)
    big_units = 4096            # 4096 KV heads x 16 query heads of partials exceed 4 MiB
    kv = mog._kv(K, V)
    out = torch.empty((1, 16, D), dtype=torch.float32, device="cuda")
    rc = mog.lib().dense_decode_noalloc(mog.C.byref(kv), mog._ptr(ld), 1 << 20, 1, big_units,
                                        big_units * 16, 128, mog._ptr(q), mog._ptr(out), None)
    assert rc == 8   # MOG_ERR_CAPACITY, before any launch
    assert b"static array" in mog.lib().mog_last_error()
