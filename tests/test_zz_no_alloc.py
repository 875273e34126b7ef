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


_RESET_SCRIPT = r'''
import ctypes as C, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import serving_mog_decode_gb300 as mog
from serving_mog_decode_gb300 import workloads as wl

lib = mog.lib()
rt = C.CDLL("libcudart.so.13")   # the runtime libmog.so was linked against (already loaded)
D, lens, h_kv, G = 128, (2000, 777), 2, 4
w = wl.Workload("noalloc-reset", batch=2, h_kv=h_kv, h_q=h_kv * G, n=max(lens), centres=32, seed=5)
K = np.zeros((2, h_kv, max(lens), D), np.uint16)
V = np.zeros_like(K)
q = np.zeros((2, h_kv * G, D), np.uint16)
for b, n in enumerate(lens):
    for h in range(h_kv):
        u = wl.UnitDraw(w, b, h, n)
        u.keys_values(K[b, h], V[b, h])
        q[b, h * G:(h + 1) * G] = u.q
ln = np.array(lens, np.int32)
H2D, D2H = 1, 2

def dev(a):
    p = C.c_void_p()
    assert rt.cudaMalloc(C.byref(p), C.c_size_t(a.nbytes)) == 0
    assert rt.cudaMemcpy(p, a.ctypes.data_as(C.c_void_p), C.c_size_t(a.nbytes), H2D) == 0
    return p

def run(noalloc):
    kp, vp, qp, lp = dev(K), dev(V), dev(q), dev(ln)
    out = np.zeros((2, h_kv * G, D), np.float32)
    op = dev(out)
    kv = mog.KV(kp.value, vp.value, K.strides[0] // 2, K.strides[1] // 2, K.strides[2] // 2)
    if noalloc:
        rc = lib.dense_decode_noalloc(C.byref(kv), lp, max(lens), 2, h_kv, h_kv * G, D, qp, op, None)
    else:
        need = C.c_size_t()
        assert lib.dense_decode_scratch_bytes(2, h_kv, h_kv * G, D, max(lens), C.byref(need)) == 0
        sp = C.c_void_p()
        assert rt.cudaMalloc(C.byref(sp), need) == 0
        rc = lib.dense_decode(C.byref(kv), lp, max(lens), 2, h_kv, h_kv * G, D, qp, op, sp, need, None)
    assert rc == 0, rc
    assert rt.cudaDeviceSynchronize() == 0
    assert rt.cudaMemcpy(out.ctypes.data_as(C.c_void_p), op, C.c_size_t(out.nbytes), D2H) == 0
    return out.astype(np.float64)

def check(o, r):
    err = np.linalg.norm(o - r, axis=-1) / np.linalg.norm(r, axis=-1)
    assert err.max() <= 1e-3, err.max()

assert rt.cudaSetDevice(0) == 0
ref = run(False)
check(run(True), ref)
assert rt.cudaDeviceReset() == 0       # ends this process's context; a new one follows
assert rt.cudaSetDevice(0) == 0
check(run(True), ref)
check(run(True), ref)
print("RESET_OK")
'''


def test_noalloc_after_device_reset():
    """The static array's device address belongs to one CUDA context.  After
    cudaDeviceReset the next call runs in a new context and must look the address up
    again.  Run in a child process (plain CUDA runtime calls, no torch), so that the reset
    does not touch this process's context."""
    import os
    import subprocess
    import sys
    buildlib.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _RESET_SCRIPT, root], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "RESET_OK" in r.stdout, r.stdout + r.stderr
