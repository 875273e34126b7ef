"""Mixture-of-Gaussians (MoG) decode attention for NVIDIA GB300.

A thin ctypes binding of ``libmog.so`` (the CUDA kernels and the C ABI in
``include/mog.h``).  This module only marshals arguments: device memory comes from
PyTorch tensors, streams from ``torch.cuda.current_stream()``, and every step of the
build and decode runs in the library's kernels.  There is no CPU fallback: if the
library is missing or fails to load, every call raises.

Sources: "Iceberg Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians"
(Abstract) and the newx.sg page on retrieval-completion attention (Abstract).
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmog.so")

MOG_OK = 0
FLAG_UNION_EXACT = 1  # MOG_FLAG_UNION_EXACT in mog.h
FLAG_SLIDING = 2      # MOG_FLAG_SLIDING in mog.h
FLAG_GROUP_SELECT = 4  # MOG_FLAG_GROUP_SELECT in mog.h
FLAG_BF16_SUMMARIES = 8  # MOG_FLAG_BF16_SUMMARIES in mog.h
FLAG_FP8_SUMMARIES = 16  # MOG_FLAG_FP8_SUMMARIES in mog.h
FLAG_KMEANSPP = 32       # MOG_FLAG_KMEANSPP in mog.h
RESIDUAL_FEATURE_MAP = 2  # MOG_RESIDUAL_FEATURE_MAP in mog.h
FM_FEATURES = 32          # MOG_FM_FEATURES in mog.h
STATUS = ["MOG_OK", "MOG_ERR_INVALID_ARG", "MOG_ERR_SHAPE", "MOG_ERR_ARENA_TOO_SMALL",
          "MOG_ERR_CUDA", "MOG_ERR_DEVICE_CHECK", "MOG_ERR_TIMEOUT", "MOG_ERR_NOT_IMPLEMENTED",
          "MOG_ERR_CAPACITY"]


class MogError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        name = STATUS[code] if 0 <= code < len(STATUS) else f"status {code}"
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


class Params(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "batch", "h_kv", "h_q", "d", "n_cap", "n_clusters", "n_sub", "top_c", "top_s",
        "n_sink", "n_recent", "iters_l1", "iters_l2", "score_mode", "residual", "flags")]


class KV(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("stride_b", C.c_int64),
                ("stride_h", C.c_int64), ("stride_n", C.c_int64), ("block_table", C.c_void_p),
                ("page_rows", C.c_int32), ("pages_per_seq", C.c_int32)]


class PagedKV:
    """A paged bf16 KV cache: page pools K, V of shape [pages, H_kv, page_rows, d]
    (heads_first) or [pages, page_rows, H_kv, d], and an int32 block table [B, pages_per_seq]
    on the device (page of position n of sequence b: block_table[b, n // page_rows]).
    Pass it as K (with V=None) wherever a cache is taken."""

    def __init__(self, K, V, block_table, page_rows, heads_first=True):
        torch = _torch()
        for t in (K, V):
            if t.dtype != torch.bfloat16 or t.dim() != 4 or t.stride(3) != 1 or not t.is_cuda:
                raise ValueError("page pools must be CUDA bf16 tensors with 4 dims, last contiguous")
        if K.shape != V.shape or K.stride() != V.stride():
            raise ValueError("K and V pools must share shape and strides")
        if block_table.dtype != torch.int32 or block_table.dim() != 2 or not block_table.is_contiguous():
            raise ValueError("block_table must be a contiguous int32 tensor [B, pages_per_seq]")
        self.K, self.V, self.block_table, self.page_rows = K, V, block_table, page_rows
        self.heads_first = heads_first
        self.h_kv = K.shape[1] if heads_first else K.shape[2]
        self.device = K.device

    def struct(self) -> KV:
        K = self.K
        sh, sn = (K.stride(1), K.stride(2)) if self.heads_first else (K.stride(2), K.stride(1))
        return KV(K.data_ptr(), self.V.data_ptr(), K.stride(0), sh, sn, self.block_table.data_ptr(),
                  self.page_rows, self.block_table.shape[1])


class Layout(C.Structure):
    _fields_ = ([(n, C.c_int32) for n in ("units", "c_max", "l_max", "n_cap", "d", "group",
                                           "top_c", "top_s")] +
                [(n, C.c_int64) for n in ("unit_info", "n_now", "perm", "sub_off",
                                           "sub_off_stride", "cl_n", "cl_ms", "cl_vbar", "sub_n",
                                           "sub_ms", "sub_vbar", "l1_assign", "status",
                                           "l1_steps", "fallback", "cl_ms16", "sub_ms16", "cl_ms8",
                                           "sub_ms8", "pp_idx", "fm_z", "fm_t")])


class TraceLayout(C.Structure):
    _fields_ = ([(n, C.c_int32) for n in ("units", "iters_l1", "iters_l2", "c_max", "l_max", "d")] +
                [(n, C.c_int64) for n in ("n_mid", "l1_cent", "l1_assign", "l2_cent", "l2_assign",
                                           "l2_steps", "bytes")])


_lib = None
_P = C.c_void_p
_SIGS = {
    "mog_status_string": (C.c_char_p, [C.c_int]),
    "mog_last_error": (C.c_char_p, []),
    "mog_arena_bytes": (C.c_int, [_P, _P, _P]),
    "mog_build": (C.c_int, [_P, _P, _P, _P, _P, C.c_size_t, _P, _P]),
    "mog_build_from_partition": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P, _P]),
    "mog_sub_off_stride": (C.c_int, [_P, _P, _P]),
    "mog_trace_layout_of": (C.c_int, [_P, _P, _P]),
    "mog_build_traced": (C.c_int, [_P, _P, _P, _P, _P, C.c_size_t, _P, C.c_size_t, _P, _P]),
    "mog_build_seeded": (C.c_int, [_P, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_size_t, _P, _P]),
    "mog_decode": (C.c_int, [_P, _P, _P, _P]),
    "mog_decode_ex": (C.c_int, [_P, _P, _P, _P, _P, _P]),
    "mog_decode_phased": (C.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    "mog_append": (C.c_int, [_P, _P, _P, _P]),
    "mog_recluster": (C.c_int, [_P, _P]),
    "mog_feature_map": (C.c_int, [_P, _P, _P]),
    "mog_get_layout": (C.c_int, [_P, _P]),
    "mog_sync_status": (C.c_int, [_P, _P]),
    "mog_decode_splits": (C.c_int, [_P, _P]),
    "mog_destroy": (None, [_P]),
    "dense_decode_scratch_bytes": (C.c_int, [C.c_int32] * 5 + [_P]),
    "dense_decode": (C.c_int, [_P, _P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                               _P, _P, _P, C.c_size_t, _P]),
    "dense_decode_noalloc": (C.c_int, [_P, _P, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                       C.c_int32, _P, _P, _P]),
    "mog_kmeans_assign_scratch_bytes": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, _P]),
    "mog_kmeans_assign": (C.c_int, [_P, C.c_int64, C.c_int32, _P, C.c_int32, C.c_int32, _P, _P,
                                    C.c_size_t, _P, _P]),
    "mog_kmeans_assign_segments": (C.c_int, [_P, C.c_int64, _P, _P, C.c_int32, _P, C.c_int32,
                                             C.c_int32, _P, _P]),
    "mog_check_bounded_wait": (C.c_int, [C.c_int32, C.c_int32, _P, _P]),
}


def lib():
    """Load libmog.so (built in-tree by ``build.py``).  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmog.so is not built ({LIB_PATH}); run "
                               "`python -m serving_mog_decode_gb300.build` first")
        l = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(rc: int, where: str):
    if rc != MOG_OK:
        detail = lib().mog_last_error().decode() if rc == 4 else ""
        raise MogError(rc, where, detail)


def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _kv(K, V):
    """KV descriptor of bf16 tensors [B, H_kv, n_cap, d] (last dim contiguous), or of a
    PagedKV passed as K."""
    if isinstance(K, PagedKV):
        return K.struct()
    torch = _torch()
    for t in (K, V):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.stride(3) != 1 or not t.is_cuda:
            raise ValueError("K and V must be CUDA bf16 tensors [B, H_kv, n_cap, d], last dim contiguous")
    if K.stride() != V.stride() or K.shape != V.shape:
        raise ValueError("K and V must share shape and strides")
    return KV(K.data_ptr(), V.data_ptr(), K.stride(0), K.stride(1), K.stride(2))


def make_params(batch, h_kv, h_q, n_cap, *, d=128, n_clusters=0, n_sub=0, top_c=8, top_s=8,
                n_sink=4, n_recent=256, iters_l1=10, iters_l2=10, score_mode=0, residual=1,
                union_exact=0, sliding=0, group_select=0, bf16_summaries=0, fp8_summaries=0,
                kmeanspp=0):
    """mog_params for a batch of `batch` sequences with h_kv KV heads and h_q query heads
    (d = 128), a KV cache of n_cap positions.  n_clusters / n_sub = 0 pick round(sqrt N)
    and ceil(log2 N) per sequence; top_c clusters and top_s subclusters per chosen cluster
    are attended exactly, with n_sink sink and n_recent recent anchors.  The flags select
    the variants: union_exact (every head of a KV group attends the union of the group's
    chosen rows), sliding (a fixed recent window whose leaving keys join the clusters),
    group_select (one selection per KV group by the log-sum-exp of its heads' scores),
    bf16_summaries or fp8_summaries (scores and residual terms from the summaries rounded to
    bf16, or to fp8 e4m3; not both), kmeanspp (first-level k-means++ seeds; build() then
    needs the draws)."""
    return Params(batch, h_kv, h_q, d, n_cap, n_clusters, n_sub, top_c, top_s, n_sink,
                  n_recent, iters_l1, iters_l2, score_mode, residual,
                  (FLAG_UNION_EXACT if union_exact else 0) | (FLAG_SLIDING if sliding else 0)
                  | (FLAG_GROUP_SELECT if group_select else 0)
                  | (FLAG_BF16_SUMMARIES if bf16_summaries else 0)
                  | (FLAG_FP8_SUMMARIES if fp8_summaries else 0)
                  | (FLAG_KMEANSPP if kmeanspp else 0))


def arena_bytes(params: Params, lengths_host) -> int:
    import numpy as np
    lh = np.ascontiguousarray(lengths_host, np.int32)
    out = C.c_size_t(0)
    _check(lib().mog_arena_bytes(C.byref(params), lh.ctypes.data_as(_P), C.byref(out)),
           "mog_arena_bytes")
    return out.value


class Handle:
    """A built MoG index over a KV cache.  Owns (references) the arena tensor; the KV
    tensors must stay alive and unmoved while the handle is used."""

    def __init__(self, ptr, arena, params, K, V, lengths_dev, lengths_host):  # K may be a PagedKV
        self._h = ptr
        self.arena = arena
        self.params = params
        self.K, self.V = K, V
        self.lengths_dev = lengths_dev
        self.lengths_host = lengths_host

    def __del__(self):
        if getattr(self, "_h", None):
            try:
                lib().mog_destroy(self._h)
            except Exception:
                pass
            self._h = None

    @property
    def group(self):
        return self.params.h_q // self.params.h_kv

    def decode(self, q, out=None, sel_in=None, sel_out=None, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if sel_in is None and sel_out is None:
            rc = lib().mog_decode(self._h, _ptr(q), _ptr(out), _stream(stream))
        else:
            rc = lib().mog_decode_ex(self._h, _ptr(q), _ptr(out), _ptr(sel_in), _ptr(sel_out),
                                     _stream(stream))
        _check(rc, "mog_decode")
        return out

    def decode_phased(self, q, out, events, sel_out=None, stream=None):
        """Decode with four torch.cuda.Event objects recorded around the three kernels."""
        for e in events:       # torch creates the CUDA event on first record
            if not e.cuda_event:
                e.record()
        arr = (C.c_void_p * 4)(*[e.cuda_event for e in events])
        _check(lib().mog_decode_phased(self._h, _ptr(q), _ptr(out), None, _ptr(sel_out), arr,
                                       _stream(stream)), "mog_decode_phased")
        return out

    def append(self, k_new, v_new, stream=None):
        _check(lib().mog_append(self._h, _ptr(k_new), _ptr(v_new), _stream(stream)), "mog_append")

    def recluster(self, stream=None):
        """Rebuild the partition and summaries over the grown sequences (mog_recluster)."""
        _check(lib().mog_recluster(self._h, _stream(stream)), "mog_recluster")

    def feature_map(self, omega, stream=None):
        """The feature-map summary for residual = 2 (mog_feature_map): omega, float32
        [FM_FEATURES, 128] frequencies drawn N(0, I), on the cache's device."""
        torch = _torch()
        om = torch.as_tensor(omega, dtype=torch.float32, device=self.arena.device).contiguous()
        if tuple(om.shape) != (FM_FEATURES, 128):
            raise ValueError(f"omega must be [{FM_FEATURES}, 128]")
        self._omega = om   # kept alive until the copy has run
        _check(lib().mog_feature_map(self._h, _ptr(om), _stream(stream)), "mog_feature_map")

    def splits(self) -> int:
        v = C.c_int32(0)
        _check(lib().mog_decode_splits(self._h, C.byref(v)), "mog_decode_splits")
        return v.value

    def layout(self) -> Layout:
        lay = Layout()
        _check(lib().mog_get_layout(self._h, C.byref(lay)), "mog_get_layout")
        return lay

    def sync_status(self, stream=None) -> int:
        return lib().mog_sync_status(self._h, _stream(stream))

    def array(self, name: str, dtype, shape):
        """A view of one arena array (see mog_layout) as a torch tensor."""
        torch = _torch()
        off = getattr(self.layout(), name)
        n = 1
        for s in shape:
            n *= s
        itemsize = torch.empty((), dtype=dtype).element_size()
        return self.arena[off:off + n * itemsize].view(dtype).view(*shape)


class Trace:
    """The build trace of mog_build_traced (see mog_trace_layout in mog.h) as torch views:
    l1_cent [U, T1, c_max, d], l1_assign [U, T1, n_mid], l2_cent [U, c_max, T2, l_max, d],
    l2_assign [U, T2, n_mid], l2_steps [U, c_max]."""

    def __init__(self, buf, lay: TraceLayout):
        torch = _torch()
        self.buf, self.layout = buf, lay
        U, T1, T2, cm, lm, d, nm = (lay.units, lay.iters_l1, lay.iters_l2, lay.c_max, lay.l_max,
                                    lay.d, lay.n_mid)

        def view(off, dtype, shape):
            n = 1
            for x in shape:
                n *= x
            return buf[off:off + 4 * n].view(dtype).view(*shape)

        self.l1_cent = view(lay.l1_cent, torch.float32, (U, T1, cm, d))
        self.l1_assign = view(lay.l1_assign, torch.int32, (U, T1, nm))
        self.l2_cent = view(lay.l2_cent, torch.float32, (U, cm, T2, lm, d))
        self.l2_assign = view(lay.l2_assign, torch.int32, (U, T2, nm))
        self.l2_steps = view(lay.l2_steps, torch.int32, (U, cm))


def trace_layout(params: Params, lengths_host) -> TraceLayout:
    import numpy as np
    lh = np.ascontiguousarray(lengths_host, np.int32)
    lay = TraceLayout()
    _check(lib().mog_trace_layout_of(C.byref(params), lh.ctypes.data_as(_P), C.byref(lay)),
           "mog_trace_layout_of")
    return lay


def build(K, V, lengths, params: Params, stream=None, partition=None, trace=False, draws=None):
    """mog_build (or mog_build_from_partition when partition=(perm, sub_off) is given, or
    mog_build_traced when trace=True, which returns (handle, Trace)).  `lengths` is a host
    sequence of int; a device copy is made.  With the k-means++ flag, draws (float64
    [units, c_max] uniforms in [0, 1), c_max from trace_layout) go to mog_build_seeded."""
    import numpy as np
    torch = _torch()
    lh = np.ascontiguousarray(lengths, np.int32)
    ld = torch.from_numpy(lh.copy()).to(K.device)  # (a PagedKV has a device too)
    nbytes = arena_bytes(params, lh)
    arena = torch.empty(nbytes + 256, dtype=torch.uint8, device=K.device)
    off = (-arena.data_ptr()) % 256
    arena = arena[off:off + nbytes]
    kv = _kv(K, V)
    h = _P()
    if params.flags & FLAG_KMEANSPP:
        if draws is None:
            raise ValueError("k-means++ seeding needs draws (float64 [units, c_max] in [0, 1))")
        lay = trace_layout(params, lh)
        dr = torch.as_tensor(draws, dtype=torch.float64, device=K.device).contiguous()
        if dr.numel() != lay.units * lay.c_max:
            raise ValueError(f"k-means++ needs draws of shape [{lay.units}, {lay.c_max}]")
        tbuf = torch.empty(lay.bytes, dtype=torch.uint8, device=K.device) if trace else None
        rc = lib().mog_build_seeded(C.byref(kv), _ptr(ld), lh.ctypes.data_as(_P), C.byref(params),
                                    _ptr(dr), _ptr(arena), nbytes, _ptr(tbuf),
                                    lay.bytes if trace else 0, _stream(stream), C.byref(h))
        _check(rc, "mog_build_seeded")
        hd = Handle(h, arena, params, K, V, ld, lh)
        return (hd, Trace(tbuf, lay)) if trace else hd
    if trace:
        lay = trace_layout(params, lh)
        tbuf = torch.empty(lay.bytes, dtype=torch.uint8, device=K.device)
        rc = lib().mog_build_traced(C.byref(kv), _ptr(ld), lh.ctypes.data_as(_P), C.byref(params),
                                    _ptr(arena), nbytes, _ptr(tbuf), lay.bytes, _stream(stream),
                                    C.byref(h))
        _check(rc, "mog_build_traced")
        return Handle(h, arena, params, K, V, ld, lh), Trace(tbuf, lay)
    if partition is None:
        rc = lib().mog_build(C.byref(kv), _ptr(ld), lh.ctypes.data_as(_P), C.byref(params),
                             _ptr(arena), nbytes, _stream(stream), C.byref(h))
        _check(rc, "mog_build")
    else:
        perm, sub_off = partition
        rc = lib().mog_build_from_partition(C.byref(kv), _ptr(ld), lh.ctypes.data_as(_P),
                                            C.byref(params), _ptr(perm), _ptr(sub_off),
                                            _ptr(arena), nbytes, _stream(stream), C.byref(h))
        _check(rc, "mog_build_from_partition")
    return Handle(h, arena, params, K, V, ld, lh)


def sub_off_stride(params: Params, lengths_host) -> int:
    import numpy as np
    lh = np.ascontiguousarray(lengths_host, np.int32)
    v = C.c_int64(0)
    _check(lib().mog_sub_off_stride(C.byref(params), lh.ctypes.data_as(_P), C.byref(v)),
           "mog_sub_off_stride")
    return v.value


def dense_scratch_bytes(batch, h_kv, h_q, n_max, d=128) -> int:
    v = C.c_size_t(0)
    _check(lib().dense_decode_scratch_bytes(batch, h_kv, h_q, d, n_max, C.byref(v)),
           "dense_decode_scratch_bytes")
    return v.value


def _check_q_out(K, q, out):
    """q must be a contiguous CUDA bf16 [B, H_q, 128] on K's device and out a contiguous
    float32 tensor of q's shape on the same device: the kernels write B*H_q*128 floats."""
    torch = _torch()
    B = q.shape[0] if isinstance(K, PagedKV) else K.shape[0]
    if (q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[0] != B or q.shape[2] != 128
            or not q.is_contiguous() or q.device != K.device):
        raise ValueError("q must be a contiguous bf16 tensor [B, H_q, 128] on the cache's device")
    if (out.dtype != torch.float32 or tuple(out.shape) != tuple(q.shape) or not out.is_contiguous()
            or out.device != q.device):
        raise ValueError("out must be a contiguous float32 tensor of q's shape on q's device")


def dense_decode(K, V, lengths_dev, n_max, q, out=None, scratch=None, stream=None):
    """Full-scan exact attention.  q: bf16 [B, H_q, d] -> out f32 [B, H_q, d]."""
    torch = _torch()
    B, H_kv = (q.shape[0], K.h_kv) if isinstance(K, PagedKV) else (K.shape[0], K.shape[1])
    H_q = q.shape[1]
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check_q_out(K, q, out)
    need = dense_scratch_bytes(B, H_kv, H_q, n_max)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=q.device)
    kv = _kv(K, V)
    _check(lib().dense_decode(C.byref(kv), _ptr(lengths_dev), n_max, B, H_kv, H_q, 128, _ptr(q),
                              _ptr(out), _ptr(scratch), scratch.numel(), _stream(stream)),
           "dense_decode")
    return out


def dense_decode_noalloc(K, V, lengths_dev, n_max, q, out, stream=None):
    """dense_decode whose scratch is the library's static device array: no device memory
    is allocated by this call (the caller supplies `out`)."""
    B, H_kv = (q.shape[0], K.h_kv) if isinstance(K, PagedKV) else (K.shape[0], K.shape[1])
    _check_q_out(K, q, out)
    kv = _kv(K, V)
    _check(lib().dense_decode_noalloc(C.byref(kv), _ptr(lengths_dev), n_max, B, H_kv, q.shape[1],
                                      128, _ptr(q), _ptr(out), _stream(stream)),
           "dense_decode_noalloc")
    return out


def kmeans_assign(x, cent, stream=None, with_recheck=False):
    """One first-level assignment step: x bf16 [n, d] (row stride x.stride(0)), cent f32
    [k, d].  Returns (assign int32 [n], rows decided by the exact fallback), plus the rows
    the tensor-core pass left to the direct pass when with_recheck."""
    torch = _torch()
    n, k = x.shape[0], cent.shape[0]
    out = torch.empty(n, dtype=torch.int32, device=x.device)
    need = C.c_size_t(0)
    _check(lib().mog_kmeans_assign_scratch_bytes(n, k, 128, C.byref(need)), "scratch")
    scratch = torch.empty(need.value, dtype=torch.uint8, device=x.device)
    counts = (C.c_int32 * 2)()
    _check(lib().mog_kmeans_assign(_ptr(x), x.stride(0), n, _ptr(cent), k, 128, _ptr(out),
                                   _ptr(scratch), need.value, _stream(stream), counts),
           "mog_kmeans_assign")
    if with_recheck:
        return out, counts[0], counts[1]
    return out, counts[0]


def kmeans_assign_segments(x, rows, seg_off, cent, stream=None):
    """Second-level assignment step: segment s = rows[seg_off[s]:seg_off[s+1]] against
    cent[s] (f32 [n_seg, k, d])."""
    torch = _torch()
    out = torch.empty(rows.shape[0], dtype=torch.int32, device=x.device)
    n_seg, k = cent.shape[0], cent.shape[1]
    _check(lib().mog_kmeans_assign_segments(_ptr(x), x.stride(0), _ptr(rows), _ptr(seg_off), n_seg,
                                            _ptr(cent), k, 128, _ptr(out), _stream(stream)),
           "mog_kmeans_assign_segments")
    return out


def check_bounded_wait(limit, arrive, scratch, stream=None) -> int:
    """Run the library's bounded mbarrier wait on a barrier that is (arrive=True) or is not
    completed; returns the status code (MOG_OK or MOG_ERR_TIMEOUT = 6)."""
    return lib().mog_check_bounded_wait(limit, 1 if arrive else 0, _ptr(scratch), _stream(stream))
