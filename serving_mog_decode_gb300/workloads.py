"""Seeded synthetic workloads: planted-centre keys, Gaussian values, queries.

This module only draws inputs.  It holds none of the attention arithmetic and is the one
piece shared by the CUDA path's tests and benchmark and by the CPU oracle's tests.

Key model (one KV head, "unit"): M centres c_j ~ N(0, I_d); each key picks a centre
z_i uniformly and is k_i = c_{z_i} + sigma_{z_i} * eps_i with eps_i ~ N(0, I_d); keys
0..3 are attention sinks 8*u for a unit vector u (normalised N(0, I) draw); a fraction
of the other keys can be scaled x4 as outliers.  Values are N(0, 1).  The query of head
g is 0.5*c_{j*_g} + 0.5*N(0, I) with j*_g drawn per query head.  Everything is drawn in
float64 and rounded to bf16 (to float32, then round-to-nearest-even to bf16).

Streams: unit (b, h) draws from SeedSequence(seed, spawn_key=(b, h)) split into four
children, used in this order of roles: structure (centres, sigmas, z, sink direction,
outliers), key noise, values, queries.  Decode step t >= 1 of the append workload uses
SeedSequence(seed, spawn_key=(b, h, 1 + t)).  Sequence lengths of variable-length
batches come from SeedSequence(seed, spawn_key=(1 << 20,)).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D = 128
CHUNK = 1 << 16


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    h_kv: int
    h_q: int
    n: int                       # context length (fixed-length batches)
    centres: int
    sigma: tuple = (0.5, 0.5)    # per-centre sigma ~ U[lo, hi] (lo == hi: constant)
    outlier_frac: float = 0.0
    n_clusters: int = 0          # 0: round(sqrt(N)) per sequence
    n_sub: int = 0               # 0: ceil(log2(N)) per sequence
    top_c: int = 8
    top_s: int = 8
    n_sink: int = 4
    n_recent: int = 256
    seed: int = 0
    n_range: tuple | None = None  # per-sequence N ~ U[lo, hi] (inclusive)
    steps: int = 0               # decode steps that each append one key/value
    d: int = D
    note: str = field(default="", compare=False)

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv


WORKLOADS = {
    "tiny-4k": Workload(
        "tiny-4k", batch=1, h_kv=1, h_q=1, n=4096, centres=256, n_clusters=64, n_sub=12,
        top_c=4, top_s=6, n_sink=4, n_recent=64, seed=0,
        note="single head, d=128, N=4096"),
    "qwen3-4b-32k": Workload(
        "qwen3-4b-32k", batch=1, h_kv=8, h_q=32, n=32768, centres=256, n_clusters=181,
        n_sub=15, top_c=8, top_s=8, n_sink=4, n_recent=256, seed=1,
        note="Qwen3-4B-shaped layer: 32 q heads / 8 KV heads, N=32768"),
    "olmo3-7b-varlen": Workload(
        "olmo3-7b-varlen", batch=8, h_kv=32, h_q=32, n=65536, centres=512, sigma=(0.3, 1.0),
        n_clusters=0, n_sub=0, top_c=8, top_s=8, n_sink=4, n_recent=256, seed=2,
        n_range=(16384, 65536), note="Olmo-3-7B-shaped MHA layer, batch 8, N in [16K, 64K]"),
    "qwen3-14b-128k": Workload(
        "qwen3-14b-128k", batch=4, h_kv=8, h_q=40, n=131072, centres=1024, outlier_frac=0.001,
        n_clusters=362, n_sub=17, top_c=12, top_s=8, n_sink=4, n_recent=256, seed=3, steps=64,
        note="Qwen3-14B-shaped layer, batch 4, N=131072, 64 appending decode steps"),
    "ctx-1m": Workload(
        "ctx-1m", batch=1, h_kv=8, h_q=32, n=1048576, centres=4096, n_clusters=1024, n_sub=20,
        top_c=16, top_s=8, n_sink=4, n_recent=512, seed=4,
        note="1M-token context, 32 q heads / 8 KV heads"),
}


def lengths(w: Workload) -> np.ndarray:
    """Per-sequence context lengths (int32[batch])."""
    if w.n_range is None:
        return np.full(w.batch, w.n, np.int32)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(w.seed, spawn_key=(1 << 20,))))
    return rng.integers(w.n_range[0], w.n_range[1] + 1, size=w.batch).astype(np.int32)


def clusters_for(w: Workload, n: int) -> tuple[int, int]:
    """(C, L) for a sequence of length n: the workload's fixed values, else
    round(sqrt(n)) clusters and ceil(log2(n)) subclusters."""
    c = w.n_clusters if w.n_clusters > 0 else int(round(math.sqrt(n)))
    l = w.n_sub if w.n_sub > 0 else int(math.ceil(math.log2(n)))
    return max(c, 1), max(l, 1)


def seed_draws(units: int, c_max: int, seed: int) -> np.ndarray:
    """Uniform draws in [0, 1), float64 [units, c_max]: the random input of k-means++
    seeding (one draw per unit and seed)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(1 << 21,))))
    return rng.random((units, c_max))


def fm_omega(m: int, d: int, seed: int) -> np.ndarray:
    """Random-feature frequencies, float64 [m, d] drawn N(0, 1): the random input of the
    feature-map residual."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(1 << 22,))))
    return rng.standard_normal((m, d))


def to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bf16 (RNE) bit patterns as uint16."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (b >> np.uint32(16)).astype(np.uint16)


def from_bf16(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values."""
    return (np.asarray(h, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _gen(ss):
    return np.random.Generator(np.random.PCG64(ss))


class UnitDraw:
    """All inputs of one KV head (b, h): keys/values [n, d] bf16 and G queries [G, d]."""

    def __init__(self, w: Workload, b: int, h: int, n: int):
        self.w, self.b, self.h, self.n = w, b, h, n
        kids = np.random.SeedSequence(w.seed, spawn_key=(b, h)).spawn(4)
        st, self._eps_ss, self._val_ss, qs = kids
        g = _gen(st)
        d, M = w.d, w.centres
        self.centres = g.standard_normal((M, d))
        lo, hi = w.sigma
        self.sig = np.full(M, lo) if lo == hi else g.uniform(lo, hi, size=M)
        self.z = g.integers(0, M, size=n)
        u = g.standard_normal(d)
        self.u = u / np.linalg.norm(u)
        n_sink = min(w.n_sink, n)
        self.n_sink = n_sink
        if w.outlier_frac > 0 and n > n_sink:
            n_out = int(round(w.outlier_frac * (n - n_sink)))
            self.outliers = np.sort(g.choice(n - n_sink, size=n_out, replace=False) + n_sink)
        else:
            self.outliers = np.zeros(0, np.int64)
        gq = _gen(qs)
        self.jstar = gq.integers(0, M, size=w.group)
        noise = gq.standard_normal((w.group, d))
        self.q = to_bf16(0.5 * self.centres[self.jstar] + 0.5 * noise)

    def keys_values(self, out_k: np.ndarray | None = None, out_v: np.ndarray | None = None):
        """Keys and values, bf16 [n, d]; written into out_k/out_v rows [0, n) if given."""
        w, n, d = self.w, self.n, self.w.d
        K = np.empty((n, d), np.uint16) if out_k is None else out_k
        V = np.empty((n, d), np.uint16) if out_v is None else out_v
        ge, gv = _gen(self._eps_ss), _gen(self._val_ss)
        out_set = set(self.outliers.tolist()) if self.outliers.size else None
        for lo in range(0, n, CHUNK):
            hi = min(n, lo + CHUNK)
            z = self.z[lo:hi]
            k = self.centres[z] + self.sig[z][:, None] * ge.standard_normal((hi - lo, d))
            if lo < self.n_sink:
                k[: self.n_sink - lo] = 8.0 * self.u
            if out_set is not None:
                idx = self.outliers[(self.outliers >= lo) & (self.outliers < hi)] - lo
                k[idx] *= 4.0
            K[lo:hi] = to_bf16(k)
            V[lo:hi] = to_bf16(gv.standard_normal((hi - lo, d)))
        return K, V

    def step(self, t: int):
        """Inputs of decode step t >= 1 of an appending workload: (k_new, v_new, q[G, d])."""
        g = _gen(np.random.SeedSequence(self.w.seed, spawn_key=(self.b, self.h, 1 + t)))
        d = self.w.d
        z = g.integers(0, self.w.centres)
        k = self.centres[z] + self.sig[z] * g.standard_normal(d)
        v = g.standard_normal(d)
        q = 0.5 * self.centres[self.jstar] + 0.5 * g.standard_normal((self.w.group, d))
        return to_bf16(k), to_bf16(v), to_bf16(q)


def make_unit(w: Workload, b: int = 0, h: int = 0, n: int | None = None):
    """(K [n, d], V [n, d], q [G, d]) bf16 bit patterns of unit (b, h)."""
    n = int(lengths(w)[b]) if n is None else n
    u = UnitDraw(w, b, h, n)
    K, V = u.keys_values()
    return K, V, u.q


def make_batch(w: Workload, n_cap: int | None = None, units=None):
    """Whole-layer inputs: K, V [B, H_kv, n_cap, d] bf16, q [B, H_q, d] bf16, lengths[B].
    `units`, if given, limits generation to those (b, h) pairs (others left zero)."""
    lens = lengths(w)
    n_cap = int(lens.max()) + w.steps if n_cap is None else n_cap
    K = np.zeros((w.batch, w.h_kv, n_cap, w.d), np.uint16)
    V = np.zeros_like(K)
    q = np.zeros((w.batch, w.h_q, w.d), np.uint16)
    G = w.group
    for b in range(w.batch):
        for h in range(w.h_kv):
            if units is not None and (b, h) not in units:
                continue
            u = UnitDraw(w, b, h, int(lens[b]))
            u.keys_values(K[b, h], V[b, h])
            q[b, h * G:(h + 1) * G] = u.q
    return K, V, q, lens
