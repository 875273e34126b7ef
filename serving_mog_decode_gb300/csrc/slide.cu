// slide.cu -- the sliding recent window: after an append, the oldest recent key of every
// KV head whose window holds more than R keys leaves the window and joins the clusters.
//
// Sources: "Iceberg Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians",
// Abstract (each group of keys is summarised by a Gaussian: count, mean, variance) and the
// retrieval-completion attention page's Abstract (sink and tail anchors attended exactly).
// The pages do not say what happens to a key that leaves the tail window; this library
// lets it join the nearest non-empty cluster and, inside it, the nearest non-empty
// subcluster (the clustering's own nearest-centroid rule against the groups' means), and
// updates both groups' count, mean, population variance and value mean in place with
// Welford's recurrence.  Its row goes to the end of its subcluster's run of the partition;
// every later non-empty subcluster moves its first row to its end to make room, which keeps
// each run contiguous (rows within a run are a set for the attention).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "exact.cuh"
#include "internal.h"

namespace mog {

constexpr int SL_THREADS = 1024;
constexpr int SL_WARPS = SL_THREADS / 32;

// keep the two smallest values and the index of the smallest (lowest index on ties)
__device__ __forceinline__ void keep2(float &b1, int &i1, float &b2, float v, int i) {
    if (v < b1 || (v == b1 && i < i1)) {
        b2 = b1;
        b1 = v;
        i1 = i;
    } else if (v < b2) {
        b2 = v;
    }
}
__device__ __forceinline__ void merge2(float &b1, int &i1, float &b2, float ob1, int oi1, float ob2) {
    if (ob1 < b1 || (ob1 == b1 && oi1 < i1)) {
        b2 = fminf(b1, ob2);
        b1 = ob1;
        i1 = oi1;
    } else {
        b2 = fminf(b2, ob1);
    }
}

struct __align__(16) SlideRed {
    float d32[MAX_C];               // fp32 distance of every group (+inf if empty)
    float mean[SL_WARPS][MOG_D];    // a candidate mean per warp for the exact rule
    float b1[SL_WARPS], b2[SL_WARPS];
    int i1[SL_WARPS];
    double d[SL_WARPS];
    int di[SL_WARPS];
    float out_b1, out_b2;
    int out_i1;
    double out_d;
    int out_di;
};

// The nearest of the k groups with count > 0 whose means sit at ms + i * ld, for the key
// whose (exact) fp32 copy xs sits in shared memory, under the exact rule; -1 when no group
// is non-empty.  Called by the whole block.  Warp w scores groups w, w + W, ... with its
// lanes over the dimensions (four each, 16-byte loads of eight groups in flight); the fp32
// sum order does not matter to the certificate, only the fp64 rule fixes an order.
__device__ int nearest_group(const float *ms, int ld, const int *cnt, int k, const float *xs,
                             SlideRed &red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float b1 = INFINITY, b2 = INFINITY;
    int i1 = 0x7fffffff;
    const float4 xv = reinterpret_cast<const float4 *>(xs)[lane];
    for (int i0 = warp; i0 < k; i0 += 8 * SL_WARPS) {
        float4 m[8];
        bool ok[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // counts and means are read together
            const int i = i0 + q * SL_WARPS;
            ok[q] = i < k && cnt[i] > 0;
            m[q] = i < k ? reinterpret_cast<const float4 *>(ms + (size_t)i * ld)[lane]
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float d0 = __fsub_rn(xv.x, m[q].x), d1 = __fsub_rn(xv.y, m[q].y);
            float d2 = __fsub_rn(xv.z, m[q].z), d3 = __fsub_rn(xv.w, m[q].w);
            float acc = __fmaf_rn(d3, d3, __fmaf_rn(d2, d2, __fmaf_rn(d1, d1, d0 * d0)));
#pragma unroll
            for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (ok[q]) keep2(b1, i1, b2, acc, i0 + q * SL_WARPS);
            if (lane == 0 && i0 + q * SL_WARPS < k) red.d32[i0 + q * SL_WARPS] = ok[q] ? acc : INFINITY;
        }
    }
    if (lane == 0) {
        red.b1[warp] = b1;
        red.b2[warp] = b2;
        red.i1[warp] = i1;
    }
    __syncthreads();
    if (warp == 0) {
        b1 = red.b1[lane];
        b2 = red.b2[lane];
        i1 = red.i1[lane];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ob1 = __shfl_xor_sync(0xffffffffu, b1, o), ob2 = __shfl_xor_sync(0xffffffffu, b2, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i1, o);
            merge2(b1, i1, b2, ob1, oi, ob2);
        }
        if (lane == 0) {
            red.out_b1 = b1;
            red.out_b2 = b2;
            red.out_i1 = i1;
        }
    }
    __syncthreads();
    b1 = red.out_b1;
    b2 = red.out_b2;
    i1 = red.out_i1;
    if (i1 == 0x7fffffff) return -1;
    if (b2 == INFINITY || certified(b1, b2)) return i1;
    // The exact rule among the groups whose fp32 distance is within the error bound: warp
    // w takes candidates w, w + W, ...; the warp stages the candidate's mean in shared
    // memory and lane 0 sums the fp64 squares in index order (the key's fp32 copy holds
    // its bf16 values exactly).
    const float thr = b1 * (1.f + 2.5f * kCertRel);
    double best = INFINITY;
    int bi = 0x7fffffff;
    float *mw = red.mean[warp];
    for (int i = warp; i < k; i += SL_WARPS) {
        if (!(red.d32[i] <= thr)) continue;
        reinterpret_cast<float4 *>(mw)[lane] = reinterpret_cast<const float4 *>(ms + (size_t)i * ld)[lane];
        __syncwarp();
        if (lane == 0) {
            double dd = 0.0;
            for (int j = 0; j < MOG_D; ++j) {
                const double df = __dsub_rn((double)xs[j], (double)mw[j]);
                dd = __dadd_rn(dd, __dmul_rn(df, df));
            }
            if (dd < best || (dd == best && i < bi)) {
                best = dd;
                bi = i;
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const double ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob < best || (ob == best && oi < bi)) {
            best = ob;
            bi = oi;
        }
    }
    if (lane == 0) {
        red.d[warp] = best;
        red.di[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
        best = red.d[lane];
        bi = red.di[lane];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const double ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ob < best || (ob == best && oi < bi)) {
                best = ob;
                bi = oi;
            }
        }
        if (lane == 0) red.out_di = bi;
    }
    __syncthreads();
    return red.out_di;
}

// Welford's update of one group (count n, mean and variance rows ms[0..d), ms[d..2d),
// value mean vb, its bf16 high/low copy vhl) by the key x and value v (shared memory).
// Threads j < d update key dimension j, threads d + j value dimension j.
__device__ __forceinline__ void welford(int n, float *ms, float *vb, uint16_t *vhl, const float *xs,
                                        const float *vs) {
    const int tid = threadIdx.x;
    const float n1 = (float)(n + 1);
    if (tid < MOG_D) {
        const int j = tid;
        const float mu = ms[j], var = ms[MOG_D + j];
        const float delta = xs[j] - mu;
        const float mu_new = mu + delta / n1;
        ms[j] = mu_new;
        ms[MOG_D + j] = ((float)n * var + delta * (xs[j] - mu_new)) / n1;
    } else if (tid < 2 * MOG_D) {
        const int j = tid - MOG_D;
        const float m = vb[j] + (vs[j] - vb[j]) / n1;
        vb[j] = m;
        const uint32_t hi = f2bf(m);
        vhl[j] = (uint16_t)hi;
        vhl[MOG_D + j] = (uint16_t)f2bf(m - bf1((uint16_t)hi));
    }
}

// One CTA per unit, after the append kernel has advanced the lengths.
__global__ void __launch_bounds__(SL_THREADS) k_slide(Dev dv, int R) {
    __shared__ __align__(16) float xs[MOG_D], vs[MOG_D];
    __shared__ SlideRed red;
    const int u = blockIdx.x, tid = threadIdx.x;
    int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], L = ui[UI_L], b = ui[UI_B], h = u % dv.h_kv;
    const int p = ui[UI_RLO];
    if (dv.n_now[b] - p <= R) return;  // the window still holds at most R keys
    const uint16_t *kr = dv.krow(b, h, p), *vr = dv.vrow(b, h, p);
    if (tid < MOG_D) {
        xs[tid] = bf1(kr[tid]);
        vs[tid] = bf1(vr[tid]);
    }
    __syncthreads();
    const size_t cg0 = (size_t)u * dv.c_max, sg0 = (size_t)u * dv.c_max * dv.l_max;
    const int c = nearest_group(dv.cl_ms + cg0 * 2 * MOG_D, 2 * MOG_D, dv.cl_n + cg0, C, xs, red);
    if (c < 0) return;  // no cluster to join: the window grows instead
    const int l = nearest_group(dv.sub_ms + (sg0 + (size_t)c * L) * 2 * MOG_D, 2 * MOG_D,
                                dv.sub_n + sg0 + (size_t)c * L, L, xs, red);
    if (l < 0) {  // a non-empty cluster has a non-empty subcluster; reaching here is corrupt
        if (tid == 0) flag_error(dv.status, ST_BAD_INDEX);
        return;
    }
    const size_t cg = cg0 + c, sg = sg0 + (size_t)c * L + l;
    const int ncl = dv.cl_n[cg], nsub = dv.sub_n[sg];
    welford(ncl, dv.cl_ms + cg * 2 * MOG_D, dv.cl_vbar + cg * MOG_D, dv.cl_vhl + cg * 2 * MOG_D, xs, vs);
    welford(nsub, dv.sub_ms + sg * 2 * MOG_D, dv.sub_vbar + sg * MOG_D, dv.sub_vhl + sg * 2 * MOG_D, xs, vs);
    // The partition: every later non-empty subcluster moves its first row to its end and
    // every later offset grows by one.  Batches of eight subclusters per thread run from
    // the top down, reads before writes, so that no batch reads a slot that a batch above
    // it has written; s_top keeps the old offset at the top of the batch below.
    const int CL = C * L, g = c * L + l;
    int *so = dv.sub_off + (size_t)u * dv.sub_off_stride;
    int *pm = dv.perm + (size_t)u * dv.n_cap;
    constexpr int B8 = 8, BATCH = B8 * SL_THREADS;
    __shared__ int s_top;
    const int first = g + 1, old_end = so[CL];
    if (tid == 0) s_top = old_end;
    __syncthreads();
    for (int bi = (CL - first + BATCH - 1) / BATCH - 1; bi >= 0; --bi) {
        const int base = first + bi * BATCH, top = min(CL, base + BATCH);
        int a[B8], e[B8], v[B8];
#pragma unroll
        for (int q = 0; q < B8; ++q) {
            const int gg = base + q * SL_THREADS + tid;
            a[q] = gg < top ? so[gg] : 0;
            e[q] = gg < top ? (gg + 1 == top ? s_top : so[gg + 1]) : 0;
        }
#pragma unroll
        for (int q = 0; q < B8; ++q) v[q] = a[q] < e[q] ? pm[a[q]] : 0;
        __syncthreads();
#pragma unroll
        for (int q = 0; q < B8; ++q) {
            const int gg = base + q * SL_THREADS + tid;
            if (gg < top) {
                if (a[q] < e[q]) pm[e[q]] = v[q];
                so[gg] = a[q] + 1;
            }
        }
        if (tid == 0) s_top = a[0];  // the old offset of subcluster `base`
        __syncthreads();
    }
    if (tid == 0) {
        pm[s_top] = p;  // the old end of subcluster g
        so[CL] = old_end + 1;
        dv.cl_n[cg] = ncl + 1;
        dv.sub_n[sg] = nsub + 1;
        ui[UI_NMID] += 1;
        ui[UI_RLO] = p + 1;
    }
}

cudaError_t launch_slide(const Dev &dv, const Plan &pl, cudaStream_t s) {
    k_slide<<<pl.units, SL_THREADS, 0, s>>>(dv, pl.R);
    return cudaGetLastError();
}

}  // namespace mog
