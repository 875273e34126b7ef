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
//
// One thread-block cluster of up to 8 CTAs per KV head shares the work: each CTA scores a
// slice of the cluster means and moves a slice of the subclusters' rows; the slices' best
// scores are merged through distributed shared memory, and cluster barriers order the
// reads of the partition before its writes.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "exact.cuh"
#include "internal.h"

namespace mog {

constexpr int SL_THREADS = 1024;
constexpr int SL_WARPS = SL_THREADS / 32;
constexpr int SL_MAX_CS = 8;  // CTAs per KV head (portable cluster size)

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
__device__ __forceinline__ void keep_min(double &best, int &bi, double d, int i) {
    if (d < best || (d == best && i < bi)) {
        best = d;
        bi = i;
    }
}

struct __align__(16) SlideRed {
    float d32[MAX_C];             // fp32 distance of every group of this CTA's slice (+inf if empty)
    float mean[SL_WARPS][MOG_D];  // a candidate mean per warp for the exact rule
    float b1[SL_WARPS], b2[SL_WARPS];
    int i1[SL_WARPS];
    double d[SL_WARPS];
    int di[SL_WARPS];
    float out_b1, out_b2;  // this CTA's result, read by the cluster
    int out_i1;
    double out_d;
    int out_di;
};

// Block-wide: the two smallest fp32 distances of the key (fp32 copy xs in shared memory)
// to the non-empty groups lo .. hi-1 (means at ms + i * ld) and the index of the smallest,
// into red.out_*; red.d32[i - lo] keeps every distance.  Warp w scores groups lo + w,
// lo + w + W, ..., its lanes over the dimensions (four each; 16-byte loads of eight groups
// in flight).  The fp32 sum order does not matter to the certificate.
__device__ void score_range(const float *ms, int ld, const int *cnt, int lo, int hi, const float *xs,
                            SlideRed &red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float b1 = INFINITY, b2 = INFINITY;
    int i1 = 0x7fffffff;
    const float4 xv = reinterpret_cast<const float4 *>(xs)[lane];
    for (int i0 = lo + warp; i0 < hi; i0 += 8 * SL_WARPS) {
        float4 m[8];
        bool ok[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // counts and means are read together
            const int i = i0 + q * SL_WARPS;
            ok[q] = i < hi && cnt[i] > 0;
            m[q] = i < hi ? reinterpret_cast<const float4 *>(ms + (size_t)i * ld)[lane]
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * SL_WARPS;
            float d0 = __fsub_rn(xv.x, m[q].x), d1 = __fsub_rn(xv.y, m[q].y);
            float d2 = __fsub_rn(xv.z, m[q].z), d3 = __fsub_rn(xv.w, m[q].w);
            float acc = __fmaf_rn(d3, d3, __fmaf_rn(d2, d2, __fmaf_rn(d1, d1, d0 * d0)));
#pragma unroll
            for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (ok[q]) keep2(b1, i1, b2, acc, i);
            if (lane == 0 && i < hi) red.d32[i - lo] = ok[q] ? acc : INFINITY;
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
}

// Block-wide: the exact rule (R5: fp64, index order, lowest index on ties) among the
// groups lo .. hi-1 whose fp32 distance (red.d32, from score_range) is at most thr, into
// red.out_d / red.out_di.  Warp w takes candidates lo + w, lo + w + W, ...; the warp
// stages the candidate's mean in shared memory and lane 0 sums the fp64 squares (the
// key's fp32 copy holds its bf16 values exactly).
__device__ void exact_range(const float *ms, int ld, int lo, int hi, float thr, const float *xs,
                            SlideRed &red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double best = INFINITY;
    int bi = 0x7fffffff;
    float *mw = red.mean[warp];
    for (int i = lo + warp; i < hi; i += SL_WARPS) {
        if (!(red.d32[i - lo] <= thr)) continue;
        reinterpret_cast<float4 *>(mw)[lane] = reinterpret_cast<const float4 *>(ms + (size_t)i * ld)[lane];
        __syncwarp();
        if (lane == 0) {
            double dd = 0.0;
            for (int j = 0; j < MOG_D; ++j) {
                const double df = __dsub_rn((double)xs[j], (double)mw[j]);
                dd = __dadd_rn(dd, __dmul_rn(df, df));
            }
            keep_min(best, bi, dd, i);
        }
        __syncwarp();
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
            keep_min(best, bi, ob, oi);
        }
        if (lane == 0) {
            red.out_d = best;
            red.out_di = bi;
        }
    }
    __syncthreads();
}

// Block-wide, one CTA: the nearest of the k groups with count > 0 under the exact rule;
// -1 when none is non-empty.
__device__ int nearest_local(const float *ms, int ld, const int *cnt, int k, const float *xs,
                             SlideRed &red) {
    score_range(ms, ld, cnt, 0, k, xs, red);
    const float b1 = red.out_b1, b2 = red.out_b2;
    const int i1 = red.out_i1;
    __syncthreads();
    if (i1 == 0x7fffffff) return -1;
    if (b2 == INFINITY || certified(b1, b2)) return i1;
    exact_range(ms, ld, 0, k, b1 * (1.f + 2.5f * kCertRel), xs, red);
    const int r = red.out_di;
    __syncthreads();
    return r;
}

// Welford's update of one group (count n, mean and variance rows ms[0..d), ms[d..2d),
// their bf16 copy ms16 and e4m3 copy ms8 (or null), value mean vb, its bf16 high/low copy
// vhl, whose high part holds the e4m3-rounded mean when ms8 is given) by the key x and
// value v (shared memory).  Threads j < d update key dimension j, threads d + j value
// dimension j.
__device__ __forceinline__ void welford(int n, float *ms, uint16_t *ms16, uint8_t *ms8, float *vb, uint16_t *vhl,
                                        const float *xs, const float *vs) {
    const int tid = threadIdx.x;
    const float n1 = (float)(n + 1);
    if (tid < MOG_D) {
        const int j = tid;
        const float mu = ms[j], var = ms[MOG_D + j];
        const float delta = xs[j] - mu;
        const float mu_new = mu + delta / n1;
        const float var_new = ((float)n * var + delta * (xs[j] - mu_new)) / n1;
        ms[j] = mu_new;
        ms[MOG_D + j] = var_new;
        if (ms16) {
            ms16[j] = (uint16_t)f2bf(mu_new);
            ms16[MOG_D + j] = (uint16_t)f2bf(var_new);
        }
        if (ms8) {
            ms8[j] = (uint8_t)f2e4m3(mu_new);
            ms8[MOG_D + j] = (uint8_t)f2e4m3(var_new);
        }
    } else if (tid < 2 * MOG_D) {
        const int j = tid - MOG_D;
        const float m = vb[j] + (vs[j] - vb[j]) / n1;
        vb[j] = m;
        const uint32_t hi = f2bf(ms8 ? e4m3_round(m) : m);
        vhl[j] = (uint16_t)hi;
        vhl[MOG_D + j] = (uint16_t)f2bf(m - bf1((uint16_t)hi));
    }
}

// One cluster of CS CTAs per unit (grid (CS, units)), after the append kernel has advanced
// the lengths.  Every decision is computed identically by all CTAs of the cluster, so that
// they take the same path through every cluster barrier.  CLU = false: one CTA per unit,
// launched without a cluster, with block barriers.
template <bool CLU>
__global__ void __launch_bounds__(SL_THREADS) k_slide(Dev dv, int R) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    auto csync = [&]() {
        if constexpr (CLU) cluster.sync();
        else __syncthreads();
    };
    __shared__ __align__(16) float xs[MOG_D], vs[MOG_D];
    __shared__ SlideRed red;
    __shared__ int s_top;
    const int CS = CLU ? (int)cluster.num_blocks() : 1, rk = CLU ? (int)cluster.block_rank() : 0;
    const int u = blockIdx.y, tid = threadIdx.x;
    int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], L = ui[UI_L], b = ui[UI_B], h = u % dv.h_kv;
    const int p = ui[UI_RLO];
    if (dv.n_now[b] - p <= R) return;  // the window still holds at most R keys (whole cluster)
    const uint16_t *kr = dv.krow(b, h, p), *vr = dv.vrow(b, h, p);
    if (tid < MOG_D) {
        xs[tid] = bf1(kr[tid]);
        vs[tid] = bf1(vr[tid]);
    }
    __syncthreads();
    const size_t cg0 = (size_t)u * dv.c_max, sg0 = (size_t)u * dv.c_max * dv.l_max;
    const float *cms = dv.cl_ms + cg0 * 2 * MOG_D;
    // 1. the nearest non-empty cluster: slices scored per CTA, merged over the cluster
    const int lo = (int)((int64_t)C * rk / CS), hi = (int)((int64_t)C * (rk + 1) / CS);
    score_range(cms, 2 * MOG_D, dv.cl_n + cg0, lo, hi, xs, red);
    csync();
    float b1 = INFINITY, b2 = INFINITY;
    int i1 = 0x7fffffff;
    for (int r = 0; r < CS; ++r) {
        const SlideRed *o = CLU ? cluster.map_shared_rank(&red, r) : &red;
        merge2(b1, i1, b2, o->out_b1, o->out_i1, o->out_b2);
    }
    int c = i1;
    if (i1 != 0x7fffffff && !(b2 == INFINITY || certified(b1, b2))) {
        exact_range(cms, 2 * MOG_D, lo, hi, b1 * (1.f + 2.5f * kCertRel), xs, red);
        csync();
        double best = INFINITY;
        int bi = 0x7fffffff;
        for (int r = 0; r < CS; ++r) {
            const SlideRed *o = CLU ? cluster.map_shared_rank(&red, r) : &red;
            keep_min(best, bi, o->out_d, o->out_di);
        }
        c = bi;
    }
    csync();  // every CTA is done reading the others' results
    if (c == 0x7fffffff) return;  // no cluster to join: the window grows instead
    // 2. the nearest non-empty subcluster of c (each CTA on its own, identically)
    const int l = nearest_local(dv.sub_ms + (sg0 + (size_t)c * L) * 2 * MOG_D, 2 * MOG_D,
                                dv.sub_n + sg0 + (size_t)c * L, L, xs, red);
    if (l < 0) {  // a non-empty cluster has a non-empty subcluster; reaching here is corrupt
        if (tid == 0 && rk == 0) flag_error(dv.status, ST_BAD_INDEX);
        return;
    }
    const size_t cgi = cg0 + c, sgi = sg0 + (size_t)c * L + l;
    const int ncl = dv.cl_n[cgi], nsub = dv.sub_n[sgi];
    // 3-4. The partition: every later non-empty subcluster moves its first row to its end and
    // every later offset grows by one.  Batches run from the top down over all threads of
    // the cluster, reads before writes (a cluster barrier between), so that no batch reads
    // a slot a batch above it has written; s_top (in every CTA) keeps the old offset at the
    // top of the batch below.
    const int CL = C * L, g = c * L + l;
    int *so = dv.sub_off + (size_t)u * dv.sub_off_stride;
    int *pm = dv.perm + (size_t)u * dv.n_cap;
    constexpr int B4 = 4;
    const int nthr = CS * SL_THREADS, gt = rk * SL_THREADS + tid, batch = B4 * nthr;
    const int first = g + 1, old_end = so[CL];
    if (tid == 0) s_top = old_end;
    csync();  // every CTA has chosen (c, l) from the means before they change
    if (rk == 0) {   // 3. Welford
        welford(ncl, dv.cl_ms + cgi * 2 * MOG_D, dv.cl_ms16 ? dv.cl_ms16 + cgi * 2 * MOG_D : nullptr,
                dv.cl_ms8 ? dv.cl_ms8 + cgi * 2 * MOG_D : nullptr, dv.cl_vbar + cgi * MOG_D,
                dv.cl_vhl + cgi * 2 * MOG_D, xs, vs);
        welford(nsub, dv.sub_ms + sgi * 2 * MOG_D, dv.sub_ms16 ? dv.sub_ms16 + sgi * 2 * MOG_D : nullptr,
                dv.sub_ms8 ? dv.sub_ms8 + sgi * 2 * MOG_D : nullptr, dv.sub_vbar + sgi * MOG_D,
                dv.sub_vhl + sgi * 2 * MOG_D, xs, vs);
    }
    for (int bi = (CL - first + batch - 1) / batch - 1; bi >= 0; --bi) {
        const int base = first + bi * batch, top = min(CL, base + batch);
        const int below_top = s_top;
        int a[B4], e[B4], v[B4];
#pragma unroll
        for (int q = 0; q < B4; ++q) {
            const int gg = base + q * nthr + gt;
            a[q] = gg < top ? so[gg] : 0;
            e[q] = gg < top ? (gg + 1 == top ? below_top : so[gg + 1]) : 0;
        }
#pragma unroll
        for (int q = 0; q < B4; ++q) v[q] = a[q] < e[q] ? pm[a[q]] : 0;
        csync();
#pragma unroll
        for (int q = 0; q < B4; ++q) {
            const int gg = base + q * nthr + gt;
            if (gg < top) {
                if (a[q] < e[q]) pm[e[q]] = v[q];
                so[gg] = a[q] + 1;
            }
        }
        if (gt == 0) {  // the old offset of subcluster `base`, to every CTA
            if constexpr (CLU) {
                for (int r = 0; r < CS; ++r) *cluster.map_shared_rank(&s_top, r) = a[0];
            } else {
                s_top = a[0];
            }
        }
        csync();
    }
    if (rk == 0 && tid == 0) {
        pm[s_top] = p;  // the old end of subcluster g
        so[CL] = old_end + 1;
        dv.cl_n[cgi] = ncl + 1;
        dv.sub_n[sgi] = nsub + 1;
        ui[UI_NMID] += 1;
        ui[UI_RLO] = p + 1;
    }
}

cudaError_t launch_slide(const Dev &dv, const Plan &pl, cudaStream_t s) {
    // CTAs per unit: one for up to 4096 subclusters (there the cluster barriers cost more
    // than they save), else one per 2048, at most 8, and few enough that every unit's
    // cluster is resident
    const int64_t groups = (int64_t)pl.c_max * pl.l_max;
    const int want = groups <= 4096 ? 1 : (int)std::min<int64_t>(SL_MAX_CS, (groups + 2047) / 2048);
    const int cs = std::max(1, std::min(want, num_sms() / std::max(1, pl.units)));
    if (cs == 1) {
        k_slide<false><<<dim3(1, pl.units), SL_THREADS, 0, s>>>(dv, pl.R);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, pl.units);
    cfg.blockDim = dim3(SL_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_slide<true>, dv, pl.R);
    if (e == cudaErrorInvalidClusterSize || e == cudaErrorInvalidConfiguration) {
        cudaGetLastError();  // no room for the clusters here: one CTA per unit instead
        k_slide<false><<<dim3(1, pl.units), SL_THREADS, 0, s>>>(dv, pl.R);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace mog
