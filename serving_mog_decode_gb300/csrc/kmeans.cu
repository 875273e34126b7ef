// kmeans.cu -- the MoG build: two-level Lloyd k-means over each KV head's mid-region keys
// and the Gaussian summaries of every cluster and subcluster.
//
// Source: "Iceberg Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians",
// Abstract (after prefill the keys of each head are partitioned hierarchically into
// O(sqrt N) clusters and O(log N) subclusters per cluster, each represented by a
// Gaussian).  The pages name no clustering algorithm; this library uses Lloyd's
// algorithm with strided seeding (centroid j starts at member floor(j*n/k) in position
// order), at most T assignment steps, a mean update between steps, an early stop when a
// step changes nothing, and empty clusters keeping their centroid.
//
// Assignment decision.  The nearest centroid is defined by D(x,c) = sum_j (x_j - c_j)^2
// evaluated in fp64 in index order, lowest index on ties.  The kernels compute D in fp32
// (difference, then fused square-accumulate: |D32 - D| <= (d+2) 2^-24 D since every term
// is non-negative) and keep the winner only when the runner-up is separated by more than
// that bound on both values (with a safety factor); every other row is recomputed with
// the exact fp64 rule.  The result therefore equals the fp64 rule bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "exact.cuh"
#include "internal.h"
#include "tc.cuh"

namespace mog {

// error factor of the tensor-core distances |c|^2 - 2 k.c (split-bf16 centroids, fp32
// accumulate): a score within TC_F (|k|^2 + |c|^2) of the exact one, with a safety margin
constexpr float TC_F = 1.0f / 8192.0f;  // 2^-13

// converged before or at step t: some step 1..t changed nothing
__device__ __forceinline__ bool converged_by(const int *changed, int t) {
    for (int s = 1; s <= t; ++s)
        if (changed[s] == 0) return true;
    return false;
}

// ------------------------------------------------------------------------------------
// First-level assignment.  One CTA: 64 rows x all centroids, 256 threads, each thread a
// 4 x 4 register tile of (row, centroid) distances; rows and centroid tiles are staged
// transposed in shared memory as fp32.
// ------------------------------------------------------------------------------------
struct AssignJob {
    const uint16_t *K;
    int64_t sb, sh, sn;
    const int *bt;  // block table of a paged cache, or null
    int pshift, pps;
    int h_kv;
    const int *unit_info;  // null: a single unit of n_single rows at K, row stride sn
    int n_single, k_single;
    const float *cent;
    int64_t cent_ustride;
    int *assign;
    int64_t assign_ustride;
    int *changed;  // [unit][T]
    int *fb_list;  // [unit][fb_ustride]
    int64_t fb_ustride;
    int *fb_cnt;  // [unit][T]
    int t, T;
    // row-list mode of the direct pass: rows[u][0 .. rows_cnt[u*T + t]) instead of all rows
    const int *rows;
    int64_t rows_ustride;
    const int *rows_cnt;
    // tensor-core pass: centroid images, squared norms, rows it leaves to the direct pass
    uint16_t *cimg;  // [unit][cimg_ustride]: per 256-centroid chunk [2 parts][2 halves][256][64]
    int64_t cimg_ustride;
    float *cnorm;  // [unit][cn_ustride]
    int64_t cn_ustride;
    int *rc_list;  // [unit][fb_ustride]
    int *rc_cnt;   // [unit][T]
    int *status;
};

constexpr int AS_ROWS = 64, AS_CENT = 64, AS_THREADS = 256, AS_PAD = 68;
constexpr size_t AS_SMEM = 2 * MOG_D * AS_PAD * sizeof(float);

// Where unit u's rows are: n mid rows, k centroids.  Row r of the unit is the key at
// position S + r of (b, h); mid_row() returns its address.
struct JobUnit {
    const uint16_t *x;  // row 0 of a contiguous unit
    int n, k, b, h, s0;
};
__device__ __forceinline__ JobUnit job_unit(const AssignJob &jb, int u) {
    JobUnit j;
    if (jb.unit_info) {
        const int *ui = jb.unit_info + u * UI_STRIDE;
        j.b = ui[UI_B];
        j.h = u % jb.h_kv;
        j.n = ui[UI_NMID];
        j.k = ui[UI_C];
        j.s0 = ui[UI_S];
        j.x = jb.K + j.b * jb.sb + j.h * jb.sh + (int64_t)j.s0 * jb.sn;
    } else {
        j.n = jb.n_single;
        j.k = jb.k_single;
        j.b = j.h = j.s0 = 0;
        j.x = jb.K;
    }
    return j;
}
__device__ __forceinline__ const uint16_t *mid_row(const AssignJob &jb, const JobUnit &j, int r) {
    if (!jb.bt) return j.x + (int64_t)r * jb.sn;
    const int64_t pos = (int64_t)j.s0 + r;
    const int64_t page = jb.bt[(int64_t)j.b * jb.pps + (pos >> jb.pshift)];
    return jb.K + page * jb.sb + j.h * jb.sh + (pos & ((1 << jb.pshift) - 1)) * jb.sn;
}

__global__ void __launch_bounds__(AS_THREADS) k_assign_l1(AssignJob jb) {
    extern __shared__ __align__(16) float as_smem[];
    float *Xs = as_smem;                  // [d][AS_PAD], rows
    float *Cs = as_smem + MOG_D * AS_PAD;  // [d][AS_PAD], centroids
    __shared__ int s_changed, s_base;
    __shared__ int s_unc[AS_ROWS];
    const int u = blockIdx.y;
    const int *chg = jb.changed + (int64_t)u * jb.T;
    if (jb.t >= 2 && converged_by(chg, jb.t - 1)) return;
    const JobUnit ju = job_unit(jb, u);
    const int n = ju.n, k = ju.k;
    const int *rl = jb.rows ? jb.rows + u * jb.rows_ustride : nullptr;
    const int nrows = rl ? jb.rows_cnt[u * jb.T + jb.t] : n;  // rows of this pass
    if (k <= 0) return;
    const float *cent = jb.cent + u * jb.cent_ustride;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    __shared__ int s_row[AS_ROWS];
    for (int r0 = blockIdx.x * AS_ROWS; r0 < nrows; r0 += gridDim.x * AS_ROWS) {
    __syncthreads();
    if (tid == 0) s_changed = 0;
    if (tid < AS_ROWS) s_row[tid] = r0 + tid < nrows ? (rl ? rl[r0 + tid] : r0 + tid) : -1;
    __syncthreads();

    // rows -> Xs[j][r] (fp32), 16-byte loads of 8 bf16
    for (int e = tid; e < AS_ROWS * 16; e += AS_THREADS) {
        int r = e >> 4, ch = e & 15;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (s_row[r] >= 0) w = *reinterpret_cast<const uint4 *>(mid_row(jb, ju, s_row[r]) + ch * 8);
        uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            Xs[(ch * 8 + 2 * q) * AS_PAD + r] = bf_lo(ws[q]);
            Xs[(ch * 8 + 2 * q + 1) * AS_PAD + r] = bf_hi(ws[q]);
        }
    }
    float b1[4], b2[4];
    int i1[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        b1[a] = INFINITY;
        b2[a] = INFINITY;
        i1[a] = 0x7fffffff;
    }
    for (int c0 = 0; c0 < k; c0 += AS_CENT) {
        __syncthreads();
        for (int e = tid; e < AS_CENT * 32; e += AS_THREADS) {
            int c = e >> 5, j4 = e & 31;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c0 + c < k) v = *reinterpret_cast<const float4 *>(cent + (int64_t)(c0 + c) * MOG_D + j4 * 4);
            Cs[(j4 * 4 + 0) * AS_PAD + c] = v.x;
            Cs[(j4 * 4 + 1) * AS_PAD + c] = v.y;
            Cs[(j4 * 4 + 2) * AS_PAD + c] = v.z;
            Cs[(j4 * 4 + 3) * AS_PAD + c] = v.w;
        }
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int bq = 0; bq < 4; ++bq) acc[a][bq] = 0.f;
#pragma unroll 4
        for (int j = 0; j < MOG_D; ++j) {
            float4 xv = *reinterpret_cast<const float4 *>(Xs + j * AS_PAD + ty * 4);
            float4 cv = *reinterpret_cast<const float4 *>(Cs + j * AS_PAD + tx * 4);
            float xa[4] = {xv.x, xv.y, xv.z, xv.w}, ca[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int bq = 0; bq < 4; ++bq) {
                    float df = __fsub_rn(xa[a], ca[bq]);
                    acc[a][bq] = __fmaf_rn(df, df, acc[a][bq]);
                }
        }
#pragma unroll
        for (int bq = 0; bq < 4; ++bq) {
            int c = c0 + tx * 4 + bq;
            if (c >= k) break;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                float dd = acc[a][bq];
                if (dd < b1[a]) {
                    b2[a] = b1[a];
                    b1[a] = dd;
                    i1[a] = c;
                } else if (dd < b2[a]) {
                    b2[a] = dd;
                }
            }
        }
    }
    // merge the 16 threads that share each row (lanes with equal ty in a half-warp)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            float ob1 = __shfl_xor_sync(0xffffffffu, b1[a], o);
            float ob2 = __shfl_xor_sync(0xffffffffu, b2[a], o);
            int oi1 = __shfl_xor_sync(0xffffffffu, i1[a], o);
            if (ob1 < b1[a] || (ob1 == b1[a] && oi1 < i1[a])) {
                b2[a] = fminf(ob2, b1[a]);
                b1[a] = ob1;
                i1[a] = oi1;
            } else {
                b2[a] = fminf(b2[a], ob1);
            }
        }
    }
    int my_changed = 0;
    if (tx == 0) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            int r = s_row[ty * 4 + a];
            s_unc[ty * 4 + a] = 0;
            if (r < 0) continue;
            int *dst = jb.assign + u * jb.assign_ustride + r;
            if (k == 1 || certified(b1[a], b2[a])) {
                int old = *dst;
                if (old != i1[a]) {
                    *dst = i1[a];
                    ++my_changed;
                }
            } else {
                s_unc[ty * 4 + a] = 1;
            }
        }
        if (my_changed) atomicAdd(&s_changed, my_changed);
    }
    __syncthreads();
    // uncertified rows: one contiguous block of the fallback list per CTA
    if (tid < 32) {
        int f0 = s_unc[tid], f1 = s_unc[tid + 32];
        int cnt = __popc(__ballot_sync(0xffffffffu, f0)) + __popc(__ballot_sync(0xffffffffu, f1));
        if (tid == 0) s_base = cnt ? atomicAdd(jb.fb_cnt + u * jb.T + jb.t, cnt) : 0;
        __syncwarp();
        int base = s_base;
        uint32_t m0 = __ballot_sync(0xffffffffu, f0), m1 = __ballot_sync(0xffffffffu, f1);
        int *fl = jb.fb_list + u * jb.fb_ustride;
        if (f0) fl[base + __popc(m0 & lanemask_lt())] = s_row[tid];
        if (f1) fl[base + __popc(m0) + __popc(m1 & lanemask_lt())] = s_row[32 + tid];
        if (tid == 0 && s_changed) atomicAdd(jb.changed + u * jb.T + jb.t, s_changed);
    }
    }  // rows of this CTA
}

// Rows the fp32 pass could not certify: one warp per row, lanes over centroids.  Only a
// centroid whose fp32 distance is within the fp32 error bound of the smallest can be the
// exact argmin, so fp32 distances pick the candidates and the exact fp64 rule decides
// among them; lowest index on ties.  The row is staged as fp32 in shared memory and read
// by broadcast; each lane streams its centroids with 16-byte loads when they are aligned.
constexpr int FB_THREADS = 256;
constexpr int FB_CTAS = 64;  // CTAs per unit

constexpr int FB_KEEP = 32;  // fp32 distances a lane keeps in registers (k <= 1024)

__global__ void __launch_bounds__(FB_THREADS) k_assign_fallback(AssignJob jb) {
    __shared__ __align__(16) float xs_all[FB_THREADS / 32][MOG_D];
    const int u = blockIdx.y;
    const int *chg = jb.changed + (int64_t)u * jb.T;
    if (jb.t >= 2 && converged_by(chg, jb.t - 1)) return;
    const JobUnit ju = job_unit(jb, u);
    const int k = ju.k;
    const int cnt = jb.fb_cnt[u * jb.T + jb.t];
    const float *cent = jb.cent + u * jb.cent_ustride;
    const bool vec = (reinterpret_cast<uintptr_t>(cent) & 15) == 0;
    const int lane = threadIdx.x & 31;
    float *xs = xs_all[threadIdx.x >> 5];
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int e = warp; e < cnt; e += nwarps) {
        int r = jb.fb_list[u * jb.fb_ustride + e];
        const uint16_t *xr = mid_row(jb, ju, r);
        __syncwarp();
        for (int jj = lane; jj < MOG_D; jj += 32) xs[jj] = bf1(xr[jj]);
        __syncwarp();
        // fp32 distance: difference, fused square-add into four partial sums (only a
        // filter: its threshold's margin is far above the rounding of any summation order)
        auto dist32 = [&](int c) {
            const float *cc = cent + (int64_t)c * MOG_D;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            if (vec) {
                const float4 *c4 = reinterpret_cast<const float4 *>(cc);
                const float4 *x4 = reinterpret_cast<const float4 *>(xs);
#pragma unroll 8
                for (int v = 0; v < MOG_D / 4; ++v) {
                    const float4 cv = __ldg(c4 + v), xv = x4[v];
                    float df = __fsub_rn(xv.x, cv.x);
                    a0 = __fmaf_rn(df, df, a0);
                    df = __fsub_rn(xv.y, cv.y);
                    a1 = __fmaf_rn(df, df, a1);
                    df = __fsub_rn(xv.z, cv.z);
                    a2 = __fmaf_rn(df, df, a2);
                    df = __fsub_rn(xv.w, cv.w);
                    a3 = __fmaf_rn(df, df, a3);
                }
            } else {
#pragma unroll 8
                for (int jj = 0; jj < MOG_D; jj += 4) {
                    float df = __fsub_rn(xs[jj], __ldg(cc + jj));
                    a0 = __fmaf_rn(df, df, a0);
                    df = __fsub_rn(xs[jj + 1], __ldg(cc + jj + 1));
                    a1 = __fmaf_rn(df, df, a1);
                    df = __fsub_rn(xs[jj + 2], __ldg(cc + jj + 2));
                    a2 = __fmaf_rn(df, df, a2);
                    df = __fsub_rn(xs[jj + 3], __ldg(cc + jj + 3));
                    a3 = __fmaf_rn(df, df, a3);
                }
            }
            return (a0 + a1) + (a2 + a3);
        };
        // fp32 distances to every centroid, kept in registers when k <= FB_KEEP * 32
        float dk[FB_KEEP];
        const bool keep = k <= FB_KEEP * 32;
        float b32 = INFINITY;
        if (keep) {
#pragma unroll
            for (int i = 0; i < FB_KEEP; ++i) {
                const int c = lane + 32 * i;
                dk[i] = c < k ? dist32(c) : INFINITY;
                b32 = fminf(b32, dk[i]);
            }
        } else {
            for (int c = lane; c < k; c += 32) b32 = fminf(b32, dist32(c));
        }
        b32 = warp_min(b32);
        // every centroid whose exact distance can be the smallest (kCertRel is above the
        // relative fp32 error on each side)
        const float thr = b32 * (1.f + 2.5f * kCertRel);
        auto d32 = [&](int i, int c) { return keep ? dk[i] : dist32(c); };
        // the candidates' double-float distances: the best and the runner-up over the warp
        double v1 = INFINITY, v2 = INFINITY;
        int i1 = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < FB_KEEP; ++i) {
            for (int c = lane + 32 * i; c < k; c += 32 * FB_KEEP) {  // (one pass when kept)
                if (d32(i, c) > thr) continue;
                const double v = df_dist(xs, cent + (int64_t)c * MOG_D);
                if (v < v1) {
                    v2 = v1;
                    v1 = v;
                    i1 = c;
                } else if (v < v2) {
                    v2 = v;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double ov1 = __shfl_xor_sync(0xffffffffu, v1, o), ov2 = __shfl_xor_sync(0xffffffffu, v2, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i1, o);
            if (ov1 < v1 || (ov1 == v1 && oi < i1)) {
                v2 = fmin(v1, ov2);
                v1 = ov1;
                i1 = oi;
            } else {
                v2 = fmin(v2, ov1);
            }
        }
        double best = v1;
        int bi = i1;
        const double win = 2.0 * kDfRel * v2 + 1e-300;  // both values' bounds, and zero
        if (v2 != INFINITY && !(v2 - v1 > win)) {  // (a single candidate is the argmin)
            // not separated: the fp64 rule over every candidate that may be the smallest
            best = INFINITY;
            bi = 0x7fffffff;
            const double lim = v1 + win;  // the fp64 argmin's double-float value is below this
            for (int c = lane; c < k; c += 32) {
                if (dist32(c) > thr) continue;  // (rare: recomputed)
                if (df_dist(xs, cent + (int64_t)c * MOG_D) > lim) continue;
                const double dd = exact_dist(xr, cent + (int64_t)c * MOG_D);
                if (dd < best) {
                    best = dd;
                    bi = c;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const double ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ob < best || (ob == best && oi < bi)) {
                    best = ob;
                    bi = oi;
                }
            }
        }
        if (lane == 0) {
            int *dst = jb.assign + u * jb.assign_ustride + r;
            if (*dst != bi) {
                *dst = bi;
                atomicAdd(jb.changed + u * jb.T + jb.t, 1);
            }
        }
    }
}

// ------------------------------------------------------------------------------------
// Stable counting sort of the first-level assignment: per-chunk histograms, a column
// scan over chunks, a scan over clusters, then one warp per chunk scatters its rows in
// order (ranks inside a warp from __match_any_sync).  perm lists positions S + i.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ bool l1_skip(const Dev &dv, int u, int t) {
    return t >= 1 && converged_by(dv.changed + (int64_t)u * dv.T1, t);
}

__global__ void k_sort_hist(Dev dv, int t) {
    extern __shared__ int hs[];
    const int u = blockIdx.y, chunk = blockIdx.x;
    if (l1_skip(dv, u, t)) return;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int n = ui[UI_NMID], C = ui[UI_C];
    const int lo = chunk * SORT_CHUNK;
    if (lo >= n) return;
    for (int c = threadIdx.x; c < C; c += blockDim.x) hs[c] = 0;
    __syncthreads();
    const int *a = dv.l1_assign + (int64_t)u * dv.n_cap;
    for (int i = lo + threadIdx.x; i < min(n, lo + SORT_CHUNK); i += blockDim.x) atomicAdd(&hs[a[i]], 1);
    __syncthreads();
    int *h = dv.hist + ((int64_t)u * dv.nchunks + chunk) * dv.c_max;
    for (int c = threadIdx.x; c < C; c += blockDim.x) h[c] = hs[c];
}

__global__ void k_sort_colscan(Dev dv, int t) {
    const int u = blockIdx.y;
    if (l1_skip(dv, u, t)) return;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int n = ui[UI_NMID], C = ui[UI_C];
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    const int nch = (int)ceil_div64(n, SORT_CHUNK);
    const int *h = dv.hist + (int64_t)u * dv.nchunks * dv.c_max + c;
    int *o = dv.offs + (int64_t)u * dv.nchunks * dv.c_max + c;
    // the chunks' counts are loaded CS_BATCH at a time, so that their latencies overlap
    constexpr int CS_BATCH = 16;
    int run = 0;
    for (int k0 = 0; k0 < nch; k0 += CS_BATCH) {
        int v[CS_BATCH];
#pragma unroll
        for (int j = 0; j < CS_BATCH; ++j) v[j] = k0 + j < nch ? h[(int64_t)(k0 + j) * dv.c_max] : 0;
#pragma unroll
        for (int j = 0; j < CS_BATCH; ++j)
            if (k0 + j < nch) {
                o[(int64_t)(k0 + j) * dv.c_max] = run;
                run += v[j];
            }
    }
    dv.ctot[(int64_t)u * dv.c_max + c] = run;
}

// exclusive scan of the cluster totals: coff[u][0..C]
__global__ void k_sort_base(Dev dv, int t) {
    __shared__ int wsum[32];
    const int u = blockIdx.x;
    if (l1_skip(dv, u, t)) return;
    const int C = dv.unit_info[u * UI_STRIDE + UI_C];
    const int *tot = dv.ctot + (int64_t)u * dv.c_max;
    int *co = dv.coff + (int64_t)u * (dv.c_max + 1);
    const int per = (int)ceil_div64(C, blockDim.x);
    const int c0 = threadIdx.x * per;
    int s = 0;
    for (int c = c0; c < min(C, c0 + per); ++c) s += tot[c];
    // block exclusive scan of s
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
        int v = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
        int inc2 = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, inc2, o);
            if (lane >= o) inc2 += y;
        }
        wsum[lane] = inc2 - v;
    }
    __syncthreads();
    int run = wsum[w] + incl - s;
    for (int c = c0; c < min(C, c0 + per); ++c) {
        co[c] = run;
        run += tot[c];
    }
    if (c0 < C && c0 + per >= C) co[C] = run;
    if (C == 0 && threadIdx.x == 0) co[0] = 0;
}

__global__ void k_sort_scatter(Dev dv, int t) {
    extern __shared__ int cnt[];
    const int u = blockIdx.y, chunk = blockIdx.x;
    if (l1_skip(dv, u, t)) return;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int n = ui[UI_NMID], C = ui[UI_C], S = ui[UI_S];
    const int lo = chunk * SORT_CHUNK;
    if (lo >= n) return;
    const int lane = threadIdx.x;
    for (int c = lane; c < C; c += 32) cnt[c] = 0;
    __syncwarp();
    const int *a = dv.l1_assign + (int64_t)u * dv.n_cap;
    const int *o = dv.offs + ((int64_t)u * dv.nchunks + chunk) * dv.c_max;
    const int *co = dv.coff + (int64_t)u * (dv.c_max + 1);
    int *perm = dv.permA + (int64_t)u * dv.n_cap;
    const int hi = min(n, lo + SORT_CHUNK);
    for (int i0 = lo; i0 < hi; i0 += 32) {
        int i = i0 + lane;
        bool valid = i < hi;
        int c = valid ? a[i] : -1;
        uint32_t grp = __match_any_sync(0xffffffffu, c);
        int rank = __popc(grp & lanemask_lt());
        if (valid) {
            int pos = co[c] + o[c] + cnt[c] + rank;
            perm[pos] = S + i;
        }
        __syncwarp();
        if (valid && rank == 0) cnt[c] += __popc(grp);
        __syncwarp();
    }
}

// Centroid update: fp32 Kahan mean of the members in sorted (position) order; 8 warps
// each sum a contiguous slice, combined in warp order.  Empty clusters keep the centroid.
__global__ void __launch_bounds__(256) k_l1_update(Dev dv, int t) {
    __shared__ float ps[8][MOG_D];
    __shared__ float pc[8][MOG_D];
    const int u = blockIdx.y, c = blockIdx.x;
    if (l1_skip(dv, u, t)) return;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    if (c >= ui[UI_C]) return;
    const int b = ui[UI_B], h = u % dv.h_kv;
    const int *co = dv.coff + (int64_t)u * (dv.c_max + 1);
    const int lo = co[c], n = co[c + 1] - lo;
    if (n == 0) return;
    const int *perm = dv.permA + (int64_t)u * dv.n_cap + lo;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = (int)((int64_t)w * n / 8), m1 = (int)((int64_t)(w + 1) * n / 8);
    Kahan acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q].init();
    // members are loaded UP_BATCH at a time (their latencies overlap) and added in order
    constexpr int UP_BATCH = 8;
    for (int m = m0; m < m1; m += UP_BATCH) {
        uint2 wv[UP_BATCH];
#pragma unroll
        for (int j = 0; j < UP_BATCH; ++j)
            if (m + j < m1) wv[j] = *reinterpret_cast<const uint2 *>(dv.krow(b, h, perm[m + j]) + lane * 4);
#pragma unroll
        for (int j = 0; j < UP_BATCH; ++j)
            if (m + j < m1) {
                acc[0].add(bf_lo(wv[j].x));
                acc[1].add(bf_hi(wv[j].x));
                acc[2].add(bf_lo(wv[j].y));
                acc[3].add(bf_hi(wv[j].y));
            }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        ps[w][lane * 4 + q] = acc[q].s;
        pc[w][lane * 4 + q] = acc[q].c;
    }
    __syncthreads();
    if (threadIdx.x < MOG_D) {
        Kahan tot;
        tot.init();
        for (int ww = 0; ww < 8; ++ww) {
            tot.add(ps[ww][threadIdx.x]);
            tot.add(-pc[ww][threadIdx.x]);
        }
        dv.cent[((int64_t)u * dv.c_max + c) * MOG_D + threadIdx.x] = tot.s / (float)n;
    }
}

// ------------------------------------------------------------------------------------
// k-means++ seeding of the first level (a variant).  Two launches per seed r:
//  k_pp_pick (one CTA per unit) draws seed r from the squared distances D2 left by round
//    r - 1;
//  k_pp_update (CTAs over the mid keys) lowers each key's D2 to its distance to seed r and
//    writes each CTA's sum of D2.  Every round reads every mid key once.
// Both are launched as programmatic dependents, each waiting for its predecessor before
// it reads what that one wrote.  D2 and the CTA sums alternate between two buffers by the
// parity of r.
// ------------------------------------------------------------------------------------

// fp32 squared distance of a bf16 key row to c (fp32, shared memory): each difference
// rounded to fp32, four partial sums (dimension j into sum j mod 4) by fused multiply-add
// in increasing j, then (s0 + s1) + (s2 + s3).  Four chains instead of one keep the
// dependent adds from limiting the kernel.
__device__ __forceinline__ float pp_dist(const uint16_t *x, const float *c) {
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    uint4 rv[16];  // the row's loads issued together: each 32-byte sector by consecutive loads
#pragma unroll
    for (int q = 0; q < 16; ++q) rv[q] = xv[q];
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const uint4 v = rv[q];
        const float *cq = c + 8 * q;
        float d;
        d = __fsub_rn(bf_lo(v.x), cq[0]); s0 = __fmaf_rn(d, d, s0);
        d = __fsub_rn(bf_hi(v.x), cq[1]); s1 = __fmaf_rn(d, d, s1);
        d = __fsub_rn(bf_lo(v.y), cq[2]); s2 = __fmaf_rn(d, d, s2);
        d = __fsub_rn(bf_hi(v.y), cq[3]); s3 = __fmaf_rn(d, d, s3);
        d = __fsub_rn(bf_lo(v.z), cq[4]); s0 = __fmaf_rn(d, d, s0);
        d = __fsub_rn(bf_hi(v.z), cq[5]); s1 = __fmaf_rn(d, d, s1);
        d = __fsub_rn(bf_lo(v.w), cq[6]); s2 = __fmaf_rn(d, d, s2);
        d = __fsub_rn(bf_hi(v.w), cq[7]); s3 = __fmaf_rn(d, d, s3);
    }
    return __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
}

// Prefix over the CTA of one double per thread, in one fixed order (shuffles within the
// warps, then the warps' sums in index order): the thread's exclusive prefix and the total.
struct PPScan {
    double excl, total;
};
__device__ __forceinline__ PPScan pp_scan(double v, double *s_w) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    double ex = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) ex = 0.0;
    if (lane == 31) s_w[warp] = inc;
    __syncthreads();
    double base = 0.0, tot = 0.0;
    for (int w = 0; w < PP_THREADS / 32; ++w) {
        if (w == warp) base = tot;
        tot += s_w[w];
    }
    __syncthreads();  // s_w is reused by the next scan
    return {base + ex, tot};
}

__global__ void __launch_bounds__(PP_THREADS) k_pp_pick(Dev dv, int r) {
    const int u = blockIdx.x, tid = threadIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], n = ui[UI_NMID];
    if (r >= C || n == 0) return;
    pdl_wait();  // D2 and the CTA sums of round r - 1 are written
    pdl_trigger();
    const int nb = (n + PP_ROWS - 1) / PP_ROWS;
    __shared__ double s_w[PP_THREADS / 32];
    __shared__ int s_blk, s_pick, s_lastpos;
    __shared__ double s_pre;
    if (tid == 0) {
        s_blk = s_pick = INT_MAX;
        s_lastpos = -1;
    }
    const int64_t U = dv.units, cm = dv.c_max;
    double ur = dv.pp_draw[u * cm + r];
    if (!(ur >= 0.0 && ur < 1.0)) {  // outside [0, 1) (or NaN): clamp and report
        if (tid == 0) flag_error(dv.status, ST_BAD_INDEX);
        ur = ur >= 1.0 ? 0x1.fffffffffffffp-1 : 0.0;
    }
    const int pr = (r + 1) & 1;
    const float *d2p = dv.pp_d2 + ((int64_t)pr * U + u) * dv.n_cap;
    const double *partp = dv.pp_part + ((int64_t)pr * U + u) * dv.pp_nblk;

    int j = min((int)floor(ur * (double)n), n - 1);  // seed 0, or every key on a seed
    if (r > 0) {
        // the CTA sums of round r - 1: the first CTA whose running sum exceeds ur * total
        const int per = (nb + PP_THREADS - 1) / PP_THREADS;
        const int e0 = min(nb, tid * per), e1 = min(nb, e0 + per);
        double loc = 0.0;
        for (int e = e0; e < e1; ++e) loc += partp[e];
        const PPScan sc = pp_scan(loc, s_w);
        if (sc.total > 0.0) {
            const double target = ur * sc.total;
            double run = sc.excl;
            for (int e = e0; e < e1; ++e) {
                const double nx = run + partp[e];
                if (nx > target) {
                    atomicMin(&s_blk, e);
                    break;
                }
                run = nx;
            }
            __syncthreads();
            int B = s_blk;
            if (B != INT_MAX) {
                if (B >= e0 && B < e1) {  // its owner: the running sum before it
                    double pre = sc.excl;
                    for (int e = e0; e < B; ++e) pre += partp[e];
                    s_pre = pre;
                }
            } else {  // ur * total rounded up to the total: the last CTA with a positive sum
                for (int e = e1 - 1; e >= e0; --e)
                    if (partp[e] > 0.0) {
                        atomicMax(&s_lastpos, e);
                        break;
                    }
            }
            __syncthreads();
            const bool found = B != INT_MAX;
            if (!found) B = max(s_lastpos, 0);
            __syncthreads();
            if (tid == 0) s_lastpos = -1;
            // inside CTA B, keys in position order, PP_PER consecutive keys a thread (the
            // order in which k_pp_update summed them)
            const int i0 = B * PP_ROWS + tid * PP_PER;
            double l2 = 0.0;
            for (int k = 0; k < PP_PER; ++k)
                if (i0 + k < n) l2 += (double)d2p[i0 + k];
            const PPScan s2 = pp_scan(l2, s_w);  // (its barrier also orders s_lastpos)
            if (found) {
                double rr = s_pre + s2.excl;
                for (int k = 0; k < PP_PER && i0 + k < n; ++k) {
                    const double nx = rr + (double)d2p[i0 + k];
                    if (nx > target) {
                        atomicMin(&s_pick, i0 + k);
                        break;
                    }
                    rr = nx;
                }
            }
            __syncthreads();
            if (s_pick == INT_MAX) {  // no crossing (rounding): the last key with D2 > 0
                for (int k = PP_PER - 1; k >= 0; --k)
                    if (i0 + k < n && d2p[i0 + k] > 0.f) {
                        atomicMax(&s_lastpos, i0 + k);
                        break;
                    }
                __syncthreads();
                j = s_lastpos >= 0 ? s_lastpos : B * PP_ROWS;
            } else {
                j = s_pick;
            }
        }
    }
    if (tid == 0) dv.pp_idx[u * cm + r] = j;
}

// One CTA per PP_ROWS mid keys, PP_PER a thread (consecutive keys across the threads, so
// that a warp's loads cover 32 adjacent rows).  Each thread reads its own rows from global
// memory: measured faster here than staging tiles in shared memory by cp.async (the
// per-SM limit on outstanding copies) or by one bulk copy per row.
__global__ void __launch_bounds__(PP_THREADS) k_pp_update(Dev dv, int r) {
    const int u = blockIdx.y, blk = blockIdx.x, tid = threadIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], n = ui[UI_NMID];
    const int nb = (n + PP_ROWS - 1) / PP_ROWS;
    if (r >= C - 1 || n == 0 || blk >= nb) return;
    __shared__ double s_w[PP_THREADS / 32];
    __shared__ float s_c[MOG_D];
    __shared__ float s_d2[PP_ROWS];
    const int64_t U = dv.units, cm = dv.c_max;
    const int pr = (r + 1) & 1, cr = r & 1;
    const int b = ui[UI_B], h = u % dv.h_kv, S = ui[UI_S];
    pdl_wait();  // seed r is picked, D2 of round r - 1 is written
    pdl_trigger();
    const float *d2p = dv.pp_d2 + ((int64_t)pr * U + u) * dv.n_cap;
    float *d2c = dv.pp_d2 + ((int64_t)cr * U + u) * dv.n_cap;
    const int j = dv.pp_idx[u * cm + r];
    if (tid < MOG_D) s_c[tid] = bf1(dv.krow(b, h, S + j)[tid]);
    __syncthreads();
    const int base = blk * PP_ROWS;
#pragma unroll 1
    for (int k = 0; k < PP_PER; ++k) {
        const int i = base + k * PP_THREADS + tid;
        float v = 0.f;
        if (i < n) {
            const float dd = pp_dist(dv.krow(b, h, S + i), s_c);
            v = r == 0 ? dd : fminf(d2p[i], dd);
            d2c[i] = v;
        }
        s_d2[k * PP_THREADS + tid] = v;
    }
    __syncthreads();
    double loc = 0.0;  // summed in the order in which k_pp_pick scans this CTA's keys
    for (int q = 0; q < PP_PER; ++q) loc += (double)s_d2[tid * PP_PER + q];
    const PPScan sc = pp_scan(loc, s_w);
    if (tid == 0) dv.pp_part[((int64_t)cr * U + u) * dv.pp_nblk + blk] = sc.total;
}

template <typename Kern, typename... Args>
static cudaError_t launch_pdl_km(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__global__ void k_l1_init(Dev dv) {
    const int u = blockIdx.y, c = blockIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], n = ui[UI_NMID];
    if (c >= C || n == 0) return;
    const int b = ui[UI_B], h = u % dv.h_kv;
    // strided seeds, or the k-means++ seeds
    const int64_t pos = ui[UI_S] + (dv.kpp ? (int64_t)dv.pp_idx[(int64_t)u * dv.c_max + c] : (int64_t)c * n / C);
    const uint16_t *row = dv.krow(b, h, pos);
    for (int j = threadIdx.x; j < MOG_D; j += blockDim.x)
        dv.cent[((int64_t)u * dv.c_max + c) * MOG_D + j] = bf1(row[j]);
}

// ------------------------------------------------------------------------------------
// Second level + summaries, one CTA per (unit, cluster).
// ------------------------------------------------------------------------------------

// One assignment of row x (bf16, 128) among k centroids cs[k][d] in shared memory: the
// direct fp32 distance in index order with its certificate; when it fails, the exact fp64
// rule over the centroids whose fp32 distance is within the fp32 error bound of the
// smallest (no other centroid can be the exact argmin; fp64 is slow on this GPU).
// The row is re-read (L1-resident) for each centroid rather than held in registers.
__device__ __forceinline__ int assign_small(const uint16_t *x, const float *cs, int k) {
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    auto dist32 = [&](int l) {
        const float *c = cs + l * MOG_D;
        float acc = 0.f;
#pragma unroll 4
        for (int q = 0; q < 16; ++q) {
            const uint4 v = xv[q];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float d0 = __fsub_rn(bf_lo(w[e]), c[8 * q + 2 * e]);
                acc = __fmaf_rn(d0, d0, acc);
                float d1 = __fsub_rn(bf_hi(w[e]), c[8 * q + 2 * e + 1]);
                acc = __fmaf_rn(d1, d1, acc);
            }
        }
        return acc;
    };
    float b1 = INFINITY, b2 = INFINITY;
    int i1 = 0;
    for (int l = 0; l < k; ++l) {
        const float acc = dist32(l);
        if (acc < b1) {
            b2 = b1;
            b1 = acc;
            i1 = l;
        } else if (acc < b2) {
            b2 = acc;
        }
    }
    if (k == 1 || certified(b1, b2)) return i1;
    const float thr = b1 * (1.f + 2.5f * kCertRel);
    double best = INFINITY;
    int bi = 0;
    for (int l = 0; l < k; ++l) {
        if (dist32(l) > thr) continue;
        double dd = exact_dist(x, cs + l * MOG_D);
        if (dd < best) {
            best = dd;
            bi = l;
        }
    }
    return bi;
}

constexpr int L2_THREADS = 256;
constexpr int L2_WARPS = L2_THREADS / 32;
constexpr int L2_CST = 160;  // bf16 row stride of the centroid images (320 B)

// Second-level assignment of n rows (row(m), m < n) among the k <= 32 centroids cs[k][d]
// (fp32, shared memory), by the whole block.  The approximate distance |c|^2 - 2 k.c is
// computed with mma.sync (keys bf16; centroids split into bf16 high + low parts; fp32
// accumulate) and a row keeps its best centroid when it passes the same certificate as
// the first-level tensor-core pass; the other rows take assign_small.  `img` (20 KB of
// shared memory) receives the centroid images, s_cn[32] the squared norms.  sa[m] holds
// the previous assignment (-1 if none) and receives the new one; returns this thread's
// count of changed rows.
//
// Fragment layout: k-step pair p (dimensions 32p..32p+31) is read as one 16-byte word
// group per thread (words 16p + 4q .. +3, q = lane % 4) of both the key rows and the
// centroid images; words 0-1 feed the even k-step and 2-3 the odd one, with the MMA's
// logical pairs q and q + 4 on the first and second word.  Keys and centroids use the
// same map, so the dot products are those of the rows.
template <class RowFn>
__device__ int l2_assign(RowFn row, int *sa, int n, int k, const float *cs, uint8_t *img,
                         float *s_cn) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t *chi = reinterpret_cast<uint32_t *>(img);
    uint32_t *clo = chi + MOG_MAX_L * L2_CST / 2;
    for (int e = tid; e < MOG_MAX_L * MOG_D / 2; e += L2_THREADS) {
        const int l = e >> 6, p = e & 63;
        float c0 = 0.f, c1 = 0.f;
        if (l < k) {
            c0 = cs[l * MOG_D + 2 * p];
            c1 = cs[l * MOG_D + 2 * p + 1];
        }
        const uint32_t hi = cvt_bf2(c0, c1);
        chi[l * (L2_CST / 2) + p] = hi;
        clo[l * (L2_CST / 2) + p] = cvt_bf2(__fsub_rn(c0, bf_lo(hi)), __fsub_rn(c1, bf_hi(hi)));
    }
    for (int l = warp; l < MOG_MAX_L; l += L2_WARPS) {
        float s2 = 0.f;
        if (l < k)
            for (int jj = lane; jj < MOG_D; jj += 32) s2 = __fmaf_rn(cs[l * MOG_D + jj], cs[l * MOG_D + jj], s2);
#pragma unroll
        for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        if (lane == 0) s_cn[l] = l < k ? s2 : INFINITY;
    }
    __syncthreads();
    float cmax = 0.f;
    for (int l = 0; l < k; ++l) cmax = fmaxf(cmax, s_cn[l]);
    const int g = lane >> 2, q = lane & 3;
    const int NT = (k + 7) >> 3;
    int my = 0;
    for (int tile = warp; tile * 16 < n; tile += L2_WARPS) {
        const int m0 = tile * 16 + g, m1 = m0 + 8;
        const uint4 *p0 = reinterpret_cast<const uint4 *>(row(min(m0, n - 1)));
        const uint4 *p1 = reinterpret_cast<const uint4 *>(row(min(m1, n - 1)));
        uint4 x0[4], x1[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            x0[p] = p0[4 * p + q];
            x1[p] = p1[4 * p + q];
        }
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t ae[4] = {x0[p].x, x1[p].x, x0[p].y, x1[p].y};
            const uint32_t ao[4] = {x0[p].z, x1[p].z, x0[p].w, x1[p].w};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                if (nt < NT) {
                    const int off = (nt * 8 + g) * (L2_CST / 2) + 16 * p + 4 * q;
                    const uint4 bh = *reinterpret_cast<const uint4 *>(chi + off);
                    const uint4 bl = *reinterpret_cast<const uint4 *>(clo + off);
                    mma_bf16(acc[nt], ae, bh.x, bh.y);
                    mma_bf16(acc[nt], ae, bl.x, bl.y);
                    mma_bf16(acc[nt], ao, bh.z, bh.w);
                    mma_bf16(acc[nt], ao, bl.z, bl.w);
                }
            }
        }
        // |k|^2 of both rows (fp32)
        float kn[2] = {0.f, 0.f};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t w0[4] = {x0[p].x, x0[p].y, x0[p].z, x0[p].w};
            const uint32_t w1[4] = {x1[p].x, x1[p].y, x1[p].z, x1[p].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kn[0] = __fmaf_rn(bf_lo(w0[e]), bf_lo(w0[e]), kn[0]);
                kn[0] = __fmaf_rn(bf_hi(w0[e]), bf_hi(w0[e]), kn[0]);
                kn[1] = __fmaf_rn(bf_lo(w1[e]), bf_lo(w1[e]), kn[1]);
                kn[1] = __fmaf_rn(bf_hi(w1[e]), bf_hi(w1[e]), kn[1]);
            }
        }
        float b1[2] = {INFINITY, INFINITY}, b2[2] = {INFINITY, INFINITY};
        int i1[2] = {0, 0};
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            if (nt < NT) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = e >> 1, col = nt * 8 + 2 * q + (e & 1);
                    const float a = __fmaf_rn(-2.f, acc[nt][e], s_cn[col]);
                    if (a < b1[r]) {
                        b2[r] = b1[r];
                        b1[r] = a;
                        i1[r] = col;
                    } else if (a < b2[r]) {
                        b2[r] = a;
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                const float ob1 = __shfl_xor_sync(0xffffffffu, b1[r], o);
                const float ob2 = __shfl_xor_sync(0xffffffffu, b2[r], o);
                const int oi = __shfl_xor_sync(0xffffffffu, i1[r], o);
                if (ob1 < b1[r] || (ob1 == b1[r] && oi < i1[r])) {
                    b2[r] = fminf(b1[r], ob2);
                    b1[r] = ob1;
                    i1[r] = oi;
                } else {
                    b2[r] = fminf(b2[r], ob1);
                }
            }
            kn[r] += __shfl_xor_sync(0xffffffffu, kn[r], 1);
            kn[r] += __shfl_xor_sync(0xffffffffu, kn[r], 2);
        }
        if (q == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int m = r ? m1 : m0;
                if (m < n) {
                    const bool cert = k == 1 || (b2[r] - TC_F * (kn[r] + cmax) >
                                                 b1[r] + TC_F * (kn[r] + s_cn[i1[r]]));
                    const int old = sa[m];
                    if (!cert) {
                        sa[m] = old - 64;  // undecided: the exact pass below
                    } else if (i1[r] != old) {
                        sa[m] = i1[r];
                        ++my;
                    }
                }
            }
        }
    }
    __syncthreads();
    for (int m = tid; m < n; m += L2_THREADS) {
        const int v = sa[m];
        if (v < -32) {
            const int a = assign_small(row(m), cs, k);
            sa[m] = a;
            my += a != v + 64;
        }
    }
    return my;
}

struct SegJob {  // standalone segmented assignment (parity export)
    const uint16_t *x;
    int64_t ld;
    const int32_t *rows, *seg_off;
    const float *cent;
    int k;
    int32_t *assign;
};

// One CTA per segment: the segment's rows against its own k centroids, by l2_assign.
__global__ void __launch_bounds__(L2_THREADS) k_assign_segments(SegJob jb) {
    extern __shared__ __align__(16) uint8_t segraw[];
    float *cs = reinterpret_cast<float *>(segraw);
    uint8_t *img = segraw + MOG_MAX_L * MOG_D * sizeof(float);
    __shared__ float s_cn[MOG_MAX_L];
    const int s = blockIdx.x;
    const int lo = jb.seg_off[s], n = jb.seg_off[s + 1] - lo;
    for (int e = threadIdx.x; e < jb.k * MOG_D; e += blockDim.x)
        cs[e] = jb.cent[(int64_t)s * jb.k * MOG_D + e];
    int32_t *sa = jb.assign + lo;
    for (int m = threadIdx.x; m < n; m += blockDim.x) sa[m] = -1;
    __syncthreads();
    const int32_t *rows = jb.rows + lo;
    l2_assign([&](int m) { return jb.x + (int64_t)rows[m] * jb.ld; }, sa, n, jb.k, cs, img, s_cn);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Row streaming for the per-cluster passes: the rows pos[a..e) of one KV head pass through
// a ring of L2_NS shared-memory stages of L2_CH rows (keys, and values when with_v), in
// order, with L2_NS - 1 stages in flight.  `grp` threads (thread ids gt = 0..grp-1) share
// the ring and synchronise on named barrier `bar`; body(m0, cnt, k, v) sees rows m0..m0+cnt
// as k[r * d + j], v[r * d + j].
constexpr int L2_CH = 32;
constexpr int L2_NS = 3;
constexpr int L2_ROWB = MOG_D * 2;
constexpr int L2_RING = L2_NS * 2 * L2_CH * L2_ROWB;  // 48 KB: stages of keys + values

template <class Body>
__device__ __forceinline__ void stream_rows(const Dev &dv, int b, int h, const int *pos, int a,
                                            int e, bool with_v, uint8_t *ring, int gt, int grp,
                                            int bar, Body &&body) {
    const int nch = (e - a + L2_CH - 1) / L2_CH;
    const int mats = with_v ? 2 : 1;
    const int stage_bytes = mats * L2_CH * L2_ROWB;
    auto issue = [&](int ci) {
        if (ci < nch) {
            uint8_t *st = ring + (ci % L2_NS) * stage_bytes;
            const int m0 = a + ci * L2_CH;
            for (int p = gt; p < mats * L2_CH * 16; p += grp) {
                const int mat = p / (L2_CH * 16), r = (p >> 4) & (L2_CH - 1), q = p & 15;
                const int m = m0 + r;
                const bool ok = m < e;
                const int64_t ps = pos[ok ? m : a];
                const uint16_t *src = (mat ? dv.vrow(b, h, ps) : dv.krow(b, h, ps)) + q * 8;
                cp_async16(smem_u32(st + (mat * L2_CH + r) * L2_ROWB + q * 16), src, ok ? 16 : 0);
            }
        }
        cp_async_commit();
    };
    for (int s = 0; s < L2_NS - 1; ++s) issue(s);
    for (int ci = 0; ci < nch; ++ci) {
        cp_async_wait<L2_NS - 2>();
        named_sync(bar, grp);  // chunk ci landed for every thread; chunk ci-1 consumed
        issue(ci + L2_NS - 1);
        const uint8_t *st = ring + (ci % L2_NS) * stage_bytes;
        const int m0 = a + ci * L2_CH;
        body(m0, min(L2_CH, e - m0), reinterpret_cast<const uint16_t *>(st),
             reinterpret_cast<const uint16_t *>(st + L2_CH * L2_ROWB));
    }
    cp_async_wait<0>();
    named_sync(bar, grp);  // the ring is free again
}

// One CTA per (unit, cluster).  With do_kmeans: the second-level Lloyd loop over the
// cluster's members (position order, strided seeding), then the final stable order by
// (subcluster, position).  Then the summaries of the cluster and its subclusters.
// Member rows are read through the shared-memory ring; every mean is an fp32 Kahan sum
// in (subcluster, position) order, every variance a second pass about that mean.
__global__ void __launch_bounds__(L2_THREADS, 3) k_l2_stats(Dev dv, int do_kmeans, TraceDev tr) {
    extern __shared__ __align__(16) uint8_t l2raw[];
    float *cs = reinterpret_cast<float *>(l2raw);  // [L][d] centroids, then subcluster key means
    uint8_t *ring = l2raw + MOG_MAX_L * MOG_D * sizeof(float);
    __shared__ int cnt[MOG_MAX_L], pref[MOG_MAX_L + 1];
    __shared__ int whist[L2_WARPS][MOG_MAX_L];
    __shared__ int s_changed, s_half;
    __shared__ float s_cm[MOG_D], s_cn[MOG_MAX_L];
    const int u = blockIdx.y, c = blockIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], L = ui[UI_L];
    if (c >= C) return;
    if (!do_kmeans && *(volatile const int *)dv.status != 0) return;  // rejected partition
    const int b = ui[UI_B], h = u % dv.h_kv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = tid & (MOG_D - 1);
    const bool upper = tid >= MOG_D;
    int *so = dv.sub_off + u * dv.sub_off_stride;
    int *permF = dv.perm + (int64_t)u * dv.n_cap;
    int lo, n;
    if (do_kmeans) {
        const int *co = dv.coff + (int64_t)u * (dv.c_max + 1);
        lo = co[c];
        n = co[c + 1] - lo;
        if (c == 0 && tid == 0) {  // record the first-level step count
            int steps = dv.T1;
            const int *chg = dv.changed + (int64_t)u * dv.T1;
            for (int s = 1; s < dv.T1; ++s)
                if (chg[s] == 0) { steps = s + 1; break; }
            dv.l1_steps[u] = ui[UI_NMID] > 0 ? steps : 0;
        }
    } else {
        lo = so[c * L];
        n = so[(c + 1) * L] - lo;
    }
    if (do_kmeans) {
        const int *pA = dv.permA + (int64_t)u * dv.n_cap + lo;
        int *sa = dv.sub_assign + (int64_t)u * dv.n_cap + lo;
        // Stable order of the members by subcluster into permF[lo, lo + n): warp w scatters
        // the contiguous member range [w n / W, (w + 1) n / W) after the members of every
        // earlier subcluster and of its subcluster in earlier warps.  Leaves cnt, pref and
        // s_half (the subcluster where the member offsets cross n / 2).
        auto order_members = [&]() {
            const int m_b = (int)((int64_t)warp * n / L2_WARPS);
            const int m_e = (int)((int64_t)(warp + 1) * n / L2_WARPS);
            int *wh = whist[warp];
            wh[lane] = 0;
            __syncwarp();
            for (int m = m_b + lane; m - lane < m_e; m += 32) {
                const int a = m < m_e ? sa[m] : -1;
                const uint32_t g = __match_any_sync(0xffffffffu, a);
                if (a >= 0 && (g & lanemask_lt()) == 0) wh[a] += __popc(g);
                __syncwarp();
            }
            __syncthreads();
            if (tid < L) {
                int t = 0;
                for (int w = 0; w < L2_WARPS; ++w) t += whist[w][tid];
                cnt[tid] = t;
            }
            __syncthreads();
            if (tid == 0) {
                pref[0] = 0;
                int best = 0;
                for (int l = 0; l < L; ++l) {
                    pref[l + 1] = pref[l] + cnt[l];
                    if (abs(2 * pref[l + 1] - n) < abs(2 * pref[best] - n)) best = l + 1;
                }
                s_half = best;
            }
            __syncthreads();
            if (tid < L) {
                int run = pref[tid];
                for (int w = 0; w < L2_WARPS; ++w) {
                    const int t = whist[w][tid];
                    whist[w][tid] = run;
                    run += t;
                }
            }
            __syncthreads();
            for (int m = m_b + lane; m - lane < m_e; m += 32) {
                const int a = m < m_e ? sa[m] : -1;
                const uint32_t g = __match_any_sync(0xffffffffu, a);
                const int base = a >= 0 ? wh[a] : 0;
                __syncwarp();
                if (a >= 0) {
                    permF[lo + base + __popc(g & lanemask_lt())] = pA[m];
                    if ((g & lanemask_lt()) == 0) wh[a] = base + __popc(g);
                }
                __syncwarp();
            }
            __syncthreads();
        };
        if (n > 0) {
            for (int e = tid; e < L * MOG_D; e += blockDim.x) {
                int l = e / MOG_D, jj = e % MOG_D;
                cs[e] = bf1(dv.krow(b, h, pA[(int64_t)l * n / L])[jj]);
            }
            for (int m = tid; m < n; m += blockDim.x) sa[m] = -1;
        }
        int steps2 = 0;
        for (int t = 0; t < dv.T2 && n > 0; ++t) {
            if (tid == 0) s_changed = 0;
            __syncthreads();
            if (tr.l2c) {  // traced build: the centroids of this step
                float *tc = tr.l2c + (((int64_t)u * dv.c_max + c) * dv.T2 + t) * dv.l_max * MOG_D;
                for (int e = tid; e < L * MOG_D; e += blockDim.x) tc[e] = cs[e];
            }
            const int my = l2_assign([&](int m) { return dv.krow(b, h, pA[m]); }, sa, n, L, cs,
                                     ring, s_cn);
            if (my) atomicAdd(&s_changed, my);
            __syncthreads();
            steps2 = t + 1;
            if (tr.l2a) {  // ... and the assignment it made
                int *ta = tr.l2a + ((int64_t)u * dv.T2 + t) * tr.nm + lo;
                for (int m = tid; m < n; m += blockDim.x) ta[m] = sa[m];
            }
            if (t > 0 && s_changed == 0) break;
            if (t + 1 == dv.T2) break;
            // update: each half of the block takes a run of subclusters; thread j of a
            // half owns dimension j and sums its subclusters' members in position order
            order_members();
            const int l_b = upper ? s_half : 0, l_e = upper ? L : s_half;
            int l = l_b, next = l_b < l_e ? pref[l_b + 1] : n;
            Kahan acc;
            acc.init();
            stream_rows(dv, b, h, permF + lo, pref[l_b], pref[l_e], false,
                        ring + (upper ? L2_RING / 2 : 0), j, MOG_D, 1 + (int)upper,
                        [&](int m0, int k, const uint16_t *sk, const uint16_t *) {
                            for (int r = 0; r < k; ++r) {
                                while (m0 + r >= next) {
                                    if (cnt[l] > 0) cs[l * MOG_D + j] = acc.s / (float)cnt[l];
                                    acc.init();
                                    ++l;
                                    next = pref[l + 1];
                                }
                                acc.add(bf1(sk[r * MOG_D + j]));
                            }
                        });
            if (pref[l_b] < pref[l_e]) cs[l * MOG_D + j] = acc.s / (float)cnt[l];
            __syncthreads();
        }
        if (tr.l2s && tid == 0) tr.l2s[(int64_t)u * dv.c_max + c] = steps2;
        // final order: (subcluster, position), stable
        order_members();
        if (tid < L) so[c * L + tid] = lo + pref[tid];
        if (tid == 0 && c == C - 1) so[C * L] = lo + n;
        __syncthreads();
    }
    // ------ summaries.  Pass 1 (keys and values): thread j < d sums key dimension j,
    // thread d + j value dimension j, per subcluster and over the cluster.  Pass 2 (keys):
    // thread j the subcluster variances, thread d + j the cluster variance.
    const int *pf = permF + lo;
    const int64_t cg = (int64_t)u * dv.c_max + c;
    const int64_t sg0 = (int64_t)u * dv.c_max * dv.l_max + (int64_t)c * L;
    // subcluster l spans [g(l), g(l + 1)) of pf; the end of the last one is this
    // cluster's end (the next entry of the offsets belongs to the next cluster's CTA)
    auto g_of = [&](int l) { return l < L ? so[c * L + l] - lo : n; };
    {
        Kahan s, tot;
        s.init();
        tot.init();
        int l = 0, g_lo = 0, g_hi = g_of(1);
        auto flush = [&]() {
            const int ng = g_hi - g_lo;
            const float mean = ng > 0 ? s.s / (float)ng : 0.f;
            const int64_t sg = sg0 + l;
            if (upper) {
                dv.sub_vbar[sg * MOG_D + j] = mean;
                // bf16 high and low parts, for the decode (fp8 summaries: the e4m3-rounded mean)
                const uint32_t hi = f2bf(dv.fp8s ? e4m3_round(mean) : mean);
                dv.sub_vhl[sg * 2 * MOG_D + j] = (uint16_t)hi;
                dv.sub_vhl[sg * 2 * MOG_D + MOG_D + j] = (uint16_t)f2bf(mean - bf1((uint16_t)hi));
            } else {
                dv.sub_ms[sg * 2 * MOG_D + j] = mean;
                if (dv.sub_ms16) dv.sub_ms16[sg * 2 * MOG_D + j] = (uint16_t)f2bf(mean);
                if (dv.sub_ms8) dv.sub_ms8[sg * 2 * MOG_D + j] = (uint8_t)f2e4m3(mean);
                cs[l * MOG_D + j] = mean;
                if (j == 0) dv.sub_n[sg] = ng;
            }
            s.init();
            ++l;
            g_lo = g_hi;
            g_hi = g_of(l + 1);
        };
        stream_rows(dv, b, h, pf, 0, n, true, ring, tid, L2_THREADS, 0,
                    [&](int m0, int k, const uint16_t *sk, const uint16_t *sv) {
                        const uint16_t *src = upper ? sv : sk;
                        for (int r = 0; r < k; ++r) {
                            while (m0 + r >= g_hi) flush();
                            const float v = bf1(src[r * MOG_D + j]);
                            s.add(v);
                            tot.add(v);
                        }
                    });
        while (l < L) flush();
        const float cmean = n > 0 ? tot.s / (float)n : 0.f;
        if (upper) {
            dv.cl_vbar[cg * MOG_D + j] = cmean;
            const uint32_t hi = f2bf(dv.fp8s ? e4m3_round(cmean) : cmean);
            dv.cl_vhl[cg * 2 * MOG_D + j] = (uint16_t)hi;
            dv.cl_vhl[cg * 2 * MOG_D + MOG_D + j] = (uint16_t)f2bf(cmean - bf1((uint16_t)hi));
        } else {
            dv.cl_ms[cg * 2 * MOG_D + j] = cmean;
            if (dv.cl_ms16) dv.cl_ms16[cg * 2 * MOG_D + j] = (uint16_t)f2bf(cmean);
            if (dv.cl_ms8) dv.cl_ms8[cg * 2 * MOG_D + j] = (uint8_t)f2e4m3(cmean);
            s_cm[j] = cmean;
            if (j == 0) dv.cl_n[cg] = n;
        }
    }
    __syncthreads();
    {
        Kahan q;
        q.init();
        int l = 0, g_lo = 0, g_hi = g_of(1);
        auto flush = [&]() {
            const int ng = g_hi - g_lo;
            if (!upper) {
                const float var = ng > 0 ? q.s / (float)ng : 0.f;
                dv.sub_ms[(sg0 + l) * 2 * MOG_D + MOG_D + j] = var;
                if (dv.sub_ms16) dv.sub_ms16[(sg0 + l) * 2 * MOG_D + MOG_D + j] = (uint16_t)f2bf(var);
                if (dv.sub_ms8) dv.sub_ms8[(sg0 + l) * 2 * MOG_D + MOG_D + j] = (uint8_t)f2e4m3(var);
            }
            q.init();
            ++l;
            g_lo = g_hi;
            g_hi = g_of(l + 1);
        };
        const float cm = s_cm[j];
        stream_rows(dv, b, h, pf, 0, n, false, ring, tid, L2_THREADS, 0,
                    [&](int m0, int k, const uint16_t *sk, const uint16_t *) {
                        for (int r = 0; r < k; ++r) {
                            const float x = bf1(sk[r * MOG_D + j]);
                            if (upper) {
                                const float df = __fsub_rn(x, cm);
                                q.add(__fmul_rn(df, df));
                            } else {
                                while (m0 + r >= g_hi) flush();
                                const float df = __fsub_rn(x, cs[l * MOG_D + j]);
                                q.add(__fmul_rn(df, df));
                            }
                        }
                    });
        if (upper) {
            const float var = n > 0 ? q.s / (float)n : 0.f;
            dv.cl_ms[cg * 2 * MOG_D + MOG_D + j] = var;
            if (dv.cl_ms16) dv.cl_ms16[cg * 2 * MOG_D + MOG_D + j] = (uint16_t)f2bf(var);
            if (dv.cl_ms8) dv.cl_ms8[cg * 2 * MOG_D + MOG_D + j] = (uint8_t)f2e4m3(var);
        } else {
            while (l < L) flush();
        }
    }
}

// ------------------------------------------------------------------------------------
// First-level assignment on the tensor cores (tcgen05, TMA-fed tiles).
//
// The approximate distance of key k to centroid c (up to |k|^2, equal for every c) is
//     a_c = |c|^2 - 2 k.c,   k.c = k.c_hi + k.c_lo   (c split into bf16 high + low parts),
// computed for 128 keys x 128 centroids per MMA group, fp32 accumulate in tensor memory.
// Its error against the exact D(k, c) - |k|^2 is below 2^-14.5 (|k|^2 + |c|^2): the split
// leaves 2^-18 |c_j| per element, the fp32 sums add at most 2^-23 per term over 256
// terms, |c|^2 is an fp32 sum of 128 squares.  The epilogue writes the column (0..63)
// into the low six mantissa bits of each score, which moves it by at most 2^-17 |a_c|
// <= 2^-16 (|k|^2 + |c|^2), below 2^-14 (|k|^2 + |c|^2) in all.  With f = 2^-13 a key keeps its best
// approximate centroid b only when every other centroid j has
//     a_j - f(|k|^2 + |c_j|^2) > a_b + f(|k|^2 + |c_b|^2),
// which makes b the unique exact argmin; every other key goes to the direct fp32 pass
// (and from there, if needed, to the exact fp64 rule).  The kernel checks the sufficient
// form  a_2 - f(|k|^2 + max_j |c_j|^2) > a_b + f(|k|^2 + |c_b|^2)  with a_2 the runner-up,
// so that a key only needs its two best scores.
// ------------------------------------------------------------------------------------
constexpr int TC_M = 128;                       // keys per tile (TMEM lanes)
constexpr int TC_NC = KM_CHUNK;                 // centroids per MMA group (TMEM columns)
constexpr uint32_t TC_A_BYTES = TC_M * 256;     // 128 keys x 128 bf16
constexpr uint32_t TC_B_HALF = TC_NC * 128;     // TC_NC rows x 64 bf16 (one 128-byte swizzle column)
constexpr uint32_t TC_B_BYTES = 4 * TC_B_HALF;  // {high, low} x {k 0-63, k 64-127}
constexpr uint32_t TC_CN_BYTES = MAX_C * 4;     // |c|^2 of every centroid
constexpr size_t TC_SMEM = 1024 + 2 * TC_A_BYTES + 2 * TC_B_BYTES + TC_CN_BYTES;
constexpr int TC_EPI = 8;                       // epilogue warps: 4 lane quarters x 2 column halves
constexpr int TC_THREADS = (TC_EPI + 1) * 32;   // + 1 producer warp
constexpr float TC_BIG = 1e37f;                 // above every score; finite, so packable

__host__ __device__ inline int tc_chunks(int k) { return (k + TC_NC - 1) / TC_NC; }

// Centroid images for the tensor-core pass: bf16 high and low parts in the 128-byte
// swizzle layout (16-byte chunk q of row r at position q ^ (r & 7)), and |c|^2 (fp32,
// +inf for padding).  Block: 8 centroids x 16 chunks of 8 dimensions.
__global__ void __launch_bounds__(128) k_cent_prep(AssignJob jb) {
    const int u = blockIdx.y;
    const int *chg = jb.changed + (int64_t)u * jb.T;
    if (jb.t >= 2 && converged_by(chg, jb.t - 1)) return;
    const int k = job_unit(jb, u).k;
    const int c = blockIdx.x * 8 + (threadIdx.x >> 4), q = threadIdx.x & 15;
    if (c >= tc_chunks(k) * TC_NC) return;
    float v[8];
    const bool real = c < k;
    const float *cp = jb.cent + u * jb.cent_ustride + (int64_t)c * MOG_D + q * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = real ? cp[i] : 0.f;
    uint32_t hi[4], lo[4];
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t h0 = f2bf(v[2 * i]), h1 = f2bf(v[2 * i + 1]);
        hi[i] = h0 | (h1 << 16);
        lo[i] = f2bf(v[2 * i] - bf1((uint16_t)h0)) | (f2bf(v[2 * i + 1] - bf1((uint16_t)h1)) << 16);
        sq = __fmaf_rn(v[2 * i], v[2 * i], sq);
        sq = __fmaf_rn(v[2 * i + 1], v[2 * i + 1], sq);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    const int ch = c / TC_NC, r = c % TC_NC, half = q >> 3, pos = (q & 7) ^ (r & 7);
    uint16_t *img = jb.cimg + u * jb.cimg_ustride + (int64_t)ch * (TC_B_BYTES / 2);
    *reinterpret_cast<uint4 *>(img + (0 * 2 + half) * (TC_B_HALF / 2) + r * 64 + pos * 8) =
        make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4 *>(img + (1 * 2 + half) * (TC_B_HALF / 2) + r * 64 + pos * 8) =
        make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (q == 0) jb.cnorm[u * jb.cn_ustride + c] = real ? sq : INFINITY;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One CTA: tiles [tile0, tile0 + ntl) of one unit (128 keys each) against all centroids,
// TC_NC at a time, in a pipeline over (tile, group) steps.  Warp 4 (one lane) is the
// producer: TMA copies of the keys, bulk copies of the centroid images, the MMAs into one
// of two tensor-memory accumulators.  Warps 0-3 are the epilogue: thread r reads its key's
// row of scores, keeps the best centroid and the runner-up bounds, and decides the key.
// Two key buffers, two centroid buffers and two accumulators let the copies, the MMAs
// and the epilogue of neighbouring steps overlap.
__global__ void __launch_bounds__(TC_THREADS, 1) k_assign_tc(AssignJob jb, const __grid_constant__ CUtensorMap kmap,
                                                             int tiles_per_cta) {
    extern __shared__ uint8_t tc_raw[];
    // barriers: a_full[2], a_free[2], a_kn[2], b_full[2], b_free[2], acc_full[2], acc_free[2], cn
    __shared__ __align__(8) uint64_t s_bar[15];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    const int u = blockIdx.y;
    const int *chg = jb.changed + (int64_t)u * jb.T;
    if (jb.t >= 2 && converged_by(chg, jb.t - 1)) return;
    const JobUnit ju = job_unit(jb, u);
    const int n = ju.n, k = ju.k;
    const int ntile = (n + TC_M - 1) / TC_M;
    const int tile0 = blockIdx.x * tiles_per_cta;
    const int ntl = min(tiles_per_cta, ntile - tile0);
    if (ntl <= 0 || k <= 0) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t raw = smem_u32(tc_raw);
    const uint32_t sA = (raw + 1023u) & ~1023u, sB = sA + 2 * TC_A_BYTES, sC = sB + 2 * TC_B_BYTES;
    const float *scn = reinterpret_cast<const float *>(tc_raw + (sC - raw));
    auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
    enum { A_FULL = 0, A_FREE = 2, A_KN = 4, B_FULL = 6, B_FREE = 8, ACC_FULL = 10, ACC_FREE = 12, CN = 14 };
    int cb = 0, ch_ = 0, crow = 0;
    if (jb.unit_info) {
        const int *ui = jb.unit_info + u * UI_STRIDE;
        cb = ui[UI_B];
        ch_ = u % jb.h_kv;
        crow = ui[UI_S];
    }
    const int nch = tc_chunks(k);
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(A_FULL + i), 1);
            mbar_init(bar(A_FREE + i), 1);
            mbar_init(bar(A_KN + i), 4);
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_FREE + i), 1);
            mbar_init(bar(ACC_FULL + i), 1);
            mbar_init(bar(ACC_FREE + i), TC_EPI);
        }
        mbar_init(bar(CN), 1);
        fence_barrier_init();
        s_fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), 2 * TC_NC);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int total = ntl * nch;

    if (warp == TC_EPI) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            const uint16_t *img = jb.cimg + u * jb.cimg_ustride;
            bool ok = true;
            mbar_expect_tx(bar(CN), (uint32_t)nch * TC_NC * 4);
            bulk_load(sC, jb.cnorm + u * jb.cn_ustride, (uint32_t)nch * TC_NC * 4, bar(CN));
            auto load_step = [&](int it) {
                const int tl = it / nch, c = it - tl * nch;
                if (c == 0) {
                    const int a = tl & 1, na = tl >> 1;
                    if (na >= 1)
                        ok = ok && mbar_wait(bar(A_FREE + a), (na - 1) & 1) && mbar_wait(bar(A_KN + a), (na - 1) & 1);
                    if (!ok) return;
                    fence_proxy_async();
                    mbar_expect_tx(bar(A_FULL + a), TC_A_BYTES);
                    const int r0 = crow + (tile0 + tl) * TC_M;
                    tma_load_4d(sA + a * TC_A_BYTES, &kmap, 0, r0, ch_, cb, bar(A_FULL + a));
                    tma_load_4d(sA + a * TC_A_BYTES + TC_A_BYTES / 2, &kmap, 64, r0, ch_, cb, bar(A_FULL + a));
                }
                const int b = it & 1, nb = it >> 1;
                if (nb >= 1) ok = ok && mbar_wait(bar(B_FREE + b), (nb - 1) & 1);
                if (!ok) return;
                const int nreal = min(TC_NC, k - c * TC_NC), ncp = (nreal + 15) & ~15;
                const uint32_t bytes = (uint32_t)ncp * 128;
                fence_proxy_async();
                mbar_expect_tx(bar(B_FULL + b), 4 * bytes);
                const uint16_t *cimg = img + (int64_t)c * (TC_B_BYTES / 2);
                for (int part = 0; part < 4; ++part)
                    bulk_load(sB + b * TC_B_BYTES + part * TC_B_HALF, cimg + part * (TC_B_HALF / 2), bytes,
                              bar(B_FULL + b));
            };
            load_step(0);
            for (int it = 0; it < total && ok; ++it) {
                if (it + 1 < total) load_step(it + 1);
                const int tl = it / nch, c = it - tl * nch;
                const int a = tl & 1, na = tl >> 1, b = it & 1, nb = it >> 1, acc = it & 1, nacc = it >> 1;
                ok = ok && mbar_wait(bar(B_FULL + b), nb & 1);
                if (c == 0) ok = ok && mbar_wait(bar(A_FULL + a), na & 1);
                if (nacc >= 1) ok = ok && mbar_wait(bar(ACC_FREE + acc), (nacc - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const int nreal = min(TC_NC, k - c * TC_NC), ncp = (nreal + 15) & ~15;
                const uint32_t idesc = idesc_bf16_f32(TC_M, ncp);
                const uint32_t d = tmem + (uint32_t)(acc * TC_NC);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t aoff = a * TC_A_BYTES + (ks >> 2) * (TC_A_BYTES / 2) + (ks & 3) * 32;
                        const uint32_t boff = b * TC_B_BYTES + (part * 2 + (ks >> 2)) * TC_B_HALF + (ks & 3) * 32;
                        tc_mma(d, smem_desc_sw128(sA + aoff), smem_desc_sw128(sB + boff), idesc, (part | ks) != 0);
                    }
                tc_commit(bar(B_FREE + b));
                tc_commit(bar(ACC_FULL + acc));
                if (c == nch - 1) tc_commit(bar(A_FREE + a));
            }
            if (!ok) atomicExch(&s_fail, 1);
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        // warp w: TMEM lanes (keys) 32*(w%4) .. +31, columns of its half w/4 of each group
        __shared__ float s_xb[TC_M][2];
        __shared__ int s_xi[TC_M];
        __shared__ float s_cmax[TC_EPI];
        const int qw = warp & 3, hw = warp >> 2, r = qw * 32 + lane;
        bool ok = mbar_wait(bar(CN), 0);
        float cmax = 0.f;  // max |c|^2 over the unit's centroids
        if (ok) {
            for (int c = tid; c < k; c += TC_EPI * 32) cmax = fmaxf(cmax, scn[c]);
            cmax = warp_max(cmax);
            if (lane == 0) s_cmax[warp] = cmax;
        }
        named_sync(1, TC_EPI * 32);
        cmax = 0.f;
        for (int w = 0; w < TC_EPI; ++w) cmax = fmaxf(cmax, s_cmax[w]);
        int chg_w = 0;
        // every epilogue warp runs every tile's two named barriers, also after a failed wait
        // (it then skips the work), so that no warp is left waiting at one
        for (int tl = 0; tl < ntl; ++tl) {
            const int a = tl & 1, na = tl >> 1;
            const int row = (tile0 + tl) * TC_M + r;
            float kn = 0.f;
            float b1 = TC_BIG, b2 = TC_BIG;  // the two smallest scores of this key (half)
            int i1 = 0;                      // a valid index even if no score is finite
            for (int c = 0; c < nch; ++c) {
                const int it = tl * nch + c, acc = it & 1, nacc = it >> 1;
                ok = ok && mbar_wait(bar(ACC_FULL + acc), nacc & 1);
                if (c == 0 && hw == 0) ok = ok && mbar_wait(bar(A_FULL + a), na & 1);
                if (!ok) continue;
                tc_fence_after();
                if (c == 0 && hw == 0) {  // this key's |k|^2 from the swizzled tile, then release it
                    const uint8_t *ta = tc_raw + (sA + a * TC_A_BYTES - raw);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(
                            ta + (q >> 3) * (TC_A_BYTES / 2) + r * 128 + (((q & 7) ^ (r & 7)) << 4));
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            kn = __fmaf_rn(bf_lo(ws[i]), bf_lo(ws[i]), kn);
                            kn = __fmaf_rn(bf_hi(ws[i]), bf_hi(ws[i]), kn);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(A_KN + a));
                }
                // this warp's columns h0 .. h0 + hcnt - 1 of the group; each score carries its
                // column (0..63) in the low six mantissa bits, so that plain min / max
                // keep the two smallest and the argmin; eight chains for ILP
                const int h0 = hw * (TC_NC / 2);
                const int hcnt = min(TC_NC / 2, min(TC_NC, k - c * TC_NC) - h0);
                float pb1[8], pb2[8];
#pragma unroll
                for (int z = 0; z < 8; ++z) pb1[z] = pb2[z] = TC_BIG;
                // both 32-column blocks are loaded before one wait
                uint32_t vr[2][32];
                const uint32_t tl0 = tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(acc * TC_NC + h0);
                if (hcnt > 0) tmem_ld32_nowait(tl0, vr[0]);
                if (hcnt > 32) tmem_ld32_nowait(tl0 + 32, vr[1]);
                tmem_wait_ld();
                // Scores are folded two at a time: with lo <= hi the pair's own order, the
                // two smallest of {b1 <= b2, lo, hi} are min(b1, lo) and
                // min(b2, hi, max(b1, lo)), the latter one three-input min.
                auto fold_block = [&](const uint32_t (&v)[32], int blk, bool full) {
                    const float4 *cn4 = reinterpret_cast<const float4 *>(scn + c * TC_NC + h0 + blk * 32);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 cn = cn4[j4];
                        const float cq[4] = {cn.x, cn.y, cn.z, cn.w};
#pragma unroll
                        for (int e = 0; e < 4; e += 2) {
                            const int j = 4 * j4 + e, z = (j >> 1) & 7;
                            const float a0 = __fmaf_rn(-2.f, __uint_as_float(v[j]), cq[e]);
                            const float a1 = __fmaf_rn(-2.f, __uint_as_float(v[j + 1]), cq[e + 1]);
                            float p0 = __uint_as_float((__float_as_uint(a0) & ~63u) | (uint32_t)(blk * 32 + j));
                            float p1 = __uint_as_float((__float_as_uint(a1) & ~63u) | (uint32_t)(blk * 32 + j + 1));
                            if (!full) {
                                if (blk * 32 + j >= hcnt) p0 = TC_BIG;
                                if (blk * 32 + j + 1 >= hcnt) p1 = TC_BIG;
                            }
                            const float lo = fminf(p0, p1), hi = fmaxf(p0, p1);
                            pb2[z] = fmin3(pb2[z], hi, fmaxf(pb1[z], lo));
                            pb1[z] = fminf(pb1[z], lo);
                        }
                    }
                };
                if (hcnt >= 64) {
                    fold_block(vr[0], 0, true);
                    fold_block(vr[1], 1, true);
                } else {
                    if (hcnt > 0) fold_block(vr[0], 0, hcnt >= 32);
                    if (hcnt > 32) fold_block(vr[1], 1, false);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ACC_FREE + acc));
#pragma unroll
                for (int z = 1; z < 8; ++z) {
                    pb2[0] = fminf(fmaxf(pb1[0], pb1[z]), fminf(pb2[0], pb2[z]));
                    pb1[0] = fminf(pb1[0], pb1[z]);
                }
                if (pb1[0] < TC_BIG) {  // fold the group into the key's running pair
                    const int ci = c * TC_NC + h0 + (int)(__float_as_uint(pb1[0]) & 63u);
                    b2 = fminf(fmaxf(b1, pb1[0]), fminf(b2, pb2[0]));
                    if (pb1[0] < b1) {
                        b1 = pb1[0];
                        i1 = ci;
                    }
                }
            }
            // the two column halves of each key: the two smallest scores and the index of
            // the smallest (scores of different columns differ in their low bits)
            if (hw == 1) {
                s_xb[r][0] = b1;
                s_xb[r][1] = b2;
                s_xi[r] = i1;
            }
            named_sync(1, TC_EPI * 32);
            if (hw == 0 && ok) {
                const float ob1 = s_xb[r][0], ob2 = s_xb[r][1];
                const int oi1 = s_xi[r];
                const float nb2 = fminf(fmaxf(b1, ob1), fminf(b2, ob2));
                if (ob1 < b1) {
                    b1 = ob1;
                    i1 = oi1;
                }
                b2 = nb2;
                const bool certain =
                    (k == 1) || (b2 - TC_F * (kn + cmax) > b1 + TC_F * (kn + scn[i1]));
                const bool valid = row < n;
                int changed = 0;
                if (valid && certain) {
                    int *dst = jb.assign + u * jb.assign_ustride + row;
                    if (*dst != i1) {
                        *dst = i1;
                        changed = 1;
                    }
                }
                chg_w += changed;
                const uint32_t unc = __ballot_sync(0xffffffffu, valid && !certain);
                if (unc) {
                    int base = 0;
                    if (lane == 0) base = atomicAdd(jb.rc_cnt + u * jb.T + jb.t, __popc(unc));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    if (valid && !certain)
                        jb.rc_list[u * jb.fb_ustride + base + __popc(unc & lanemask_lt())] = row;
                }
            }
            named_sync(1, TC_EPI * 32);
        }
        chg_w = __reduce_add_sync(0xffffffffu, chg_w);
        if (lane == 0 && chg_w) atomicAdd(jb.changed + u * jb.T + jb.t, chg_w);
        if (!ok) atomicExch(&s_fail, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (s_fail && tid == 0) flag_error(jb.status, ST_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, 2 * TC_NC);
}

// ------------------------------------------------------------------------------------
// launchers
// ------------------------------------------------------------------------------------
static AssignJob build_job(const Dev &dv, int t) {
    AssignJob jb;
    jb.K = dv.K;
    jb.sb = dv.sb;
    jb.sh = dv.sh;
    jb.sn = dv.sn;
    jb.bt = dv.bt;
    jb.pshift = dv.pshift;
    jb.pps = dv.pps;
    jb.h_kv = dv.h_kv;
    jb.unit_info = dv.unit_info;
    jb.n_single = 0;
    jb.k_single = 0;
    jb.cent = dv.cent;
    jb.cent_ustride = (int64_t)dv.c_max * MOG_D;
    jb.assign = dv.l1_assign;
    jb.assign_ustride = dv.n_cap;
    jb.changed = dv.changed;
    jb.fb_list = dv.fb_list;
    jb.fb_ustride = dv.n_cap;
    jb.fb_cnt = dv.fb_cnt;
    jb.t = t;
    jb.T = dv.T1;
    jb.rows = nullptr;
    jb.rows_ustride = 0;
    jb.rows_cnt = nullptr;
    jb.cimg = dv.cimg;
    jb.cimg_ustride = dv.cimg_ustride;
    jb.cnorm = dv.cnorm;
    jb.cn_ustride = dv.cn_ustride;
    jb.rc_list = dv.rc_list;
    jb.rc_cnt = dv.rc_cnt;
    jb.status = dv.status;
    return jb;
}

static cudaError_t set_smem(const void *fn, size_t bytes) { return ensure_smem(fn, bytes); }

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// Tensor map of bf16 keys [b][h][row][128] (element strides sn, sh, sb), boxes of 64
// dimensions x TC_M rows in the 128-byte swizzle.  False if TMA cannot describe it.
static bool key_map(CUtensorMap *map, const uint16_t *base, int64_t rows, int64_t h, int64_t b,
                    int64_t sn, int64_t sh, int64_t sb) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)MOG_D, (cuuint64_t)rows, (cuuint64_t)h, (cuuint64_t)b};
    const cuuint64_t strides[3] = {(cuuint64_t)sn * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
    for (int i = 0; i < 3; ++i)
        if (strides[i] == 0 || (strides[i] & 15) || strides[i] >= (1ull << 40)) return false;
    const cuuint32_t box[4] = {64, (cuuint32_t)TC_M, 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One assignment step: the tensor-core pass over every row (when the keys have a tensor
// map), the direct fp32 pass over the rows it could not decide (else over every row),
// then the exact fp64 rule for whatever the direct pass could not certify.
static cudaError_t assign_step(const AssignJob &jb, const CUtensorMap *kmap, int units, int n_max,
                               int k_max, cudaStream_t s) {
    cudaError_t e;
    if ((e = set_smem((const void *)k_assign_l1, AS_SMEM)) != cudaSuccess) return e;
    if (kmap) {
        if ((e = set_smem((const void *)k_assign_tc, TC_SMEM)) != cudaSuccess) return e;
        k_cent_prep<<<dim3(tc_chunks(k_max) * (TC_NC / 8), units), 128, 0, s>>>(jb);
        // persistent CTAs: about one per SM, each over a run of its unit's tiles
        const int ntile = (int)ceil_div64(n_max, TC_M);
        const int per_unit = std::max(1, num_sms() / std::max(units, 1));
        const int tpc = (int)ceil_div64(ntile, per_unit);
        k_assign_tc<<<dim3((int)ceil_div64(ntile, tpc), units), TC_THREADS, TC_SMEM, s>>>(jb, *kmap, tpc);
        AssignJob jl = jb;
        jl.rows = jb.rc_list;
        jl.rows_ustride = jb.fb_ustride;
        jl.rows_cnt = jb.rc_cnt;
        const int gx = std::max(1, std::min((int)ceil_div64(n_max, AS_ROWS), 2 * num_sms() / std::max(units, 1)));
        k_assign_l1<<<dim3(gx, units), AS_THREADS, AS_SMEM, s>>>(jl);
    } else {
        AssignJob jf = jb;
        jf.rows = nullptr;
        k_assign_l1<<<dim3((int)ceil_div64(n_max, AS_ROWS), units), AS_THREADS, AS_SMEM, s>>>(jf);
    }
    k_assign_fallback<<<dim3(FB_CTAS, units), FB_THREADS, 0, s>>>(jb);
    return cudaGetLastError();
}

static size_t l2_smem() { return MOG_MAX_L * MOG_D * sizeof(float) + L2_RING; }

cudaError_t launch_build(const Dev &dv, const Plan &pl, cudaStream_t s, const TraceDev &tr) {
    cudaError_t e;
    if ((e = set_smem((const void *)k_assign_l1, AS_SMEM)) != cudaSuccess) return e;
    if ((e = set_smem((const void *)k_l2_stats, l2_smem())) != cudaSuccess) return e;
    if ((e = set_smem((const void *)k_sort_hist, pl.c_max * sizeof(int))) != cudaSuccess) return e;
    if ((e = set_smem((const void *)k_sort_scatter, pl.c_max * sizeof(int))) != cudaSuccess) return e;
    const int U = pl.units;
    if (pl.n_mid_max > 0) {
        if (dv.kpp) {
            for (int r = 0; r < pl.c_max && e == cudaSuccess; ++r) {
                e = launch_pdl_km(k_pp_pick, dim3(U), dim3(PP_THREADS), 0, s, dv, r);
                if (e == cudaSuccess && r + 1 < pl.c_max)
                    e = launch_pdl_km(k_pp_update, dim3(pl.pp_nblk, U), dim3(PP_THREADS), 0, s, dv, r);
            }
            if (e != cudaSuccess) return e;
        }
        k_l1_init<<<dim3(pl.c_max, U), 128, 0, s>>>(dv);
        CUtensorMap kmap;
        // TMA tiles need contiguous rows: a paged cache takes the direct fp32 pass
        const bool tma = !dv.bt && key_map(&kmap, dv.K, pl.n_cap, dv.h_kv, pl.batch, dv.sn, dv.sh, dv.sb);
        for (int t = 0; t < pl.T1; ++t) {
            AssignJob jb = build_job(dv, t);
            if (tr.l1c &&  // traced build: the centroids this step assigns to
                (e = cudaMemcpy2DAsync(tr.l1c + (int64_t)t * pl.c_max * MOG_D,
                                       4 * (size_t)pl.T1 * pl.c_max * MOG_D, dv.cent,
                                       4 * (size_t)pl.c_max * MOG_D, 4 * (size_t)pl.c_max * MOG_D, U,
                                       cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
                return e;
            if ((e = assign_step(jb, tma ? &kmap : nullptr, U, pl.n_mid_max, pl.c_max, s)) != cudaSuccess)
                return e;
            if (tr.l1a &&  // ... and the assignment it made
                (e = cudaMemcpy2DAsync(tr.l1a + (int64_t)t * tr.nm, 4 * (size_t)pl.T1 * tr.nm,
                                       dv.l1_assign, 4 * (size_t)pl.n_cap, 4 * (size_t)pl.n_mid_max, U,
                                       cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
                return e;
            k_sort_hist<<<dim3(pl.nchunks, U), 256, pl.c_max * sizeof(int), s>>>(dv, t);
            k_sort_colscan<<<dim3((int)ceil_div64(pl.c_max, 128), U), 128, 0, s>>>(dv, t);
            k_sort_base<<<U, 1024, 0, s>>>(dv, t);
            k_sort_scatter<<<dim3(pl.nchunks, U), 32, pl.c_max * sizeof(int), s>>>(dv, t);
            if (t + 1 < pl.T1) k_l1_update<<<dim3(pl.c_max, U), 256, 0, s>>>(dv, t);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    k_l2_stats<<<dim3(pl.c_max, U), L2_THREADS, l2_smem(), s>>>(dv, 1, tr);
    return cudaGetLastError();
}

cudaError_t launch_stats_only(const Dev &dv, const Plan &pl, cudaStream_t s) {
    cudaError_t e;
    if ((e = set_smem((const void *)k_l2_stats, l2_smem())) != cudaSuccess) return e;
    k_l2_stats<<<dim3(pl.c_max, pl.units), L2_THREADS, l2_smem(), s>>>(dv, 0, TraceDev{});
    return cudaGetLastError();
}

cudaError_t launch_assign_l1(const uint16_t *x, int64_t ld, int n, const float *cent, int k,
                             int32_t *assign, const KmScratch &ks, cudaStream_t s) {
    AssignJob jb;
    jb.K = x;
    jb.sb = jb.sh = 0;
    jb.sn = ld;
    jb.bt = nullptr;
    jb.pshift = jb.pps = 0;
    jb.h_kv = 1;
    jb.unit_info = nullptr;
    jb.n_single = n;
    jb.k_single = k;
    jb.cent = cent;
    jb.cent_ustride = 0;
    jb.assign = assign;
    jb.assign_ustride = 0;
    jb.changed = ks.changed;
    jb.fb_list = ks.fb_list;
    jb.fb_ustride = 0;
    jb.fb_cnt = ks.fb_cnt;
    jb.t = 0;
    jb.T = 1;
    jb.rows = nullptr;
    jb.rows_ustride = 0;
    jb.rows_cnt = nullptr;
    jb.cimg = ks.cimg;
    jb.cimg_ustride = 0;
    jb.cnorm = ks.cnorm;
    jb.cn_ustride = 0;
    jb.rc_list = ks.rc_list;
    jb.rc_cnt = ks.rc_cnt;
    jb.status = ks.status;
    if (n <= 0) return cudaSuccess;
    CUtensorMap kmap;
    const bool tma = key_map(&kmap, x, n, 1, 1, ld, ld * n, ld * n);
    return assign_step(jb, tma ? &kmap : nullptr, 1, n, k, s);
}

// Self-check of the bounded wait the tensor-core pass uses: thread 0 initialises an
// mbarrier that expects one arrival and waits on it with `limit` polls.  With arrive != 0
// thread 1 arrives first and the wait completes; without, nothing completes the phase and
// the wait gives up, records ST_TIMEOUT in status[0] and the kernel returns.
__global__ void k_wait_check(int limit, int arrive, int *status) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 1)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(b, 0, limit)) flag_error(status, ST_TIMEOUT);
}

cudaError_t launch_wait_check(int limit, int arrive, int *status, cudaStream_t s) {
    k_wait_check<<<1, 32, 0, s>>>(limit, arrive, status);
    return cudaGetLastError();
}

cudaError_t launch_assign_segments(const uint16_t *x, int64_t ld, const int32_t *rows,
                                   const int32_t *seg_off, int n_seg, const float *cent, int k,
                                   int32_t *assign, cudaStream_t s) {
    SegJob jb{x, ld, rows, seg_off, cent, k, assign};
    cudaError_t e;
    if (n_seg > 0) {
        if ((e = set_smem((const void *)k_assign_segments, l2_smem())) != cudaSuccess) return e;
        k_assign_segments<<<n_seg, L2_THREADS, l2_smem(), s>>>(jb);
    }
    return cudaGetLastError();
}

}  // namespace mog
