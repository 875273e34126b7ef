// fmap.cu -- the feature-map residual, a second estimator of the mass the selection leaves
// out (the retrieval-completion page on newx.sg, Abstract and AI Summary: a fixed-size
// feature-map summary of the mid region, built at prefill, estimates the numerator and
// denominator of the keys not retrieved; the exact and estimated parts are added
// unnormalised and normalised once).
//
// The feature map is the positive random-feature map of the softmax kernel,
//     phi_i(x) = m^(-1/2) exp(w_i.x - |x|^2/2),  i < m = MOG_FM_FEATURES,  w_i ~ N(0, I),
// applied to q~ = sqrt(tau) q and k~ = sqrt(tau) k, so that phi(q~).phi(k~) estimates
// exp(tau q.k) without bias.  The build keeps, for every subcluster s and feature i,
//     Z[s][i][j] = sum_{k in s} exp(w_i.k~ - |k~|^2/2 - M_i) v_kj   (j < d),
//     Z[s][i][d] = sum_{k in s} exp(w_i.k~ - |k~|^2/2 - M_i),
// with M_i = |w_i|^2/2 - FM_SHIFT: since w.x - |x|^2/2 <= |w|^2/2, every term is at most
// exp(FM_SHIFT), and the typical term stays far above the fp32 underflow.  T, the sum over
// all subclusters, summarises the whole mid region.  At decode, head g's estimate of the
// keys it does not attend exactly is
//     sum_i exp(a_i) (T[i] - sum_{s chosen by g} Z[s][i]),
//     a_i = w_i.q~ - |q~|^2/2 + M_i - ln m,
// one more (max, sum, vector) state for the merge.  Reading the chosen subclusters' sums
// replaces computing phi of every retrieved row inside the rows kernel.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace mog {

constexpr float FM_SHIFT = 40.f;
constexpr int FM_THREADS = 256, FM_CHUNK = 16;  // build: key rows per chunk
constexpr int FM_PF = FM_CHUNK * FM_M / FM_THREADS;  // build: projections per thread

// M_i of every feature (fp32, index order), once per mog_feature_map
__global__ void k_fm_prep(Dev dv) {
    const int i = threadIdx.x;
    if (i >= FM_M) return;
    float s = 0.f;
    for (int j = 0; j < MOG_D; ++j) s = fmaf(dv.fm_omega[i * MOG_D + j], dv.fm_omega[i * MOG_D + j], s);
    dv.fm_mi[i] = 0.5f * s - FM_SHIFT;
}

// One CTA per (cluster, unit): every subcluster's Z, then the cluster's sum of them.
// Thread t owns feature i = t / 8 and the value dimensions j = t % 8 + 8 q (q < 16).
__global__ void __launch_bounds__(FM_THREADS) k_fm_stats(Dev dv) {
    const int c = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], L = ui[UI_L];
    if (c >= C) return;
    __shared__ float s_om[FM_M][MOG_D + 1];  // padded rows: a warp's projections read 16 features at once
    __shared__ float s_k[FM_CHUNK][MOG_D + 1];
    __shared__ float s_v[FM_CHUNK][MOG_D];
    __shared__ float s_phi[FM_CHUNK][FM_M + 1];
    __shared__ float s_kk[FM_CHUNK];
    __shared__ float s_mi[FM_M];
    for (int e = tid; e < FM_M * MOG_D; e += FM_THREADS) s_om[e / MOG_D][e % MOG_D] = dv.fm_omega[e];
    if (tid < FM_M) s_mi[tid] = dv.fm_mi[tid];
    const float st = sqrtf(dv.tau);
    const int b = ui[UI_B], h = u % dv.h_kv;
    const int *so = dv.sub_off + (int64_t)u * dv.sub_off_stride;
    const int *pm = dv.perm + (int64_t)u * dv.n_cap;
    const int fi = tid >> 3, fj = tid & 7;
    float cacc[MOG_D / 8], cden = 0.f;  // the cluster's sums
#pragma unroll
    for (int q = 0; q < MOG_D / 8; ++q) cacc[q] = 0.f;
    for (int l = 0; l < L; ++l) {
        const int g = c * L + l, lo = so[g], hi = so[g + 1];
        float acc[MOG_D / 8], den = 0.f;
#pragma unroll
        for (int q = 0; q < MOG_D / 8; ++q) acc[q] = 0.f;
        for (int r0 = lo; r0 < hi; r0 += FM_CHUNK) {
            const int nr = min(FM_CHUNK, hi - r0);
            __syncthreads();  // the previous chunk is consumed (and s_om is written)
            for (int e = tid; e < nr * 16; e += FM_THREADS) {
                const int r = e >> 4, ch = e & 15;
                const int pos = pm[r0 + r];
                const uint4 kw = *reinterpret_cast<const uint4 *>(dv.krow(b, h, pos) + ch * 8);
                const uint4 vw = *reinterpret_cast<const uint4 *>(dv.vrow(b, h, pos) + ch * 8);
                const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w}, vv[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    s_k[r][ch * 8 + 2 * w] = st * bf_lo(kk[w]);
                    s_k[r][ch * 8 + 2 * w + 1] = st * bf_hi(kk[w]);
                    s_v[r][ch * 8 + 2 * w] = bf_lo(vv[w]);
                    s_v[r][ch * 8 + 2 * w + 1] = bf_hi(vv[w]);
                }
            }
            __syncthreads();
            if (tid < nr) {
                float s = 0.f;
                for (int j = 0; j < MOG_D; ++j) s = fmaf(s_k[tid][j], s_k[tid][j], s);
                s_kk[tid] = s;
            }
            // projections: thread t takes row t / (FM_M / FM_PF) and FM_PF features
            const int pr = tid / (FM_M / FM_PF), pf = (tid % (FM_M / FM_PF)) * FM_PF;
            float p[FM_PF];
#pragma unroll
            for (int f = 0; f < FM_PF; ++f) p[f] = 0.f;
            if (pr < nr)
                for (int j = 0; j < MOG_D; ++j) {
                    const float x = s_k[pr][j];
#pragma unroll
                    for (int f = 0; f < FM_PF; ++f) p[f] = fmaf(s_om[pf + f][j], x, p[f]);
                }
            __syncthreads();  // s_kk
            if (pr < nr)
#pragma unroll
                for (int f = 0; f < FM_PF; ++f) s_phi[pr][pf + f] = __expf(p[f] - 0.5f * s_kk[pr] - s_mi[pf + f]);
            __syncthreads();
            for (int r = 0; r < nr; ++r) {
                const float ph = s_phi[r][fi];
#pragma unroll
                for (int q = 0; q < MOG_D / 8; ++q) acc[q] = fmaf(ph, s_v[r][fj + 8 * q], acc[q]);
                den += ph;
            }
        }
        float *z = dv.fm_z + (((int64_t)u * dv.c_max * dv.l_max + g) * FM_M + fi) * FM_W;
#pragma unroll
        for (int q = 0; q < MOG_D / 8; ++q) {
            z[fj + 8 * q] = acc[q];
            cacc[q] += acc[q];
        }
        if (fj == 0) z[MOG_D] = den;
        if (fj < FM_W - MOG_D - 1) z[MOG_D + 1 + fj] = 0.f;  // the row's padding
        cden += den;
    }
    float *zc = dv.fm_zc + (((int64_t)u * dv.c_max + c) * FM_M + fi) * FM_W;
#pragma unroll
    for (int q = 0; q < MOG_D / 8; ++q) zc[fj + 8 * q] = cacc[q];
    if (fj == 0) zc[MOG_D] = cden;
    if (fj < FM_W - MOG_D - 1) zc[MOG_D + 1 + fj] = 0.f;
}

// T[u] = the sum of the unit's cluster sums, in cluster order: one thread per entry.
__global__ void k_fm_total(Dev dv) {
    const int u = blockIdx.y, o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= FM_M * FM_W) return;
    const int C = dv.unit_info[u * UI_STRIDE + UI_C];
    const float *zc = dv.fm_zc + (int64_t)u * dv.c_max * FM_M * FM_W + o;
    float s = 0.f;
    if (o % FM_W <= MOG_D)
        for (int c = 0; c < C; ++c) s += zc[(int64_t)c * FM_M * FM_W];
    dv.fm_t[(int64_t)u * FM_M * FM_W + o] = s;
}

// Decode: CTA (k, g, u) contracts with head g's feature weights exp(a_i - max a) either T
// (k = FM_NCH) or the sums of head g's chosen subclusters e with e = k (mod FM_NCH), and
// writes the (d + 1)-vector; the merge takes T's vector minus the others.
__global__ void __launch_bounds__(FM_THREADS) k_fm_resid(Dev dv, const uint16_t *q, int SW) {
    const int k = blockIdx.x, g = blockIdx.y, u = blockIdx.z, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    __shared__ float s_q[MOG_D], s_a[FM_M], s_acc[FM_M * FM_W];
    __shared__ float s_qq;
    pdl_wait();  // the selection of this step
    pdl_trigger();
    const int G = dv.G;
    const float st = sqrtf(dv.tau);
    const uint16_t *qg = q + ((int64_t)u * G + g) * MOG_D;
    if (tid < MOG_D) s_q[tid] = st * bf1(qg[tid]);
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int j = 0; j < MOG_D; ++j) s = fmaf(s_q[j], s_q[j], s);
        s_qq = s;
    }
    __syncthreads();
    // a_i: warp w takes features FM_M / 8 at a time (4w .. 4w + 3)
    for (int f = 0; f < FM_M / (FM_THREADS / 32); ++f) {
        const int i = warp * (FM_M / (FM_THREADS / 32)) + f;
        float s = 0.f;
        for (int j = lane; j < MOG_D; j += 32) s = fmaf(dv.fm_omega[i * MOG_D + j], s_q[j], s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) s_a[i] = s - 0.5f * s_qq + dv.fm_mi[i] - logf((float)FM_M);
    }
    __syncthreads();
    float amax = -INFINITY;
    for (int i = 0; i < FM_M; ++i) amax = fmaxf(amax, s_a[i]);
    // the chunk's sum of Z (or T)
    constexpr int PER = (FM_M * FM_W + FM_THREADS - 1) / FM_THREADS;
    float acc[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) acc[p] = 0.f;
    const int L = dv.unit_info[u * UI_STRIDE + UI_L];
    if (k == FM_NCH) {
        const float *t = dv.fm_t + (int64_t)u * FM_M * FM_W;
#pragma unroll
        for (int p = 0; p < PER; ++p) {
            const int o = tid + p * FM_THREADS;
            if (o < FM_M * FM_W) acc[p] = t[o];
        }
    } else {
        // this CTA's chosen subclusters, listed first so that their loads go out together
        __shared__ int s_sub[(MOG_MAX_UNION * MOG_MAX_L + FM_NCH - 1) / FM_NCH];
        __shared__ int s_ns;
        if (tid == 0) {
            const int *sel = dv.sel + ((int64_t)u * G + g) * SW;
            const int tc = dv.tc, ts = dv.ts;
            int ns = 0;
            for (int e = k; e < tc * ts; e += FM_NCH) {
                const int cl = sel[e / ts], sb = sel[tc + e];
                if (cl >= 0 && sb >= 0) s_sub[ns++] = cl * L + sb;
            }
            s_ns = ns;
        }
        __syncthreads();
        const float *z0 = dv.fm_z + (int64_t)u * dv.c_max * dv.l_max * FM_M * FM_W;
#pragma unroll 4
        for (int e = 0; e < s_ns; ++e) {
            const float *z = z0 + (int64_t)s_sub[e] * FM_M * FM_W;
#pragma unroll
            for (int p = 0; p < PER; ++p) {
                const int o = tid + p * FM_THREADS;
                if (o < FM_M * FM_W) acc[p] += __ldg(z + o);
            }
        }
    }
#pragma unroll
    for (int p = 0; p < PER; ++p) {
        const int o = tid + p * FM_THREADS;
        if (o < FM_M * FM_W) s_acc[o] = acc[p];
    }
    __syncthreads();
    float *out = dv.fm_vec + (((int64_t)u * G + g) * (FM_NCH + 1) + k) * FM_W;
    if (tid <= MOG_D) {
        float s = 0.f;
        for (int i = 0; i < FM_M; ++i) s = fmaf(__expf(s_a[i] - amax), s_acc[i * FM_W + tid], s);
        out[tid] = s;
    }
    if (k == FM_NCH && tid == 0) dv.fm_mref[u * G + g] = amax;
}

cudaError_t launch_fm_build(const Dev &dv, const Plan &pl, cudaStream_t s) {
    k_fm_prep<<<1, FM_M, 0, s>>>(dv);
    k_fm_stats<<<dim3(pl.c_max, pl.units), FM_THREADS, 0, s>>>(dv);
    k_fm_total<<<dim3((FM_M * FM_W + 255) / 256, pl.units), 256, 0, s>>>(dv);
    return cudaGetLastError();
}

cudaError_t launch_fm_resid(const Dev &dv, const uint16_t *q, int SW, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(FM_NCH + 1, dv.G, dv.units);
    cfg.blockDim = dim3(FM_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_fm_resid, dv, q, SW);
}

}  // namespace mog
