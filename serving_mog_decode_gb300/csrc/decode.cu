// decode.cu -- one MoG decode step, three kernels chained with programmatic dependent
// launch, plus the append of a new token.
//
// Sources: "Iceberg Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians",
// Abstract (the query is scored against the cluster and subcluster summaries, the most
// relevant are attended exactly, the rest of the cache is approximated from the groups'
// means and variances); newx.sg paper page on retrieval-completion attention, Abstract
// (sink/tail anchors attended exactly; exact and estimated numerator and denominator
// added in the unnormalised domain, one normalisation).
//
//  k_dec_score  (units x P1 CTAs): log-mass score of every cluster for the G query heads
//               of a KV head, s = ln n + tau q.mu + tau^2/2 sum_j q_j^2 var_j; each CTA
//               keeps the top-tc of its slice; the last CTA of a unit merges them
//               (score descending, index ascending), records the selection and the union
//               of selected clusters over the G heads.
//  k_dec_sub    (units x G*tc CTAs): one union cluster per CTA: subcluster scores, top-ts
//               per head that selected the cluster, residual masks of the rest, and the
//               compacted list of rows (positions, head masks) to attend exactly.
//  k_dec_attend (units x P CTAs): rows [p*T/P, (p+1)*T/P) of the unit's exact list (anchors
//               first) through the attention engine, the Gaussian residual terms of a
//               slice of the unselected groups, one partial per CTA; the last CTA of the
//               unit merges the partials and normalises once.
#include "attend.cuh"
#include "internal.h"

namespace mog {

struct DecArgs {
    Dev dv;
    const uint16_t *q;      // [units*G][d]
    float *out;             // [units*G][d]
    const int32_t *sel_in;  // [units*G][SW] or null
    int SW;
    float *cand_s;  // [units][P1][G][tc]
    int *cand_i;
};

// per-head score weights, float4-chunked: w[g][k] (k < 32) holds tau*q over dims 4k..4k+3,
// w[g][32 + k] holds tau^2/2 * q^2 over the same dims
__device__ __forceinline__ void load_weights(float4 *w, const uint16_t *q, int G, float tau) {
    for (int e = threadIdx.x; e < G * 32; e += blockDim.x) {
        const int g = e / 32, k = e % 32;
        const uint2 raw = *reinterpret_cast<const uint2 *>(q + (size_t)g * MOG_D + 4 * k);
        const float q0 = bf_lo(raw.x), q1 = bf_hi(raw.x), q2 = bf_lo(raw.y), q3 = bf_hi(raw.y);
        w[g * 64 + k] = make_float4(tau * q0, tau * q1, tau * q2, tau * q3);
        const float t2 = 0.5f * tau * tau;
        w[g * 64 + 32 + k] = make_float4(t2 * q0 * q0, t2 * q1 * q1, t2 * q2 * q2, t2 * q3 * q3);
    }
}

// Scores of one group by 4 cooperating lanes (lanes 4i..4i+3 of a warp): lane part q reads
// the float4 chunks k = q + 4i of the mean and of the variance.  Returns, on all 4 lanes,
// the log-mass exponent res[g] (the residual's) and the selection score sel[g].
template <int GT>
__device__ __forceinline__ void quad_scores(const float *ms, int n, bool valid, const float4 *w,
                                            int G, int mode, float (&res)[GT], float (&sel)[GT]) {
    const int q = threadIdx.x & 3;
    float4 mu[8], va[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (valid) {
            mu[i] = *reinterpret_cast<const float4 *>(ms + 4 * (q + 4 * i));
            va[i] = *reinterpret_cast<const float4 *>(ms + MOG_D + 4 * (q + 4 * i));
        } else {
            mu[i] = va[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    const float ln = n > 0 ? logf((float)n) : 0.f;
#pragma unroll
    for (int g = 0; g < GT; ++g) {
        if (g >= G) break;
        float dm = 0.f, dq = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 a = w[g * 64 + q + 4 * i], b = w[g * 64 + 32 + q + 4 * i];
            dm += a.x * mu[i].x + a.y * mu[i].y + a.z * mu[i].z + a.w * mu[i].w;
            dq += b.x * va[i].x + b.y * va[i].y + b.z * va[i].z + b.w * va[i].w;
        }
        dm += __shfl_xor_sync(0xffffffffu, dm, 1);
        dm += __shfl_xor_sync(0xffffffffu, dm, 2);
        dq += __shfl_xor_sync(0xffffffffu, dq, 1);
        dq += __shfl_xor_sync(0xffffffffu, dq, 2);
        const bool ok = valid && n > 0;
        res[g] = ok ? ln + dm + dq : -INFINITY;
        sel[g] = !ok ? -INFINITY : (mode == 0 ? res[g] : dm);
    }
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}

// Running (max, sum, acc) of a softmax-weighted sum over 4 output dimensions, log2 domain.
struct OnlineAcc {
    float m, l;
    float4 a;
    __device__ __forceinline__ void init() {
        m = -INFINITY;
        l = 0.f;
        a = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ __forceinline__ void absorb(float ex, const float *v4) {
        if (ex > m) {
            const float sc = exp2f(m - ex);
            l *= sc;
            a.x *= sc;
            a.y *= sc;
            a.z *= sc;
            a.w *= sc;
            m = ex;
        }
        const float wgt = exp2f(ex - m);
        const float4 v = *reinterpret_cast<const float4 *>(v4);
        l += wgt;
        a.x += wgt * v.x;
        a.y += wgt * v.y;
        a.z += wgt * v.z;
        a.w += wgt * v.w;
    }
};

constexpr int SC_SLICE = 32;                 // clusters per scoring CTA
constexpr int SC_THREADS = 4 * SC_SLICE;     // 4 lanes per cluster

// K1: grid (ceil(c_max/32), units).  Scores of a 32-cluster slice for all G heads (clusters
// beyond a unit's C have count 0 and score -inf); the slice's top-tc per head (rank
// counting, score desc then index asc) as a sorted candidate list cand[u][g][slice][tc].
template <int GT>
__global__ void __launch_bounds__(SC_THREADS) k_dec_score(DecArgs a) {
    const Dev &dv = a.dv;
    const int G = dv.G, tc = dv.tc;
    __shared__ float4 w[GT * 64];
    __shared__ float ssel[GT][SC_SLICE];
    const int u = blockIdx.y, p = blockIdx.x;
    const int cl = threadIdx.x >> 2, q4 = threadIdx.x & 3;
    const int c = p * SC_SLICE + cl;
    const bool valid = c < dv.c_max;
    // everything read here is written before the decode step starts
    const float *ms = dv.cl_ms + ((size_t)u * dv.c_max + (valid ? c : 0)) * 2 * MOG_D;
    const int n = valid ? dv.cl_n[(size_t)u * dv.c_max + c] : 0;
    load_weights(w, a.q + (size_t)u * G * MOG_D, G, dv.tau);
    __syncthreads();
    float res[GT], sl[GT];
    quad_scores<GT>(ms, n, valid, w, G, dv.score_mode, res, sl);
    pdl_wait();  // the previous step's readers of cscore/cand are done
    pdl_trigger();
    float *cres = dv.cscore + (size_t)u * 2 * G * dv.c_max;  // [0][g][c] selection, [1][g][c] residual
    if (valid && q4 == 0) {
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            if (g >= G) break;
            cres[(size_t)g * dv.c_max + c] = sl[g];
            cres[((size_t)G + g) * dv.c_max + c] = res[g];
        }
    }
    if (q4 == 0) {
#pragma unroll
        for (int g = 0; g < GT; ++g)
            if (g < G) ssel[g][cl] = valid ? sl[g] : -INFINITY;
    }
    __syncthreads();
    if (tc == 0) return;
    const int P1 = gridDim.x, c0 = p * SC_SLICE;
    const int span = max(SC_SLICE, tc);
    for (int e = threadIdx.x; e < G * span; e += SC_THREADS) {
        const int g = e / span, i = e % span;
        float *cs = a.cand_s + (((size_t)u * G + g) * P1 + p) * tc;
        int *ci = a.cand_i + (((size_t)u * G + g) * P1 + p) * tc;
        if (i < SC_SLICE) {
            const float v = ssel[g][i];
            int rank = 0;
#pragma unroll 8
            for (int k = 0; k < SC_SLICE; ++k) rank += ranks_before(ssel[g][k], k, v, i);
            if (rank < tc) {
                cs[rank] = v;
                ci[rank] = v == -INFINITY ? -1 : c0 + i;
            }
        } else if (i < tc) {
            cs[i] = -INFINITY;
            ci[i] = -1;
        }
    }
}

constexpr int SB_THREADS = 256;
constexpr int SB_CHUNK = 32;  // cluster residual items staged per pass

// K2: grid (max(1, min(c_max, G*tc)), units).  Every CTA merges the per-slice candidate
// lists into each head's top-tc clusters (or takes the caller's selection), forms the union
// over the G heads (ascending cluster index) and takes union slot j: subcluster scores,
// top-ts per head that selected the cluster, the compacted exact rows, and the Gaussian
// residual partial of (a) the unselected subclusters of its cluster and (b) a slice of the
// clusters that some head did not select.
template <int GT>
__global__ void __launch_bounds__(SB_THREADS) k_dec_sub(DecArgs a) {
    extern __shared__ __align__(16) uint8_t sbm[];
    const Dev &dv = a.dv;
    const int G = dv.G, tc = dv.tc, ts = dv.ts;
    const int u = blockIdx.y, j = blockIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], L = ui[UI_L];
    const int P1 = (int)ceil_div64(dv.c_max, SC_SLICE);
    const int NC = P1 * tc;  // candidates per head
    // dynamic shared memory, every region 16-byte aligned
    const size_t ncw = ((size_t)G * NC + 3) & ~(size_t)3;
    float *cand_s = reinterpret_cast<float *>(sbm);                        // [G][NC]
    int *cand_i = reinterpret_cast<int *>(cand_s + ncw);                    // [G][NC]
    uint32_t *cselm = reinterpret_cast<uint32_t *>(cand_i + ncw);           // [c_max]
    float *vst = reinterpret_cast<float *>(cselm + ((dv.c_max + 3) & ~3));  // [32 + SB_CHUNK][d]
    float *vcl = vst + (size_t)MOG_MAX_L * MOG_D;
    __shared__ float4 w[GT * 64];
    __shared__ int selc[GT][MOG_MAX_UNION];
    __shared__ float sres[GT][MOG_MAX_L];
    __shared__ float ssl[GT][MOG_MAX_L];
    __shared__ uint32_t smask[MOG_MAX_L];
    __shared__ int sso[MOG_MAX_L + 1], snn[MOG_MAX_L], spref[MOG_MAX_L + 1];
    __shared__ float iex[SB_CHUNK][GT];
    __shared__ uint32_t ineed[SB_CHUNK];
    __shared__ int s_wcnt[SB_THREADS / 32], s_cj, s_uc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t allm = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    // ---- 0. before the dependency: weights, cleared tables ----
    load_weights(w, a.q + (size_t)u * G * MOG_D, G, dv.tau);
    for (int e = tid; e < G * MOG_MAX_UNION; e += SB_THREADS) selc[e / MOG_MAX_UNION][e % MOG_MAX_UNION] = -1;
    for (int e = tid; e < C; e += SB_THREADS) cselm[e] = 0u;
    if (tid < MOG_MAX_L) smask[tid] = 0u;
    pdl_wait();
    pdl_trigger();
    // ---- 1. every head's top-tc clusters ----
    if (tc > 0 && !a.sel_in) {
        const size_t base = (size_t)u * G * NC;
        for (int e = tid; e < G * NC; e += SB_THREADS) {
            cp_async4(smem_u32(cand_s + e), a.cand_s + base + e);
            cp_async4(smem_u32(cand_i + e), a.cand_i + base + e);
        }
        cp_async_commit();
        cp_async_wait<0>();
    }
    __syncthreads();
    if (tc > 0) {
        if (a.sel_in) {
            for (int e = tid; e < G * tc; e += SB_THREADS) {
                const int g = e / tc, r = e % tc;
                const int cc = a.sel_in[((size_t)u * G + g) * a.SW + r];
                selc[g][r] = (cc >= 0 && cc < C && dv.cl_n[(size_t)u * dv.c_max + cc] > 0) ? cc : -1;
            }
        } else {
            // element (g, list p, position r): its rank over all lists of head g is r plus,
            // for every other list, the length of that list's prefix ranking before it
            for (int e = tid; e < G * NC; e += SB_THREADS) {
                const int g = e / NC, pr = e % NC, pl = pr / tc, r = pr % tc;
                const float *cs = cand_s + (size_t)g * NC;
                const int *ci = cand_i + (size_t)g * NC;
                const int x = ci[pr];
                if (x < 0) continue;
                const float v = cs[pr];
                int rank = r;
                for (int q = 0; q < P1 && rank < tc; ++q) {
                    if (q == pl) continue;
                    int lo = 0, hi = tc;  // first position not ranking before (v, x)
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        const int xm = ci[q * tc + mid];
                        if (xm >= 0 && ranks_before(cs[q * tc + mid], xm, v, x)) lo = mid + 1;
                        else hi = mid;
                    }
                    rank += lo;
                }
                if (rank < tc) selc[g][rank] = x;
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < G * tc; e += SB_THREADS) {
        const int cc = selc[e / tc][e % tc];
        if (cc >= 0) atomicOr(&cselm[cc], 1u << (e / tc));
    }
    __syncthreads();
    // ---- 2. union over the heads, ascending; this CTA's slot ----
    {
        const int per = (int)ceil_div64(C, SB_THREADS);
        const int cA = tid * per, cB = min(C, cA + per);
        int cnt = 0;
        for (int cc = cA; cc < cB; ++cc) cnt += cselm[cc] != 0u;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wcnt[warp] = incl;
        __syncthreads();
        int base = incl - cnt;
        for (int k = 0; k < warp; ++k) base += s_wcnt[k];
        if (tid == SB_THREADS - 1) s_uc = base + cnt;
        if (j >= base && j < base + cnt) {
            int k = base;
            for (int cc = cA; cc < cB; ++cc)
                if (cselm[cc]) {
                    if (k == j) s_cj = cc;
                    ++k;
                }
        }
    }
    __syncthreads();
    const int Uc = s_uc;
    const int R = max(Uc, 1);
    if (j >= R) return;
    const bool has_slot = j < Uc;
    const int c = has_slot ? s_cj : 0;
    const uint32_t hm = has_slot ? cselm[c] : 0u;
    int *selu = dv.sel + (size_t)u * G * a.SW;
    if (j == 0) {
        if (tid == 0) dv.ucount[u] = Uc;
        for (int e = tid; e < G * tc; e += SB_THREADS) {
            const int g = e / tc, r = e % tc;
            selu[(size_t)g * a.SW + r] = selc[g][r];
            if (selc[g][r] < 0)
                for (int k = 0; k < ts; ++k) selu[(size_t)g * a.SW + tc + r * ts + k] = -1;
        }
    }
    // ---- 3. one batch of loads: subcluster summaries and value means, the first chunk of
    //         the cluster residual slice ----
    const size_t g0 = (size_t)u * dv.c_max * dv.l_max + (size_t)c * L;
    const int *so = dv.sub_off + (size_t)u * dv.sub_off_stride + (size_t)c * L;
    const int nsub = (dv.residual && has_slot) ? L : 0;
    const int cA = (int)((int64_t)C * j / R), cB = (int)((int64_t)C * (j + 1) / R);
    const int ncl = dv.residual ? cB - cA : 0;
    const float *cres = dv.cscore + ((size_t)u * 2 + 1) * G * dv.c_max;
    auto stage_clusters = [&](int k0) {  // cluster items k0 .. k0 + SB_CHUNK of the slice
        const int cnt = min(SB_CHUNK, ncl - k0);
        for (int e = tid; e < cnt * 32; e += SB_THREADS) {
            const int cc = cA + k0 + e / 32, k = e % 32;
            cp_async16(smem_u32(vcl + (size_t)(e / 32) * MOG_D + 4 * k),
                       dv.cl_vbar + ((size_t)u * dv.c_max + cc) * MOG_D + 4 * k, 16);
        }
        cp_async_commit();
        for (int e = tid; e < cnt; e += SB_THREADS) {
            const int cc = cA + k0 + e;
            ineed[e] = dv.cl_n[(size_t)u * dv.c_max + cc] > 0 ? (allm & ~cselm[cc]) : 0u;
#pragma unroll
            for (int g = 0; g < GT; ++g)
                if (g < G) iex[e][g] = cres[(size_t)g * dv.c_max + cc];
        }
    };
    if (nsub > 0)
        for (int e = tid; e < L * 32; e += SB_THREADS)
            cp_async16(smem_u32(vst + (size_t)(e / 32) * MOG_D + 4 * (e % 32)),
                       dv.sub_vbar + (g0 + e / 32) * MOG_D + 4 * (e % 32), 16);
    if (ncl > 0) stage_clusters(0);
    else cp_async_commit();
    if (has_slot) {
        if (tid <= L) sso[tid] = so[tid];
        if (tid < L) snn[tid] = dv.sub_n[g0 + tid];
        const int l = tid >> 2;
        const bool valid = l < L;
        float res[GT], sl[GT];
        quad_scores<GT>(dv.sub_ms + (g0 + (valid ? l : 0)) * 2 * MOG_D,
                        valid ? dv.sub_n[g0 + l] : 0, valid, w, G, dv.score_mode, res, sl);
        if (valid && (tid & 3) == 0) {
#pragma unroll
            for (int g = 0; g < GT; ++g)
                if (g < G) {
                    sres[g][l] = res[g];
                    ssl[g][l] = sl[g];
                }
        }
    }
    __syncthreads();
    // ---- 4. top-ts subclusters per head that selected c; compacted exact rows ----
    if (has_slot) {
        for (int g = warp; g < G; g += SB_THREADS / 32) {
            if (!((hm >> g) & 1u)) continue;
            int rk = -1;
            for (int r = 0; r < tc; ++r)
                if (selc[g][r] == c) { rk = r; break; }
            if (rk < 0) continue;
            int *subs = selu + (size_t)g * a.SW + tc + (size_t)rk * ts;
            if (a.sel_in) {
                const int32_t *si = a.sel_in + ((size_t)u * G + g) * a.SW + tc + (size_t)rk * ts;
                for (int r = lane; r < ts; r += 32) {
                    const int l2 = si[r];
                    const bool ok = l2 >= 0 && l2 < L && snn[l2] > 0;
                    subs[r] = ok ? l2 : -1;
                    if (ok) atomicOr(&smask[l2], 1u << g);
                }
            } else {
                for (int r = lane; r < ts; r += 32) subs[r] = -1;
                __syncwarp();
                const float v = lane < L ? ssl[g][lane] : -INFINITY;
                int rank = 0;
                for (int k = 0; k < L; ++k) rank += ranks_before(ssl[g][k], k, v, lane);
                if (lane < L && v != -INFINITY && rank < ts) {
                    subs[rank] = lane;
                    atomicOr(&smask[lane], 1u << g);
                }
            }
        }
        __syncthreads();
        if (warp == 0) {  // prefix of the selected subclusters' sizes
            const int cnt = lane < L && smask[lane] ? sso[lane + 1] - sso[lane] : 0;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane < L) spref[lane + 1] = incl;
            if (lane == 0) {
                spref[0] = 0;
                dv.slotcoff[(size_t)u * MOG_MAX_UNION + j] = sso[0];
            }
            if (lane == L - 1) dv.slotcnt[(size_t)u * MOG_MAX_UNION + j] = incl;
        }
        __syncthreads();
        const int tot = spref[L];
        const int *perm = dv.perm + (size_t)u * dv.n_cap;
        int *rp = dv.rowpos + (size_t)u * dv.n_cap + sso[0];
        uint32_t *rm = dv.rowmask + (size_t)u * dv.n_cap + sso[0];
        for (int i = tid; i < tot; i += SB_THREADS) {
            int k = 0;
            while (spref[k + 1] <= i) ++k;
            rp[i] = perm[sso[k] + (i - spref[k])];
            rm[i] = smask[k];
        }
    }
    // ---- 5. Gaussian residual partial: thread (g, quad) owns dims 4*quad..+3 of head
    //         g = warp and, when G > 8, also of head warp + 8 ----
    const int rq = tid & 31;
    OnlineAcc st[2];
    st[0].init();
    st[1].init();
    const int hA = warp, hB = warp + SB_THREADS / 32;
    cp_async_wait<0>();
    __syncthreads();
    for (int l = 0; l < nsub; ++l) {
        if (snn[l] <= 0) continue;
        const uint32_t need = hm & ~smask[l];
        const float *vrow = vst + (size_t)l * MOG_D + 4 * rq;
        if (hA < G && ((need >> hA) & 1u)) st[0].absorb(sres[hA][l] * LOG2E, vrow);
        if (hB < G && ((need >> hB) & 1u)) st[1].absorb(sres[hB][l] * LOG2E, vrow);
    }
    for (int k0 = 0; k0 < ncl; k0 += SB_CHUNK) {
        if (k0 > 0) {  // further chunks of the cluster slice (large C, few slots)
            __syncthreads();
            stage_clusters(k0);
            cp_async_wait<0>();
            __syncthreads();
        }
        const int cnt = min(SB_CHUNK, ncl - k0);
        for (int e = 0; e < cnt; ++e) {
            const float *vrow = vcl + (size_t)e * MOG_D + 4 * rq;
            if (hA < G && ((ineed[e] >> hA) & 1u)) st[0].absorb(iex[e][hA] * LOG2E, vrow);
            if (hB < G && ((ineed[e] >> hB) & 1u)) st[1].absorb(iex[e][hB < GT ? hB : 0] * LOG2E, vrow);
        }
    }
    float *rbase = dv.partials + ((size_t)u * PART_SLOTS + MAX_SPLITS + j) * G * PART_W;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int g = k == 0 ? hA : hB;
        if (g >= G) continue;
        float *r = rbase + (size_t)g * PART_W;
        if (rq == 0) {
            r[0] = st[k].m;
            r[1] = st[k].l;
        }
        *reinterpret_cast<float4 *>(r + PART_ACC + 4 * rq) = st[k].a;
    }
}

constexpr int SUPER = 256;  // rows resolved per pass
constexpr int RB = 2;       // residual partials staged per pass in the attention kernel

// K3: grid (P, units).  Rows [p*T/P, (p+1)*T/P) of the unit's exact list (anchors first),
// plus residual partials [p*R/P, (p+1)*R/P) from k_dec_sub, into one partial; the last CTA
// of the unit merges the P partials and normalises once.
template <int GT>
__global__ void __launch_bounds__(AT_THREADS) k_dec_attend(DecArgs a) {
    extern __shared__ __align__(128) uint8_t asm_[];
    const Dev &dv = a.dv;
    const int G = dv.G;
    __shared__ int spre[MOG_MAX_UNION + 1];
    __shared__ int scoff[MOG_MAX_UNION];
    __shared__ int spos[SUPER];
    __shared__ uint32_t smk[SUPER];
    __shared__ int s_last;
    const int u = blockIdx.y, p = blockIdx.x, P = dv.P;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int b = ui[UI_B], h = u % dv.h_kv;
    const int S = ui[UI_S], rlo = ui[UI_RLO];
    const int nnow = dv.n_now[b];
    const int s_cnt = min(S, nnow), r_cnt = max(0, nnow - rlo);
    const int n_anchor = s_cnt + r_cnt;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t allm = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    uint32_t qa[8][4];
    load_q_frags(qa, a.q + (size_t)u * G * MOG_D, G);
    pdl_wait();  // below: outputs of the subcluster kernel
    pdl_trigger();
    const int Uc = dv.tc > 0 ? dv.ucount[u] : 0;
    const int R = max(Uc, 1);
    // shared memory: [tiles (AT_SMEM)][RB staged residual partials]; after the tile loop
    // the warp states go right before the staged partials, at the end of the tile area
    float *stR = reinterpret_cast<float *>(asm_ + AT_SMEM);
    float *stA = stR - (size_t)AT_WARPS * G * PART_W;
    // residual partials of this CTA: fetch now, merge at the end
    const int ra = (int)((int64_t)R * p / P), rb = (int)((int64_t)R * (p + 1) / P);
    const float *rsrc = dv.partials + ((size_t)u * PART_SLOTS + MAX_SPLITS) * G * PART_W;
    {
        const int cnt = min(RB, rb - ra);
        for (int q = tid; q < cnt * G * PART_W / 4; q += AT_THREADS)
            cp_async16(smem_u32(stR + 4 * q), rsrc + (size_t)ra * G * PART_W + 4 * q, 16);
        cp_async_commit();
    }
    if (warp == 0) {  // slot prefix over <= 256 slots
        int run = n_anchor;
        for (int j0 = 0; j0 < Uc; j0 += 32) {
            const int j = j0 + lane;
            int cnt = 0;
            if (j < Uc) {
                const size_t sj = (size_t)u * MOG_MAX_UNION + j;
                cnt = dv.slotcnt[sj];
                scoff[j] = dv.slotcoff[sj];
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (j < Uc) spre[j] = run + incl - cnt;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) spre[Uc] = run;
    }
    __syncthreads();
    const int T = spre[Uc];
    const int r0 = (int)((int64_t)T * p / P), r1 = (int)((int64_t)T * (p + 1) / P);
    const uint16_t *kb = dv.K + b * dv.sb + h * dv.sh;
    const uint16_t *vb = dv.V + b * dv.sb + h * dv.sh;
    const int *rowpos = dv.rowpos + (size_t)u * dv.n_cap;
    const uint32_t *rowmask = dv.rowmask + (size_t)u * dv.n_cap;
    WarpAcc acc;
    acc.init();
    const float scale2 = dv.tau * LOG2E;
    int sbase = r0, ns = 0, nt = 0;
    auto resolve = [&]() {
        ns = min(SUPER, r1 - sbase);
        for (int t = tid; t < ns; t += AT_THREADS) {
            const int i = sbase + t;
            int pos;
            uint32_t mk;
            if (i < n_anchor) {
                pos = i < s_cnt ? i : rlo + (i - s_cnt);
                mk = allm;
            } else {
                int lo = 0, hi = Uc - 1;  // last slot with spre[slot] <= i
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (spre[mid] <= i) lo = mid;
                    else hi = mid - 1;
                }
                const int k = scoff[lo] + (i - spre[lo]);
                pos = rowpos[k];
                mk = rowmask[k];
            }
            if ((unsigned)pos >= (unsigned)dv.n_cap) {  // corrupt row list: flag, skip
                flag_error(dv.status, ST_BAD_INDEX);
                pos = 0;
                mk = 0u;
            }
            spos[t] = pos;
            smk[t] = mk;
        }
        __syncthreads();
        nt = (int)ceil_div64(ns, AT_ROWS);
    };
    auto issue = [&](int t) {
        const int rbs = t * AT_ROWS;
        issue_tile(asm_ + (t % AT_STAGES) * AT_STAGE_BYTES, min(AT_ROWS, ns - rbs), kb, vb, dv.sn,
                   [&](int r, int64_t &pos, uint32_t &mk) {
                       pos = spos[rbs + r];
                       mk = smk[rbs + r];
                   });
    };
    while (sbase < r1) {
        resolve();
#pragma unroll
        for (int s = 0; s < AT_STAGES - 1; ++s) {
            if (s < nt) issue(s);
            cp_async_commit();
        }
        for (int t = 0; t < nt; ++t) {
            cp_async_wait<AT_STAGES - 2>();
            __syncthreads();
            if (t + AT_STAGES - 1 < nt) issue(t + AT_STAGES - 1);
            cp_async_commit();
            compute_tile(acc, qa, asm_ + (t % AT_STAGES) * AT_STAGE_BYTES, scale2);
        }
        cp_async_wait<0>();
        __syncthreads();
        sbase += SUPER;
    }
    cp_async_wait<0>();
    warp_state_out(acc, stA, G);
    __syncthreads();
    float *part = dv.partials + ((size_t)u * PART_SLOTS + p) * G * PART_W;
    const int nres = max(0, min(RB, rb - ra));
    if (rb - ra <= RB) {
        merge_states(stA, AT_WARPS + nres, G, part);  // stA and stR are contiguous
    } else {
        // more residual partials than one stage: fold them in RB at a time through the
        // (now free) tile area: run[0] holds the running state, run[1..] the staged chunk
        float *run = reinterpret_cast<float *>(asm_);
        float *tmp = run + (size_t)(1 + RB) * G * PART_W;
        merge_states(stA, AT_WARPS + nres, G, tmp);
        for (int k0 = ra + RB; k0 < rb; k0 += RB) {
            __syncthreads();
            for (int q = tid; q < G * PART_W; q += AT_THREADS) run[q] = tmp[q];
            const int cnt = min(RB, rb - k0);
            for (int q = tid; q < cnt * G * PART_W / 4; q += AT_THREADS)
                cp_async16(smem_u32(run + (size_t)G * PART_W + 4 * q), rsrc + (size_t)k0 * G * PART_W + 4 * q, 16);
            cp_async_commit();
            cp_async_wait<0>();
            __syncthreads();
            merge_states(run, 1 + cnt, G, k0 + RB >= rb ? part : tmp);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(dv.counters + u * 4 + 1, 1u);
        s_last = (t == (unsigned)P - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) dv.counters[u * 4 + 1] = 0u;
    merge_global_out(dv.partials + (size_t)u * PART_SLOTS * G * PART_W, P, G,
                     reinterpret_cast<float *>(asm_), AT_SMEM / 4, a.out + (size_t)u * G * MOG_D);
}

// Append one token per sequence at position n_now[b], then advance n_now[b].
__global__ void k_append(Dev dv, const uint16_t *kn, const uint16_t *vn) {
    const int b = blockIdx.x;
    const int pos = dv.n_now[b];
    for (int e = threadIdx.x; e < dv.h_kv * 16; e += blockDim.x) {
        const int h = e / 16, ch = e % 16;
        const size_t src = ((size_t)b * dv.h_kv + h) * MOG_D + ch * 8;
        uint16_t *kd = dv.Kw + b * dv.sb + h * dv.sh + (int64_t)pos * dv.sn + ch * 8;
        uint16_t *vd = dv.Vw + b * dv.sb + h * dv.sh + (int64_t)pos * dv.sn + ch * 8;
        *reinterpret_cast<uint4 *>(kd) = *reinterpret_cast<const uint4 *>(kn + src);
        *reinterpret_cast<uint4 *>(vd) = *reinterpret_cast<const uint4 *>(vn + src);
    }
    __syncthreads();
    if (threadIdx.x == 0) dv.n_now[b] = pos + 1;
}

// ------------------------------------------------------------------------------------
template <typename K>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              const DecArgs &a) {
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
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

size_t sub_smem_bytes(int G, int c_max, int tc) {
    const int P1 = (int)ceil_div64(c_max, SC_SLICE);
    const size_t ncw = ((size_t)G * P1 * tc + 3) & ~(size_t)3;  // 16-byte multiples
    return sizeof(float) * 2 * ncw + sizeof(uint32_t) * ((c_max + 3) & ~3) +
           sizeof(float) * (MOG_MAX_L + SB_CHUNK) * MOG_D;  // value means staged
}

template <int GT>
static cudaError_t launch_steps(const DecArgs &a, cudaStream_t s, cudaEvent_t const *events) {
    const Dev &dv = a.dv;
    cudaError_t e;
    if (events && (e = cudaEventRecord(events[0], s)) != cudaSuccess) return e;
    const int P1 = (int)ceil_div64(dv.c_max, SC_SLICE);
    if ((e = launch_pdl(k_dec_score<GT>, dim3(P1, dv.units), dim3(SC_THREADS), 0, s, a)) != cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[1], s)) != cudaSuccess) return e;
    const size_t sm2 = sub_smem_bytes(dv.G, dv.c_max, dv.tc);
    if ((e = ensure_smem((const void *)k_dec_sub<GT>, sm2)) != cudaSuccess) return e;
    const int nslot = max(1, min(dv.c_max, dv.G * dv.tc));
    if ((e = launch_pdl(k_dec_sub<GT>, dim3(nslot, dv.units), dim3(SB_THREADS), sm2, s, a)) != cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[2], s)) != cudaSuccess) return e;
    const size_t sm3 = AT_SMEM + sizeof(float) * RB * dv.G * PART_W;
    if ((e = ensure_smem((const void *)k_dec_attend<GT>, sm3)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_dec_attend<GT>, dim3(dv.P, dv.units), dim3(AT_THREADS), sm3, s, a)) != cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[3], s)) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_decode(const Dev &dv, const Plan &pl, const void *q, float *out,
                          const int32_t *sel_in, int32_t *sel_out, cudaStream_t s,
                          cudaEvent_t const *events) {
    DecArgs a;
    a.dv = dv;
    a.q = static_cast<const uint16_t *>(q);
    a.out = out;
    a.sel_in = sel_in;
    a.SW = dv.tc + dv.tc * dv.ts;
    a.cand_s = dv.cand_s;
    a.cand_i = dv.cand_i;
    const int G = dv.G;
    cudaError_t e;
    if (G <= 1) e = launch_steps<1>(a, s, events);
    else if (G <= 2) e = launch_steps<2>(a, s, events);
    else if (G <= 4) e = launch_steps<4>(a, s, events);
    else if (G <= 8) e = launch_steps<8>(a, s, events);
    else e = launch_steps<16>(a, s, events);
    if (e != cudaSuccess) return e;
    if (sel_out && a.SW > 0)
        e = cudaMemcpyAsync(sel_out, dv.sel, sizeof(int32_t) * (size_t)dv.units * G * a.SW,
                            cudaMemcpyDeviceToDevice, s);
    return e;
}

cudaError_t launch_append(const Dev &dv, const Plan &pl, const void *k_new, const void *v_new,
                          cudaStream_t s) {
    k_append<<<pl.batch, 128, 0, s>>>(dv, static_cast<const uint16_t *>(k_new),
                                      static_cast<const uint16_t *>(v_new));
    return cudaGetLastError();
}

}  // namespace mog
