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
#include <algorithm>

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

constexpr int SL_STAGES = 2;                  // tile buffers of the slot kernel
constexpr int SL_SPLIT = 2;                   // CTAs per union slot (halves of its rows)
constexpr int SL_ANCHOR = 2;                  // anchor CTAs per unit
constexpr int SL_CHUNK = 32;                  // cluster residual items staged per pass
constexpr int SUPER = 256;                    // row positions resolved per pass
constexpr int SL_AREA = SL_STAGES * AT_STAGE_BYTES;  // 66 KB: selection / tiles / residual

// Bytes of the slot kernel's phase-shared area (selection tables, then tiles, then the
// residual staging); the selection (G*tc ints) follows it.
__host__ __device__ inline size_t slot_area_bytes(int G, int c_max, int tc) {
    const int P1 = (int)ceil_div64(c_max, SC_SLICE);
    const size_t ncw = ((size_t)G * P1 * tc + 3) & ~(size_t)3;
    const size_t sel = sizeof(float) * 2 * ncw + sizeof(uint32_t) * ((c_max + 3) & ~3);
    const size_t res = sizeof(float) * ((size_t)(AT_WARPS + 1) * G * PART_W + (MOG_MAX_L + SL_CHUNK) * MOG_D);
    size_t m = sel > res ? sel : res;
    m = m > (size_t)SL_AREA ? m : (size_t)SL_AREA;
    return (m + 15) & ~(size_t)15;
}

size_t slot_smem_bytes(int G, int c_max, int tc) {
    return slot_area_bytes(G, c_max, tc) + sizeof(int) * (((size_t)G * tc + 3) & ~(size_t)3);
}

// Attention over `nrows` rows whose positions/masks come from `resolve(i0, n)` (filling
// spos/smk for rows i0..i0+n), SUPER rows at a time, two tile buffers.
template <typename Resolve>
__device__ __forceinline__ void slot_rows(WarpAcc &acc, const uint32_t (&qa)[8][4], uint8_t *area,
                                          int nrows, const uint16_t *kb, const uint16_t *vb,
                                          int64_t sn, int *spos, uint32_t *smk, float scale2,
                                          Resolve resolve) {
    for (int sb = 0; sb < nrows; sb += SUPER) {
        const int ns = min(SUPER, nrows - sb);
        resolve(sb, ns);
        __syncthreads();
        const int nt = (int)ceil_div64(ns, AT_ROWS);
        auto issue = [&](int t) {
            const int rb = t * AT_ROWS;
            issue_tile(area + (t % SL_STAGES) * AT_STAGE_BYTES, min(AT_ROWS, ns - rb), kb, vb, sn,
                       [&](int r, int64_t &pos, uint32_t &mk) {
                           pos = spos[rb + r];
                           mk = smk[rb + r];
                       });
        };
        issue(0);
        cp_async_commit();
        if (nt > 1) issue(1);
        cp_async_commit();
        for (int t = 0; t < nt; ++t) {
            cp_async_wait<1>();
            __syncthreads();
            compute_tile(acc, qa, area + (t % SL_STAGES) * AT_STAGE_BYTES, scale2);
            __syncthreads();
            if (t + 2 < nt) issue(t + 2);
            cp_async_commit();
        }
        cp_async_wait<0>();
        __syncthreads();
    }
}

// K2: grid (SL_ANCHOR + SL_SPLIT * min(c_max, G*tc), units).
//  - CTAs a < SL_ANCHOR attend to the anchor rows (sinks, recent and appended keys); they
//    need nothing from the scoring kernel and run ahead of it.
//  - CTA SL_ANCHOR + SL_SPLIT*j + part merges the per-slice candidate lists into every
//    head's top-tc clusters (or takes the caller's selection), forms the union over the G
//    heads (ascending cluster index) and takes union slot j: subcluster scores, top-ts per
//    head that selected the cluster, then attention over `part`'s half of the members of
//    the selected subclusters; part 0 adds the Gaussian residual of the unselected
//    subclusters of that cluster and of a slice of the clusters some head did not select.
//  Every CTA writes one partial (max, sum, acc); the last CTA of the unit merges them
//  and normalises once.
template <int GT>
__global__ void __launch_bounds__(AT_THREADS) k_dec_slot(DecArgs a) {
    extern __shared__ __align__(128) uint8_t area[];
    const Dev &dv = a.dv;
    const int G = dv.G, tc = dv.tc, ts = dv.ts;
    __shared__ float4 w[GT * 64];
    __shared__ float sres[GT][MOG_MAX_L];
    __shared__ float ssl[GT][MOG_MAX_L];
    __shared__ uint32_t smask[MOG_MAX_L];
    __shared__ int sso[MOG_MAX_L + 1], snn[MOG_MAX_L], spref[MOG_MAX_L + 1];
    __shared__ int spos[SUPER];
    __shared__ uint32_t smk[SUPER];
    __shared__ float iex[SL_CHUNK][GT];
    __shared__ uint32_t ineed[SL_CHUNK];
    __shared__ int s_wcnt[AT_WARPS], s_cj, s_uc, s_last;
    const int u = blockIdx.y, r = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int b = ui[UI_B], h = u % dv.h_kv, C = ui[UI_C], L = ui[UI_L];
    const int S = ui[UI_S], rlo = ui[UI_RLO];
    const uint32_t allm = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    const uint16_t *kb = dv.K + b * dv.sb + h * dv.sh;
    const uint16_t *vb = dv.V + b * dv.sb + h * dv.sh;
    const float scale2 = dv.tau * LOG2E;
    uint32_t qa[8][4];
    load_q_frags(qa, a.q + (size_t)u * G * MOG_D, G);
    WarpAcc acc;
    acc.init();
    float *states = reinterpret_cast<float *>(area);  // after the tiles: [AT_WARPS + 1][G][PART_W]
    float *part_out;
    bool has_res = false;
    if (r < SL_ANCHOR) {
        // ------------------------------- anchors ---------------------------------------
        pdl_trigger();
        const int nnow = dv.n_now[b];
        const int s_cnt = min(S, nnow), n_anchor = s_cnt + max(0, nnow - rlo);
        const int i0 = (int)((int64_t)n_anchor * r / SL_ANCHOR), i1 = (int)((int64_t)n_anchor * (r + 1) / SL_ANCHOR);
        slot_rows(acc, qa, area, i1 - i0, kb, vb, dv.sn, spos, smk, scale2, [&](int sb, int ns) {
            for (int t = tid; t < ns; t += AT_THREADS) {
                const int i = i0 + sb + t;
                spos[t] = i < s_cnt ? i : rlo + (i - s_cnt);
                smk[t] = allm;
            }
        });
        part_out = dv.partials + ((size_t)u * PART_SLOTS + r) * G * PART_W;
    } else {
        // ------------------------------- a union slot -----------------------------------
        const int j = (r - SL_ANCHOR) / SL_SPLIT, part = (r - SL_ANCHOR) % SL_SPLIT;
        const int P1 = (int)ceil_div64(dv.c_max, SC_SLICE);
        const int NC = P1 * tc;
        const size_t ncw = ((size_t)G * NC + 3) & ~(size_t)3;
        float *cand_s = reinterpret_cast<float *>(area);                       // [G][NC]
        int *cand_i = reinterpret_cast<int *>(cand_s + ncw);                    // [G][NC]
        uint32_t *cselm = reinterpret_cast<uint32_t *>(cand_i + ncw);           // [c_max]
        // the selection itself outlives the shared area (tiles reuse it): tail region
        int *selc = reinterpret_cast<int *>(area + slot_area_bytes(G, dv.c_max, tc));  // [G][tc]
        load_weights(w, a.q + (size_t)u * G * MOG_D, G, dv.tau);
        for (int e = tid; e < G * tc; e += AT_THREADS) selc[e] = -1;
        for (int e = tid; e < C; e += AT_THREADS) cselm[e] = 0u;
        if (tid < MOG_MAX_L) smask[tid] = 0u;
        pdl_wait();  // candidate lists of the scoring kernel
        pdl_trigger();
        if (tc > 0 && !a.sel_in) {
            const size_t base = (size_t)u * G * NC;
            for (int e = tid; e < G * NC; e += AT_THREADS) {
                cp_async4(smem_u32(cand_s + e), a.cand_s + base + e);
                cp_async4(smem_u32(cand_i + e), a.cand_i + base + e);
            }
            cp_async_commit();
            cp_async_wait<0>();
        }
        __syncthreads();
        if (tc > 0) {
            if (a.sel_in) {
                for (int e = tid; e < G * tc; e += AT_THREADS) {
                    const int g = e / tc, rr = e % tc;
                    const int cc = a.sel_in[((size_t)u * G + g) * a.SW + rr];
                    selc[g * tc + rr] =
                        (cc >= 0 && cc < C && dv.cl_n[(size_t)u * dv.c_max + cc] > 0) ? cc : -1;
                }
            } else {
                // element (g, list p, position r): its rank over all lists of head g is r
                // plus, for every other list, the length of that list's prefix ranking
                // before it
                for (int e = tid; e < G * NC; e += AT_THREADS) {
                    const int g = e / NC, pr = e % NC, pl = pr / tc, rr = pr % tc;
                    const float *cs = cand_s + (size_t)g * NC;
                    const int *ci = cand_i + (size_t)g * NC;
                    const int x = ci[pr];
                    if (x < 0) continue;
                    const float v = cs[pr];
                    int rank = rr;
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
                    if (rank < tc) selc[g * tc + rank] = x;
                }
            }
        }
        __syncthreads();
        for (int e = tid; e < G * tc; e += AT_THREADS) {
            const int cc = selc[(e / tc) * tc + e % tc];
            if (cc >= 0) atomicOr(&cselm[cc], 1u << (e / tc));
        }
        __syncthreads();
        {  // union over the heads, ascending; this CTA's slot
            const int per = (int)ceil_div64(C, AT_THREADS);
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
            if (tid == AT_THREADS - 1) s_uc = base + cnt;
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
        const int Uc = s_uc, R = max(Uc, 1);
        part_out = nullptr;
        if (j < R) {
            part_out = dv.partials + ((size_t)u * PART_SLOTS + r) * G * PART_W;
            const bool has_slot = j < Uc;
            const int c = has_slot ? s_cj : 0;
            const uint32_t hm = has_slot ? cselm[c] : 0u;
            int *selu = dv.sel + (size_t)u * G * a.SW;
            if (j == 0 && part == 0) {
                if (tid == 0) dv.ucount[u] = Uc;
                for (int e = tid; e < G * tc; e += AT_THREADS) {
                    const int g = e / tc, rr = e % tc;
                    const int cc = selc[g * tc + rr];
                    selu[(size_t)g * a.SW + rr] = cc;
                    if (cc < 0)
                        for (int k = 0; k < ts; ++k) selu[(size_t)g * a.SW + tc + rr * ts + k] = -1;
                }
            }
            const size_t g0 = (size_t)u * dv.c_max * dv.l_max + (size_t)c * L;
            const int *so = dv.sub_off + (size_t)u * dv.sub_off_stride + (size_t)c * L;
            int nrows = 0, row0 = 0;
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
                __syncthreads();
                for (int g = warp; g < G; g += AT_WARPS) {  // top-ts of each head that chose c
                    if (!((hm >> g) & 1u)) continue;
                    int rk = -1;
                    for (int rr = 0; rr < tc; ++rr)
                        if (selc[g * tc + rr] == c) { rk = rr; break; }
                    if (rk < 0) continue;
                    int *subs = selu + (size_t)g * a.SW + tc + (size_t)rk * ts;
                    if (a.sel_in) {
                        const int32_t *si = a.sel_in + ((size_t)u * G + g) * a.SW + tc + (size_t)rk * ts;
                        for (int rr = lane; rr < ts; rr += 32) {
                            const int l2 = si[rr];
                            const bool ok = l2 >= 0 && l2 < L && snn[l2] > 0;
                            if (part == 0) subs[rr] = ok ? l2 : -1;
                            if (ok) atomicOr(&smask[l2], 1u << g);
                        }
                    } else {
                        if (part == 0)
                            for (int rr = lane; rr < ts; rr += 32) subs[rr] = -1;
                        __syncwarp();
                        const float v = lane < L ? ssl[g][lane] : -INFINITY;
                        int rank = 0;
                        for (int k = 0; k < L; ++k) rank += ranks_before(ssl[g][k], k, v, lane);
                        if (lane < L && v != -INFINITY && rank < ts) {
                            if (part == 0) subs[rank] = lane;
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
                    if (lane == 0) spref[0] = 0;
                }
                __syncthreads();
                const int T = spref[L];
                row0 = (int)((int64_t)T * part / SL_SPLIT);
                nrows = (int)((int64_t)T * (part + 1) / SL_SPLIT) - row0;
            }
            // ---------------- exact rows of this half ----------------
            const int *perm = dv.perm + (size_t)u * dv.n_cap;
            slot_rows(acc, qa, area, nrows, kb, vb, dv.sn, spos, smk, scale2, [&](int sb, int ns) {
                for (int t = tid; t < ns; t += AT_THREADS) {
                    const int i = row0 + sb + t;
                    int k = 0;
                    while (spref[k + 1] <= i) ++k;
                    int pos = perm[sso[k] + (i - spref[k])];
                    uint32_t mk = smask[k];
                    if ((unsigned)pos >= (unsigned)dv.n_cap) {  // corrupt partition: flag, skip
                        flag_error(dv.status, ST_BAD_INDEX);
                        pos = 0;
                        mk = 0u;
                    }
                    spos[t] = pos;
                    smk[t] = mk;
                }
            });
            // ---------------- Gaussian residual (part 0) ----------------
            if (part == 0 && dv.residual) {
                has_res = true;
                float *vst = states + (size_t)(AT_WARPS + 1) * G * PART_W;  // [32 + SL_CHUNK][d]
                float *vcl = vst + (size_t)MOG_MAX_L * MOG_D;
                const int nsub = has_slot ? L : 0;
                const int cA = (int)((int64_t)C * j / R), cB = (int)((int64_t)C * (j + 1) / R);
                const int ncl = cB - cA;
                const float *cres = dv.cscore + ((size_t)u * 2 + 1) * G * dv.c_max;
                auto stage_clusters = [&](int k0) {
                    const int cnt = min(SL_CHUNK, ncl - k0);
                    for (int e = tid; e < cnt * 32; e += AT_THREADS) {
                        const int cc = cA + k0 + e / 32, k = e % 32;
                        cp_async16(smem_u32(vcl + (size_t)(e / 32) * MOG_D + 4 * k),
                                   dv.cl_vbar + ((size_t)u * dv.c_max + cc) * MOG_D + 4 * k, 16);
                    }
                    cp_async_commit();
                    for (int e = tid; e < cnt; e += AT_THREADS) {
                        const int cc = cA + k0 + e;
                        uint32_t chose = 0u;  // heads that selected cc
                        for (int q = 0; q < G * tc; ++q)
                            if (selc[q] == cc) chose |= 1u << (q / tc);
                        ineed[e] = dv.cl_n[(size_t)u * dv.c_max + cc] > 0 ? (allm & ~chose) : 0u;
#pragma unroll
                        for (int g = 0; g < GT; ++g)
                            if (g < G) iex[e][g] = cres[(size_t)g * dv.c_max + cc];
                    }
                };
                for (int e = tid; e < nsub * 32; e += AT_THREADS)
                    cp_async16(smem_u32(vst + (size_t)(e / 32) * MOG_D + 4 * (e % 32)),
                               dv.sub_vbar + (g0 + e / 32) * MOG_D + 4 * (e % 32), 16);
                if (ncl > 0) stage_clusters(0);
                else cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                // thread (warp, lane) owns dims 4*lane..+3 of heads warp, warp + 4, ...
                OnlineAcc st[MOG_MAX_G / AT_WARPS];
#pragma unroll
                for (int k = 0; k < MOG_MAX_G / AT_WARPS; ++k) st[k].init();
                for (int l = 0; l < nsub; ++l) {
                    if (snn[l] <= 0) continue;
                    const uint32_t need = hm & ~smask[l];
                    const float *vrow = vst + (size_t)l * MOG_D + 4 * lane;
#pragma unroll
                    for (int k = 0; k < MOG_MAX_G / AT_WARPS; ++k) {
                        const int g = warp + AT_WARPS * k;
                        if (g < G && ((need >> g) & 1u)) st[k].absorb(sres[g < GT ? g : 0][l] * LOG2E, vrow);
                    }
                }
                for (int k0 = 0; k0 < ncl; k0 += SL_CHUNK) {
                    if (k0 > 0) {
                        __syncthreads();
                        stage_clusters(k0);
                        cp_async_wait<0>();
                        __syncthreads();
                    }
                    const int cnt = min(SL_CHUNK, ncl - k0);
                    for (int e = 0; e < cnt; ++e) {
                        const float *vrow = vcl + (size_t)e * MOG_D + 4 * lane;
#pragma unroll
                        for (int k = 0; k < MOG_MAX_G / AT_WARPS; ++k) {
                            const int g = warp + AT_WARPS * k;
                            if (g < G && ((ineed[e] >> g) & 1u)) st[k].absorb(iex[e][g < GT ? g : 0] * LOG2E, vrow);
                        }
                    }
                }
                float *rs = states + (size_t)AT_WARPS * G * PART_W;  // state AT_WARPS
#pragma unroll
                for (int k = 0; k < MOG_MAX_G / AT_WARPS; ++k) {
                    const int g = warp + AT_WARPS * k;
                    if (g >= G) continue;
                    float *o = rs + (size_t)g * PART_W;
                    if (lane == 0) {
                        o[0] = st[k].m;
                        o[1] = st[k].l;
                    }
                    *reinterpret_cast<float4 *>(o + PART_ACC + 4 * lane) = st[k].a;
                }
            }
        }
    }
    // ------------------- this CTA's partial; the unit's last CTA merges ------------------
    if (part_out) {
        warp_state_out(acc, states, G);
        __syncthreads();
        merge_states(states, AT_WARPS + (has_res ? 1 : 0), G, part_out);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(dv.counters + u * 4 + 1, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) dv.counters[u * 4 + 1] = 0u;
    const int Uc = dv.tc > 0 ? __ldcg(dv.ucount + u) : 0;
    const int nparts = SL_ANCHOR + SL_SPLIT * max(Uc, 1);
    merge_global_out(dv.partials + (size_t)u * PART_SLOTS * G * PART_W, nparts, G,
                     reinterpret_cast<float *>(area), SL_AREA / 4, a.out + (size_t)u * G * MOG_D);
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

template <int GT>
static cudaError_t launch_steps(const DecArgs &a, cudaStream_t s, cudaEvent_t const *events) {
    const Dev &dv = a.dv;
    cudaError_t e;
    if (events && (e = cudaEventRecord(events[0], s)) != cudaSuccess) return e;
    const int P1 = (int)ceil_div64(dv.c_max, SC_SLICE);
    if ((e = launch_pdl(k_dec_score<GT>, dim3(P1, dv.units), dim3(SC_THREADS), 0, s, a)) != cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[1], s)) != cudaSuccess) return e;
    const size_t sm = slot_smem_bytes(dv.G, dv.c_max, dv.tc);
    if ((e = ensure_smem((const void *)k_dec_slot<GT>, sm)) != cudaSuccess) return e;
    const int nslot = max(1, min(dv.c_max, dv.G * dv.tc));
    if ((e = launch_pdl(k_dec_slot<GT>, dim3(SL_ANCHOR + SL_SPLIT * nslot, dv.units), dim3(AT_THREADS), sm, s,
                        a)) != cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[2], s)) != cudaSuccess) return e;
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
