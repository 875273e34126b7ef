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

// per-head score weights: w[g][0..d) = tau q, w[g][d..2d) = tau^2/2 q^2
__device__ __forceinline__ void load_weights(float *w, const uint16_t *q, int G, float tau) {
    for (int e = threadIdx.x; e < G * MOG_D; e += blockDim.x) {
        const int g = e / MOG_D, j = e % MOG_D;
        const float qv = bf1(q[(size_t)g * MOG_D + j]);
        w[g * 2 * MOG_D + j] = tau * qv;
        w[g * 2 * MOG_D + MOG_D + j] = 0.5f * tau * tau * qv * qv;
    }
}

// warp-cooperative: scores of one group (summary ms[2d]) for heads g < G.
// Returns through res[g], sel[g] on every lane.
__device__ __forceinline__ void group_scores(const float *ms, int n, const float *w, int G,
                                             int mode, float *res, float *sel) {
    const int lane = threadIdx.x & 31;
    const float4 mu = *reinterpret_cast<const float4 *>(ms + lane * 4);
    const float4 va = *reinterpret_cast<const float4 *>(ms + MOG_D + lane * 4);
    const float ln = n > 0 ? logf((float)n) : 0.f;
    for (int g = 0; g < G; ++g) {
        const float4 wm = *reinterpret_cast<const float4 *>(w + g * 2 * MOG_D + lane * 4);
        const float4 wv = *reinterpret_cast<const float4 *>(w + g * 2 * MOG_D + MOG_D + lane * 4);
        float dm = wm.x * mu.x + wm.y * mu.y + wm.z * mu.z + wm.w * mu.w;
        float dq = wv.x * va.x + wv.y * va.y + wv.z * va.z + wv.w * va.w;
        dm = warp_sum(dm);
        dq = warp_sum(dq);
        const float r = n > 0 ? ln + dm + dq : -INFINITY;
        res[g] = r;
        sel[g] = mode == 0 ? r : (n > 0 ? dm : -INFINITY);
    }
}

// warp argmax over (value desc, index asc); returns the winner on every lane
__device__ __forceinline__ void warp_best(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ranks_before(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

constexpr int SC_THREADS = 256;
constexpr int SC_SLICE = 64;  // clusters per score CTA at most (two per lane)
constexpr int SC_PER_WARP = SC_SLICE / (SC_THREADS / 32);

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}

__global__ void __launch_bounds__(SC_THREADS) k_dec_score(DecArgs a) {
    extern __shared__ __align__(16) float scs[];
    const Dev &dv = a.dv;
    const int G = dv.G, tc = dv.tc;
    float *w = scs;                               // [G][2d]
    float *ssel = w + G * 2 * MOG_D;              // [G][SC_SLICE]
    float *stg_s = ssel + G * SC_SLICE;           // [8 warps][P1*tc]
    int *stg_i = reinterpret_cast<int *>(stg_s + 8 * dv.P1 * max(tc, 1));
    __shared__ int s_last;
    __shared__ int s_wcnt[8];
    pdl_wait();
    pdl_trigger();
    const int u = blockIdx.y, p = blockIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C];
    const int c0 = (int)((int64_t)C * p / dv.P1), c1 = (int)((int64_t)C * (p + 1) / dv.P1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // summaries of this warp's clusters, loaded before the weights are ready
    float4 mu[SC_PER_WARP], va[SC_PER_WARP];
    int nn[SC_PER_WARP];
#pragma unroll
    for (int k = 0; k < SC_PER_WARP; ++k) {
        const int c = c0 + warp + 8 * k;
        nn[k] = 0;
        if (c < c1) {
            const float *ms = dv.cl_ms + ((size_t)u * dv.c_max + c) * 2 * MOG_D;
            mu[k] = *reinterpret_cast<const float4 *>(ms + lane * 4);
            va[k] = *reinterpret_cast<const float4 *>(ms + MOG_D + lane * 4);
            nn[k] = dv.cl_n[(size_t)u * dv.c_max + c];
        }
    }
    load_weights(w, a.q + (size_t)u * G * MOG_D, G, dv.tau);
    __syncthreads();
    float *cres = dv.cscore + (size_t)u * 2 * G * dv.c_max;  // [0][g][c] selection, [1][g][c] residual
#pragma unroll
    for (int k = 0; k < SC_PER_WARP; ++k) {
        const int c = c0 + warp + 8 * k;
        if (c >= c1) break;
        const int n = nn[k];
        const float ln = n > 0 ? logf((float)n) : 0.f;
        for (int g = 0; g < G; ++g) {
            const float4 wm = *reinterpret_cast<const float4 *>(w + g * 2 * MOG_D + lane * 4);
            const float4 wv = *reinterpret_cast<const float4 *>(w + g * 2 * MOG_D + MOG_D + lane * 4);
            float dm = wm.x * mu[k].x + wm.y * mu[k].y + wm.z * mu[k].z + wm.w * mu[k].w;
            float dq = wv.x * va[k].x + wv.y * va[k].y + wv.z * va[k].z + wv.w * va[k].w;
            dm = warp_sum(dm);
            dq = warp_sum(dq);
            const float r = n > 0 ? ln + dm + dq : -INFINITY;
            const float sl = dv.score_mode == 0 ? r : (n > 0 ? dm : -INFINITY);
            if (lane == 0) {
                cres[(size_t)g * dv.c_max + c] = sl;
                cres[((size_t)G + g) * dv.c_max + c] = r;
                ssel[g * SC_SLICE + (c - c0)] = sl;
            }
        }
        if (lane == 0) dv.cselmask[(size_t)u * dv.c_max + c] = 0u;
    }
    __syncthreads();
    // local top-tc of this slice, per head
    const int ns = c1 - c0;
    for (int g = warp; g < G && tc > 0; g += SC_THREADS / 32) {
        float v0 = lane < ns ? ssel[g * SC_SLICE + lane] : -INFINITY;
        float v1 = lane + 32 < ns ? ssel[g * SC_SLICE + lane + 32] : -INFINITY;
        float *cs = a.cand_s + (((size_t)u * G + g) * dv.P1 + p) * tc;
        int *ci = a.cand_i + (((size_t)u * G + g) * dv.P1 + p) * tc;
        for (int r = 0; r < tc; ++r) {
            float bv;
            int bi;
            if (ranks_before(v1, c0 + lane + 32, v0, c0 + lane)) {
                bv = v1;
                bi = c0 + lane + 32;
            } else {
                bv = v0;
                bi = c0 + lane;
            }
            warp_best(bv, bi);
            if (bv == -INFINITY) {
                for (int rr = r + lane; rr < tc; rr += 32) {
                    cs[rr] = -INFINITY;
                    ci[rr] = -1;
                }
                break;
            }
            if (lane == 0) {
                cs[r] = bv;
                ci[r] = bi;
            }
            if (bi == c0 + lane) v0 = -INFINITY;
            if (bi == c0 + lane + 32) v1 = -INFINITY;
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(dv.counters + u * 4 + 0, 1u);
        s_last = (t == (unsigned)dv.P1 - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) dv.counters[u * 4 + 0] = 0u;
    // ---- last CTA of the unit: merge the P1 sorted candidate lists of every head ----
    int *sel = dv.sel + (size_t)u * G * a.SW;
    const int ncand = dv.P1 * tc;
    for (int g = warp; g < G; g += SC_THREADS / 32) {
        int *sg = sel + (size_t)g * a.SW;
        for (int e = lane; e < a.SW; e += 32) sg[e] = -1;
        __syncwarp();
        if (tc == 0) continue;
        if (a.sel_in) {
            const int32_t *si = a.sel_in + ((size_t)u * G + g) * a.SW;
            for (int r = lane; r < tc; r += 32) {
                const int c = si[r];
                sg[r] = (c >= 0 && c < C && dv.cl_n[(size_t)u * dv.c_max + c] > 0) ? c : -1;
            }
        } else {
            float *ss = stg_s + warp * ncand;
            int *sx = stg_i + warp * ncand;
            const size_t base = ((size_t)u * G + g) * ncand;
            for (int e = lane; e < ncand; e += 32) {
                cp_async4(smem_u32(ss + e), a.cand_s + base + e);
                cp_async4(smem_u32(sx + e), a.cand_i + base + e);
            }
            cp_async_commit();
            cp_async_wait<0>();
            __syncwarp();
            // lane k walks lists k and k+32
            int p0 = 0, p1 = 0;
            for (int r = 0; r < tc; ++r) {
                float va = -INFINITY, vb = -INFINITY;
                int ia = 0x7fffffff, ib = 0x7fffffff;
                if (lane < dv.P1 && p0 < tc && sx[lane * tc + p0] >= 0) {
                    va = ss[lane * tc + p0];
                    ia = sx[lane * tc + p0];
                }
                if (lane + 32 < dv.P1 && p1 < tc && sx[(lane + 32) * tc + p1] >= 0) {
                    vb = ss[(lane + 32) * tc + p1];
                    ib = sx[(lane + 32) * tc + p1];
                }
                const bool takeb = ranks_before(vb, ib, va, ia);
                float bv = takeb ? vb : va;
                int bi = takeb ? ib : ia;
                warp_best(bv, bi);
                if (bv == -INFINITY) break;
                if (lane == 0) sg[r] = bi;
                if (!takeb && ia == bi) ++p0;
                else if (takeb && ib == bi) ++p1;
            }
        }
        __syncwarp();
        for (int r = lane; r < tc; r += 32)
            if (sg[r] >= 0) atomicOr(dv.cselmask + (size_t)u * dv.c_max + sg[r], 1u << g);
    }
    __syncthreads();
    // union of the selected clusters over the G heads, ascending cluster index
    {
        const int per = (int)ceil_div64(C, SC_THREADS);
        const int cA = threadIdx.x * per, cB = min(C, cA + per);
        const uint32_t *cm = dv.cselmask + (size_t)u * dv.c_max;
        int cnt = 0;
        for (int c = cA; c < cB; ++c) cnt += __ldcg(cm + c) != 0u;
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
        for (int c = cA; c < cB; ++c) {
            const uint32_t m = __ldcg(cm + c);
            if (m) {
                dv.ucl[(size_t)u * MOG_MAX_UNION + base] = c;
                dv.uhm[(size_t)u * MOG_MAX_UNION + base] = m;
                ++base;
            }
        }
        if (threadIdx.x == SC_THREADS - 1) dv.ucount[u] = base;
    }
}

constexpr int SUB_THREADS = 128;

__global__ void __launch_bounds__(SUB_THREADS) k_dec_sub(DecArgs a) {
    extern __shared__ __align__(16) float sbs[];
    const Dev &dv = a.dv;
    const int G = dv.G;
    float *w = sbs;                        // [G][2d]
    float *sres = w + G * 2 * MOG_D;       // [G][32]
    float *ssel = sres + G * MOG_MAX_L;    // [G][32]
    __shared__ uint32_t smask[MOG_MAX_L];
    __shared__ int spref[MOG_MAX_L + 1];
    __shared__ int sso[MOG_MAX_L + 1];
    __shared__ int snn[MOG_MAX_L];
    pdl_wait();
    pdl_trigger();
    const int u = blockIdx.y, j = blockIdx.x;
    if (j >= dv.ucount[u]) return;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int L = ui[UI_L];
    const int c = dv.ucl[(size_t)u * MOG_MAX_UNION + j];
    const uint32_t hm = dv.uhm[(size_t)u * MOG_MAX_UNION + j];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int *so = dv.sub_off + (size_t)u * dv.sub_off_stride + (size_t)c * L;
    const size_t g0 = (size_t)u * dv.c_max * dv.l_max + (size_t)c * L;
    if (threadIdx.x <= (unsigned)L) sso[threadIdx.x] = so[threadIdx.x];
    if (threadIdx.x < (unsigned)L) snn[threadIdx.x] = dv.sub_n[g0 + threadIdx.x];
    if (threadIdx.x < MOG_MAX_L) smask[threadIdx.x] = 0u;
    load_weights(w, a.q + (size_t)u * G * MOG_D, G, dv.tau);
    __syncthreads();
    float res[MOG_MAX_G], sl[MOG_MAX_G];
    for (int l = warp; l < L; l += SUB_THREADS / 32) {
        group_scores(dv.sub_ms + (g0 + l) * 2 * MOG_D, snn[l], w, G, dv.score_mode, res, sl);
        if (lane == 0)
            for (int g = 0; g < G; ++g) {
                sres[g * MOG_MAX_L + l] = res[g];
                ssel[g * MOG_MAX_L + l] = sl[g];
            }
    }
    __syncthreads();
    int *selu = dv.sel + (size_t)u * G * a.SW;
    for (int g = warp; g < G; g += SUB_THREADS / 32) {
        if (!((hm >> g) & 1u)) continue;
        int *sg = selu + (size_t)g * a.SW;
        int rk = -1;  // rank of c in this head's cluster list
        for (int r0 = 0; r0 < dv.tc; r0 += 32) {
            const int r = r0 + lane;
            const uint32_t b = __ballot_sync(0xffffffffu, r < dv.tc && sg[r] == c);
            if (b) {
                rk = r0 + __ffs(b) - 1;
                break;
            }
        }
        if (rk < 0) continue;
        int *subs = sg + dv.tc + rk * dv.ts;
        if (a.sel_in) {
            const int32_t *si = a.sel_in + ((size_t)u * G + g) * a.SW + dv.tc + rk * dv.ts;
            for (int r = lane; r < dv.ts; r += 32) {
                const int l = si[r];
                const bool ok = l >= 0 && l < L && snn[l] > 0;
                subs[r] = ok ? l : -1;
                if (ok) atomicOr(&smask[l], 1u << g);
            }
        } else {
            float v = lane < L ? ssel[g * MOG_MAX_L + lane] : -INFINITY;
            for (int r = 0; r < dv.ts; ++r) {
                float bv = v;
                int bi = lane;
                warp_best(bv, bi);
                if (bv == -INFINITY) break;
                if (lane == 0) {
                    subs[r] = bi;
                    atomicOr(&smask[bi], 1u << g);
                }
                if (bi == lane) v = -INFINITY;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x < (unsigned)L) {
        const int l = threadIdx.x;
        dv.subres[((size_t)u * MOG_MAX_UNION + j) * MOG_MAX_L + l] = snn[l] > 0 ? (hm & ~smask[l]) : 0u;
        for (int g = 0; g < G; ++g)
            dv.subscore[(((size_t)u * MOG_MAX_UNION + j) * G + g) * MOG_MAX_L + l] = sres[g * MOG_MAX_L + l];
    }
    if (threadIdx.x == 0) {
        spref[0] = 0;
        for (int l = 0; l < L; ++l) spref[l + 1] = spref[l] + (smask[l] ? sso[l + 1] - sso[l] : 0);
        dv.slotcnt[(size_t)u * MOG_MAX_UNION + j] = spref[L];
        dv.slotcoff[(size_t)u * MOG_MAX_UNION + j] = sso[0];
    }
    __syncthreads();
    // compacted rows of the selected subclusters, one flat parallel pass
    const int tot = spref[L];
    const int *perm = dv.perm + (size_t)u * dv.n_cap;
    int *rp = dv.rowpos + (size_t)u * dv.n_cap + sso[0];
    uint32_t *rm = dv.rowmask + (size_t)u * dv.n_cap + sso[0];
    for (int i = threadIdx.x; i < tot; i += SUB_THREADS) {
        int l = 0;
        while (spref[l + 1] <= i) ++l;
        rp[i] = perm[sso[l] + (i - spref[l])];
        rm[i] = smask[l];
    }
}

constexpr int SUPER = 256;  // rows resolved per pass

template <int GT>
__global__ void __launch_bounds__(AT_THREADS) k_dec_attend(DecArgs a) {
    extern __shared__ __align__(128) uint8_t asm_[];
    const Dev &dv = a.dv;
    const int G = dv.G;
    __shared__ int spre[MOG_MAX_UNION + 1];
    __shared__ int scoff[MOG_MAX_UNION];
    __shared__ int sucl[MOG_MAX_UNION];
    __shared__ int spos[SUPER];
    __shared__ uint32_t smk[SUPER];
    __shared__ int s_last;
    pdl_wait();
    pdl_trigger();
    const int u = blockIdx.y, p = blockIdx.x, P = dv.P;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int b = ui[UI_B], h = u % dv.h_kv, C = ui[UI_C], L = ui[UI_L];
    const int S = ui[UI_S], rlo = ui[UI_RLO];
    const int nnow = dv.n_now[b];
    const int s_cnt = min(S, nnow), r_cnt = max(0, nnow - rlo);
    const int n_anchor = s_cnt + r_cnt;
    const int Uc = dv.ucount[u];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t allm = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    if (warp == 0) {  // slot prefix over <= 256 slots
        int run = n_anchor;
        for (int j0 = 0; j0 < Uc; j0 += 32) {
            const int j = j0 + lane;
            int cnt = 0;
            if (j < Uc) {
                const size_t sj = (size_t)u * MOG_MAX_UNION + j;
                cnt = dv.slotcnt[sj];
                scoff[j] = dv.slotcoff[sj];
                sucl[j] = dv.ucl[sj];
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
    uint32_t qa[8][4];
    load_q_frags(qa, a.q + (size_t)u * G * MOG_D, G);
    WarpAcc acc;
    acc.init();
    const float scale2 = dv.tau * LOG2E;
    float *stB = reinterpret_cast<float *>(asm_ + AT_SMEM);        // [AT_WARPS][G][PART_W]
    float *stA = stB - AT_WARPS * G * PART_W;                      // aliases the tile area

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
        const int rb = t * AT_ROWS;
        issue_tile(asm_ + (t % AT_STAGES) * AT_STAGE_BYTES, min(AT_ROWS, ns - rb), kb, vb, dv.sn,
                   [&](int r, int64_t &pos, uint32_t &mk) {
                       pos = spos[rb + r];
                       mk = smk[rb + r];
                   });
    };
    auto prologue = [&]() {
#pragma unroll
        for (int s = 0; s < AT_STAGES - 1; ++s) {
            if (s < nt) issue(s);
            cp_async_commit();
        }
    };
    if (sbase < r1) {
        resolve();
        prologue();
    }
    // ---------- Gaussian residual of this CTA's slice of unselected groups ----------
    // (runs while the first tiles are in flight; per-warp online softmax over items)
    {
        const int I = Uc * L;
        const int cA = (int)((int64_t)C * p / P), cB = (int)((int64_t)C * (p + 1) / P);
        const int iA = (int)((int64_t)I * p / P), iB = (int)((int64_t)I * (p + 1) / P);
        const float *cres = dv.cscore + ((size_t)u * 2 + 1) * G * dv.c_max;
        const int ncl = dv.residual ? cB - cA : 0, nsub = dv.residual ? iB - iA : 0;
        float M[GT], racc[GT][4], rl[GT];
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            M[g] = -INFINITY;
            rl[g] = 0.f;
            racc[g][0] = racc[g][1] = racc[g][2] = racc[g][3] = 0.f;
        }
        for (int e = warp; e < ncl + nsub; e += AT_WARPS) {
            uint32_t need;
            const float *ex;
            size_t stride;
            const float *vbar;
            if (e < ncl) {
                const int c = cA + e;
                need = dv.cl_n[(size_t)u * dv.c_max + c] > 0
                           ? (allm & ~__ldcg(dv.cselmask + (size_t)u * dv.c_max + c)) : 0u;
                ex = cres + c;
                stride = dv.c_max;
                vbar = dv.cl_vbar + ((size_t)u * dv.c_max + c) * MOG_D;
            } else {
                const int it = iA + (e - ncl), jj = it / L, l = it % L;
                need = dv.subres[((size_t)u * MOG_MAX_UNION + jj) * MOG_MAX_L + l];
                ex = dv.subscore + (((size_t)u * MOG_MAX_UNION + jj) * G) * MOG_MAX_L + l;
                stride = MOG_MAX_L;
                vbar = dv.sub_vbar + ((size_t)u * dv.c_max * dv.l_max + (size_t)sucl[jj] * L + l) * MOG_D;
            }
            const float4 v = *reinterpret_cast<const float4 *>(vbar + lane * 4);
            float exv[GT];
#pragma unroll
            for (int g = 0; g < GT; ++g) exv[g] = (g < G && ((need >> g) & 1u)) ? ex[g * stride] * LOG2E : -INFINITY;
#pragma unroll
            for (int g = 0; g < GT; ++g) {
                if (exv[g] == -INFINITY) continue;
                if (exv[g] > M[g]) {
                    const float sc = exp2f(M[g] - exv[g]);
                    rl[g] *= sc;
                    racc[g][0] *= sc;
                    racc[g][1] *= sc;
                    racc[g][2] *= sc;
                    racc[g][3] *= sc;
                    M[g] = exv[g];
                }
                const float wgt = exp2f(exv[g] - M[g]);
                rl[g] += wgt;
                racc[g][0] += wgt * v.x;
                racc[g][1] += wgt * v.y;
                racc[g][2] += wgt * v.z;
                racc[g][3] += wgt * v.w;
            }
        }
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            if (g >= G) break;
            float *r = stB + ((size_t)warp * G + g) * PART_W;
            if (lane == 0) {
                r[0] = M[g];
                r[1] = rl[g];
            }
            *reinterpret_cast<float4 *>(r + PART_ACC + lane * 4) =
                make_float4(racc[g][0], racc[g][1], racc[g][2], racc[g][3]);
        }
    }
    // ---------------------------- exact rows, tile pipeline ----------------------------
    while (sbase < r1) {
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
        if (sbase < r1) {
            resolve();
            prologue();
        }
    }
    warp_state_out(acc, stA, G);
    __syncthreads();
    float *part = dv.partials + ((size_t)u * MAX_SPLITS + p) * G * PART_W;
    merge_states(stA, 2 * AT_WARPS, G, part);  // stA and stB are contiguous
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
    merge_global_out(dv.partials + (size_t)u * MAX_SPLITS * G * PART_W, P, G,
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
static size_t score_smem(const Dev &dv) {
    return sizeof(float) * ((size_t)dv.G * 2 * MOG_D + (size_t)dv.G * SC_SLICE) +
           (sizeof(float) + sizeof(int)) * 8 * (size_t)dv.P1 * (size_t)max(dv.tc, 1);
}
static size_t sub_smem(const Dev &dv) {
    return sizeof(float) * ((size_t)dv.G * 2 * MOG_D + 2 * (size_t)dv.G * MOG_MAX_L);
}

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
static cudaError_t launch_attend(const DecArgs &a, cudaStream_t s) {
    const size_t sm = AT_SMEM + sizeof(float) * AT_WARPS * a.dv.G * PART_W;
    cudaError_t e = ensure_smem((const void *)k_dec_attend<GT>, sm);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_dec_attend<GT>, dim3(a.dv.P, a.dv.units), dim3(AT_THREADS), sm, s, a);
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
    cudaError_t e;
    const size_t ss = score_smem(dv);
    if ((e = ensure_smem((const void *)k_dec_score, ss)) != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[0], s)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_dec_score, dim3(dv.P1, dv.units), dim3(SC_THREADS), ss, s, a)) != cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[1], s)) != cudaSuccess) return e;
    if (dv.tc > 0) {
        if ((e = launch_pdl(k_dec_sub, dim3(min(dv.c_max, dv.G * dv.tc), dv.units), dim3(SUB_THREADS), sub_smem(dv), s,
                            a)) != cudaSuccess)
            return e;
    }
    if (events && (e = cudaEventRecord(events[2], s)) != cudaSuccess) return e;
    const int G = dv.G;
    if (G <= 1) e = launch_attend<1>(a, s);
    else if (G <= 2) e = launch_attend<2>(a, s);
    else if (G <= 4) e = launch_attend<4>(a, s);
    else if (G <= 8) e = launch_attend<8>(a, s);
    else e = launch_attend<16>(a, s);
    if (e != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[3], s)) != cudaSuccess) return e;
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
