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
// One kernel per decode step: a thread-block cluster of CS CTAs per KV head ("unit"),
// all hand-offs in distributed shared memory behind cluster barriers:
//  P1  CTA k scores its slice of clusters for the G query heads of the unit,
//      s = ln n + tau q.mu + tau^2/2 sum_j q_j^2 var_j, and keeps its slice's top-tc per head;
//  P2  every CTA reads all slices' candidates, derives each head's top-tc clusters (score
//      descending, index ascending) and their union over the heads (ascending index);
//  P3  CTA k takes union slots k, k+CS, ...: subcluster scores, top-ts per head that chose
//      the cluster, the member rows of the chosen subclusters (written to a row list), and
//      the Gaussian residual of the unselected subclusters and of its own slice clusters;
//  P4  the unit's exact rows (anchors, then the slots' rows) are split evenly over the CS
//      CTAs and attended (mma.sync engine), giving one partial (max, sum, acc) per CTA;
//  P5  CTA k merges a slice of the output over all partials and normalises once.
#include <cooperative_groups.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

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

constexpr int RCH = 64;  // slice clusters staged per residual pass
constexpr int PCH = 64;  // (slot, subcluster) pairs staged per residual pass
// dynamic shared memory of the decode kernel: the 227 KB block limit less its static arrays
constexpr int MD_SMEM_MAX = 226 * 1024;

__host__ __device__ constexpr int md_warps(int GT) { return GT <= 4 ? 12 : 8; }

// Shared-memory layout of the decode kernel (byte offsets).
struct MdLay {
    int CS, SL, KC, NSLOT, SPC, warps;  // KC: candidates per slice and head
    int cand_s, cand_i, pub_cnt, pub_coff;                 // read by other CTAs
    int w, csl, crs, cnn, allc_s, allc_i, selc, bm, ucl;  // local
    int sres, ssl, snn, sso, spref, smask, shm, slm, slp, rst, area;
    int total;
};

// area: the staged value means and the residual warp states of P3.
__host__ __device__ inline MdLay md_layout(int G, int tc, int c_max, int CS, int warps) {
    MdLay m;
    int o = 0;
    auto take = [&](int bytes, int align) {
        o = (o + align - 1) & ~(align - 1);
        const int r = o;
        o += bytes;
        return r;
    };
    const int tcc = tc > 0 ? tc : 1;
    m.CS = CS;
    m.warps = warps;
    m.SL = (c_max + CS - 1) / CS;
    m.KC = m.SL < tcc ? m.SL : tcc;
    m.NSLOT = tc > 0 ? (c_max < G * tc ? c_max : G * tc) : 1;
    m.SPC = (m.NSLOT + CS - 1) / CS;
    m.cand_s = take(4 * G * m.KC, 16);
    m.cand_i = take(4 * G * m.KC, 16);
    m.pub_cnt = take(4 * m.SPC, 16);
    m.pub_coff = take(4 * m.SPC, 16);
    m.w = take(16 * 64 * G, 16);
    m.csl = take(4 * G * m.SL, 16);
    m.crs = take(4 * G * m.SL, 16);
    m.cnn = take(4 * m.SL, 16);
    m.allc_s = take(4 * CS * G * m.KC, 16);
    m.allc_i = take(4 * CS * G * m.KC, 16);
    m.selc = take(4 * G * tcc, 16);
    m.bm = take(4 * ((c_max + 31) / 32), 16);
    m.ucl = take(4 * m.NSLOT, 16);
    m.sres = take(4 * m.SPC * G * MOG_MAX_L, 16);
    m.ssl = take(4 * m.SPC * G * MOG_MAX_L, 16);
    m.snn = take(4 * m.SPC * MOG_MAX_L, 16);
    m.sso = take(4 * m.SPC * (MOG_MAX_L + 1), 16);
    m.spref = take(4 * m.SPC * (MOG_MAX_L + 1), 16);
    m.smask = take(4 * m.SPC * MOG_MAX_L, 16);
    m.shm = take(4 * m.SPC, 16);
    m.slm = take(4 * m.SL, 16);
    m.slp = take(4 * (m.SPC + 1), 16);
    m.rst = take(4 * G * PART_W, 16);
    m.area = take((PCH + RCH) * MOG_D * 4 + warps * G * PART_W * 4, 128);
    m.total = (o + 15) & ~15;
    return m;
}

// The last j in [0, n) with a[j] <= x, for a non-decreasing a with a[0] <= x.
__device__ __forceinline__ int last_le(const int *a, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int GT>
__global__ void __launch_bounds__(md_warps(GT) * 32, 1) k_mog_decode(DecArgs a, MdLay m) {
    namespace cg = cooperative_groups;
    constexpr int W = md_warps(GT), NT = W * 32;
    extern __shared__ __align__(128) uint8_t sm[];
    cg::cluster_group cluster = cg::this_cluster();
    const Dev &dv = a.dv;
    const int G = dv.G, tc = dv.tc, ts = dv.ts, tcc = max(tc, 1);
    const int CS = m.CS, k = (int)cluster.block_rank();
    const int u = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *cand_s = reinterpret_cast<float *>(sm + m.cand_s);
    int *cand_i = reinterpret_cast<int *>(sm + m.cand_i);
    int *pub_cnt = reinterpret_cast<int *>(sm + m.pub_cnt);
    int *pub_coff = reinterpret_cast<int *>(sm + m.pub_coff);
    float4 *w = reinterpret_cast<float4 *>(sm + m.w);
    float *csl = reinterpret_cast<float *>(sm + m.csl);
    float *crs = reinterpret_cast<float *>(sm + m.crs);
    int *cnn = reinterpret_cast<int *>(sm + m.cnn);
    float *allc_s = reinterpret_cast<float *>(sm + m.allc_s);
    int *allc_i = reinterpret_cast<int *>(sm + m.allc_i);
    int *selc = reinterpret_cast<int *>(sm + m.selc);
    uint32_t *bm = reinterpret_cast<uint32_t *>(sm + m.bm);
    int *ucl = reinterpret_cast<int *>(sm + m.ucl);
    float *sres = reinterpret_cast<float *>(sm + m.sres);
    float *ssl = reinterpret_cast<float *>(sm + m.ssl);
    int *snn = reinterpret_cast<int *>(sm + m.snn);
    int *sso = reinterpret_cast<int *>(sm + m.sso);
    int *spref = reinterpret_cast<int *>(sm + m.spref);
    uint32_t *smask = reinterpret_cast<uint32_t *>(sm + m.smask);
    uint32_t *shm = reinterpret_cast<uint32_t *>(sm + m.shm);  // heads that chose slot s
    uint32_t *slm = reinterpret_cast<uint32_t *>(sm + m.slm);  // heads that chose slice cluster
    int *slp = reinterpret_cast<int *>(sm + m.slp);            // row prefix over this CTA's slots
    float *rst = reinterpret_cast<float *>(sm + m.rst);
    uint8_t *area = sm + m.area;
    __shared__ int s_wsum[W], s_uc;

    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int b = ui[UI_B], h = u % dv.h_kv, C = ui[UI_C], L = ui[UI_L];
    const int S = ui[UI_S], rlo = ui[UI_RLO];
    const int nnow = dv.n_now[b];
    const int s_cnt = min(S, nnow), n_anchor = s_cnt + max(0, nnow - rlo);
    const uint32_t allm = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    const size_t ug = (size_t)u * dv.c_max;               // cluster index base
    const size_t usg = (size_t)u * dv.c_max * dv.l_max;   // subcluster index base
    const uint16_t *qg = a.q + (size_t)u * G * MOG_D;
    int *selu = dv.sel + (size_t)u * G * a.SW;
    const bool resid = dv.residual != 0;

    // ------------------------------------------------------------ P0: query, weights
    uint32_t qa[8][4];
    load_q_frags(qa, qg, G);
    load_weights(w, qg, G, dv.tau);
    pdl_wait();
    pdl_trigger();
    __syncthreads();

    // ------------------------------------------------- P1: score this CTA's clusters
    const int c0 = k * m.SL;
    const int ns = max(0, min(C - c0, m.SL));
    for (int base = 0; base < ns; base += NT / 4) {
        const int cl = base + (tid >> 2);
        const bool valid = cl < ns;
        const int c = c0 + (valid ? cl : 0);
        const int n = valid ? dv.cl_n[ug + c] : 0;
        float res[GT], sl[GT];
        quad_scores<GT>(dv.cl_ms + (ug + c) * 2 * MOG_D, n, valid, w, G, dv.score_mode, res, sl);
        if (valid && (tid & 3) == 0) {
#pragma unroll
            for (int g = 0; g < GT; ++g)
                if (g < G) {
                    csl[g * m.SL + cl] = sl[g];
                    crs[g * m.SL + cl] = res[g];
                }
            cnn[cl] = n;
        }
    }
    __syncthreads();
    const int KC = m.KC;
    if (tc > 0) {  // this slice's top-KC per head (KC = min(slice, tc)), sorted, -1 padded
        const int span = max(ns, KC);
        for (int e = tid; e < G * span; e += NT) {
            const int g = e / span, i = e % span;
            if (i < ns) {
                const float v = csl[g * m.SL + i];
                int rank = 0;
                for (int kk = 0; kk < ns; ++kk) rank += ranks_before(csl[g * m.SL + kk], kk, v, i);
                if (rank < KC) {
                    cand_s[g * KC + rank] = v;
                    cand_i[g * KC + rank] = v == -INFINITY ? -1 : c0 + i;
                }
            } else {
                cand_s[g * KC + i] = -INFINITY;
                cand_i[g * KC + i] = -1;
            }
        }
    }
    for (int e = tid; e < G * tcc; e += NT) selc[e] = -1;
    for (int e = tid; e < (dv.c_max + 31) / 32; e += NT) bm[e] = 0u;
    for (int e = tid; e < m.SL; e += NT) slm[e] = 0u;
    cluster.sync();  // S1: candidates of every slice are published

    // ------------------------------------------------------- P2: selection and union
    if (tc > 0) {
        if (a.sel_in) {
            for (int e = tid; e < G * tc; e += NT) {
                const int g = e / tc, r = e % tc;
                const int cc = a.sel_in[((size_t)u * G + g) * a.SW + r];
                selc[e] = (cc >= 0 && cc < C && dv.cl_n[ug + cc] > 0) ? cc : -1;
            }
        } else {
            for (int e = tid; e < CS * G * KC; e += NT) {  // gather [g][src][r]
                const int src = e / (G * KC), rem = e % (G * KC), g = rem / KC, r = rem % KC;
                allc_s[(g * CS + src) * KC + r] = cluster.map_shared_rank(cand_s, src)[rem];
                allc_i[(g * CS + src) * KC + r] = cluster.map_shared_rank(cand_i, src)[rem];
            }
            __syncthreads();
            // element (g, list p, position r): rank over all lists of head g = r plus, for
            // every other list, the length of its prefix that ranks before the element
            for (int e = tid; e < G * CS * KC; e += NT) {
                const int g = e / (CS * KC), pr = e % (CS * KC), pl = pr / KC, r = pr % KC;
                const float *cs = allc_s + (size_t)g * CS * KC;
                const int *ci = allc_i + (size_t)g * CS * KC;
                const int x = ci[pr];
                if (x < 0) continue;
                const float v = cs[pr];
                int rank = r;
                for (int q = 0; q < CS && rank < tc; ++q) {
                    if (q == pl) continue;
                    int lo = 0, hi = KC;
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        const int xm = ci[q * KC + mid];
                        if (xm >= 0 && ranks_before(cs[q * KC + mid], xm, v, x)) lo = mid + 1;
                        else hi = mid;
                    }
                    rank += lo;
                }
                if (rank < tc) selc[g * tc + rank] = x;
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < G * tc; e += NT) {
        const int c = selc[e];
        if (c < 0) continue;
        atomicOr(&bm[c >> 5], 1u << (c & 31));
        if (c >= c0 && c < c0 + ns) atomicOr(&slm[c - c0], 1u << (e / tc));
    }
    __syncthreads();
    {  // union = set bits of bm, ascending: ucl[0 .. Uc)
        const int nw = (dv.c_max + 31) / 32;
        const int per = (nw + NT - 1) / NT;
        const int w0 = tid * per, w1 = min(nw, w0 + per);
        int cnt = 0;
        for (int i = w0; i < w1; ++i) cnt += __popc(bm[i]);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int base = incl - cnt;
        for (int kk = 0; kk < warp; ++kk) base += s_wsum[kk];
        if (tid == NT - 1) s_uc = base + cnt;
        for (int i = w0; i < w1; ++i) {
            uint32_t bits = bm[i];
            while (bits) {
                const int bit = __ffs(bits) - 1;
                bits &= bits - 1;
                ucl[base++] = i * 32 + bit;
            }
        }
    }
    __syncthreads();
    const int Uc = s_uc;
    if (k == 0) {  // the cluster part of the exported selection
        for (int e = tid; e < G * tc; e += NT) {
            const int g = e / tc, r = e % tc;
            selu[(size_t)g * a.SW + r] = selc[e];
            if (selc[e] < 0)
                for (int kk = 0; kk < ts; ++kk) selu[(size_t)g * a.SW + tc + r * ts + kk] = -1;
        }
    }

    // ----------------------------------------- P3: this CTA's union slots, residual
    const int nmy = Uc > k ? (Uc - k + CS - 1) / CS : 0;  // slots k, k+CS, ...
    const int npair = nmy * L;                              // (slot, subcluster) pairs
    float *vst = reinterpret_cast<float *>(area);           // [PCH][d] subcluster means
    float *vcl = vst + (size_t)PCH * MOG_D;                 // [RCH][d] slice cluster means
    float *rws = vcl + (size_t)RCH * MOG_D;                 // [W][G][PART_W] residual states
    for (int e = tid; e < nmy * (L + 1); e += NT) {
        const int s = e / (L + 1), i = e % (L + 1);
        const int c = ucl[k + s * CS];
        sso[s * (MOG_MAX_L + 1) + i] = dv.sub_off[(size_t)u * dv.sub_off_stride + (size_t)c * L + i];
        if (i < L) snn[s * MOG_MAX_L + i] = dv.sub_n[usg + (size_t)c * L + i];
    }
    auto stage_pairs = [&](int p0) {  // value means of pairs p0 .. p0 + PCH
        const int cnt = min(PCH, npair - p0);
        for (int e = tid; e < cnt * 32; e += NT) {
            const int pr = p0 + e / 32, s = pr / L, l = pr % L;
            cp_async16(smem_u32(vst + (size_t)(e / 32) * MOG_D + 4 * (e % 32)),
                       dv.sub_vbar + (usg + (size_t)ucl[k + s * CS] * L + l) * MOG_D + 4 * (e % 32), 16);
        }
    };
    if (resid && npair > 0) stage_pairs(0);
    auto stage_slice = [&](int k0) {
        const int cnt = min(RCH, ns - k0);
        for (int e = tid; e < cnt * 32; e += NT)
            cp_async16(smem_u32(vcl + (size_t)(e / 32) * MOG_D + 4 * (e % 32)),
                       dv.cl_vbar + (ug + c0 + k0 + e / 32) * MOG_D + 4 * (e % 32), 16);
    };
    if (resid && ns > 0) stage_slice(0);
    cp_async_commit();
    for (int base = 0; base < npair; base += NT / 4) {  // subcluster scores, 4 lanes a pair
        const int pr = base + (tid >> 2);
        const bool valid = pr < npair;
        const int s = valid ? pr / L : 0, l = valid ? pr % L : 0;
        const size_t gi = usg + (valid ? (size_t)ucl[k + s * CS] * L + l : 0);
        float res[GT], sl[GT];
        quad_scores<GT>(dv.sub_ms + gi * 2 * MOG_D, valid ? dv.sub_n[gi] : 0, valid, w, G,
                        dv.score_mode, res, sl);
        if (valid && (tid & 3) == 0) {
#pragma unroll
            for (int g = 0; g < GT; ++g)
                if (g < G) {
                    sres[(s * G + g) * MOG_MAX_L + l] = res[g];
                    ssl[(s * G + g) * MOG_MAX_L + l] = sl[g];
                }
        }
    }
    for (int e = tid; e < nmy * MOG_MAX_L; e += NT) smask[e] = 0u;
    for (int e = tid; e < nmy; e += NT) shm[e] = 0u;
    __syncthreads();
    // top-ts subclusters of every head that chose a slot's cluster
    for (int e = warp; e < nmy * G; e += W) {
        const int s = e / G, g = e % G;
        const int c = ucl[k + s * CS];
        int rk = -1;
        for (int r = 0; r < tc; ++r)
            if (selc[g * tc + r] == c) { rk = r; break; }
        if (rk < 0) continue;
        if (lane == 0) atomicOr(&shm[s], 1u << g);
        int *subs = selu + (size_t)g * a.SW + tc + (size_t)rk * ts;
        const int *nn = snn + s * MOG_MAX_L;
        if (a.sel_in) {
            const int32_t *si = a.sel_in + ((size_t)u * G + g) * a.SW + tc + (size_t)rk * ts;
            for (int r = lane; r < ts; r += 32) {
                const int l2 = si[r];
                const bool ok = l2 >= 0 && l2 < L && nn[l2] > 0;
                subs[r] = ok ? l2 : -1;
                if (ok) atomicOr(&smask[s * MOG_MAX_L + l2], 1u << g);
            }
        } else {
            for (int r = lane; r < ts; r += 32) subs[r] = -1;
            __syncwarp();
            const float *sc = ssl + (s * G + g) * MOG_MAX_L;
            const float v = lane < L ? sc[lane] : -INFINITY;
            int rank = 0;
            for (int kk = 0; kk < L; ++kk) rank += ranks_before(sc[kk], kk, v, lane);
            if (lane < L && v != -INFINITY && rank < ts) {
                subs[rank] = lane;
                atomicOr(&smask[s * MOG_MAX_L + lane], 1u << g);
            }
        }
    }
    __syncthreads();
    for (int s = warp; s < nmy; s += W) {  // prefix of the chosen subclusters' sizes
        const int *so = sso + s * (MOG_MAX_L + 1);
        const int cnt = lane < L && smask[s * MOG_MAX_L + lane] ? so[lane + 1] - so[lane] : 0;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane < L) spref[s * (MOG_MAX_L + 1) + lane + 1] = incl;
        if (lane == 0) {
            spref[s * (MOG_MAX_L + 1)] = 0;
            pub_coff[s] = so[0];
        }
        if (lane == L - 1) pub_cnt[s] = incl;
    }
    __syncthreads();
    if (warp == 0) {  // row prefix over this CTA's slots
        int run = 0;
        for (int s0 = 0; s0 < nmy; s0 += 32) {
            const int s = s0 + lane;
            const int cnt = s < nmy ? spref[s * (MOG_MAX_L + 1) + L] : 0;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (s < nmy) slp[s] = run + incl - cnt;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) slp[nmy] = run;
    }
    __syncthreads();
    {  // member rows of the chosen subclusters -> the unit's row list (perm order); four
       // independent perm loads in flight per thread
        const int *perm = dv.perm + (size_t)u * dv.n_cap;
        int *rowpos = dv.rowpos + (size_t)u * dv.n_cap;
        uint32_t *rowmask = dv.rowmask + (size_t)u * dv.n_cap;
        const int tot = slp[nmy];
        for (int i0 = tid; i0 < tot; i0 += 4 * NT) {
            int src[4], dst[4];
            uint32_t mk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * NT;
                src[j] = -1;
                if (i < tot) {
                    const int s = last_le(slp, nmy, i);
                    const int ii = i - slp[s];
                    const int *sp = spref + s * (MOG_MAX_L + 1);
                    const int kk = last_le(sp, L, ii);
                    const int *so = sso + s * (MOG_MAX_L + 1);
                    src[j] = so[kk] + (ii - sp[kk]);
                    dst[j] = so[0] + ii;
                    mk[j] = smask[s * MOG_MAX_L + kk];
                }
            }
            int pv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) pv[j] = src[j] >= 0 ? __ldg(perm + src[j]) : 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (src[j] >= 0) {
                    rowpos[dst[j]] = pv[j];
                    rowmask[dst[j]] = mk[j];
                }
        }
    }
    // Gaussian residual: warps take items (pairs, then slice clusters) round-robin; lane
    // owns dims 4*lane..+3; per-warp states are merged into rst
    {
        OnlineAcc st[GT];
#pragma unroll
        for (int g = 0; g < GT; ++g) st[g].init();
        if (resid) {
            cp_async_wait<0>();
            __syncthreads();
            for (int p0 = 0; p0 < npair; p0 += PCH) {
                if (p0 > 0) {  // further pairs (many slots per CTA)
                    __syncthreads();
                    stage_pairs(p0);
                    cp_async_commit();
                    cp_async_wait<0>();
                    __syncthreads();
                }
                const int cnt = min(PCH, npair - p0);
                for (int e = warp; e < cnt; e += W) {
                    const int s = (p0 + e) / L, l = (p0 + e) % L;
                    if (snn[s * MOG_MAX_L + l] <= 0) continue;
                    const uint32_t need = shm[s] & ~smask[s * MOG_MAX_L + l];
                    const float *vrow = vst + (size_t)e * MOG_D + 4 * lane;
#pragma unroll
                    for (int g = 0; g < GT; ++g)
                        if (g < G && ((need >> g) & 1u))
                            st[g].absorb(sres[(s * G + g) * MOG_MAX_L + l] * LOG2E, vrow);
                }
            }
            for (int k0 = 0; k0 < ns; k0 += RCH) {
                if (k0 > 0) {
                    __syncthreads();
                    stage_slice(k0);
                    cp_async_commit();
                    cp_async_wait<0>();
                    __syncthreads();
                }
                const int cnt = min(RCH, ns - k0);
                for (int e = warp; e < cnt; e += W) {
                    const int cl = k0 + e;
                    if (cnn[cl] <= 0) continue;
                    const uint32_t need = allm & ~slm[cl];
                    const float *vrow = vcl + (size_t)e * MOG_D + 4 * lane;
#pragma unroll
                    for (int g = 0; g < GT; ++g)
                        if (g < G && ((need >> g) & 1u)) st[g].absorb(crs[g * m.SL + cl] * LOG2E, vrow);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            if (g >= G) break;
            float *o = rws + ((size_t)warp * G + g) * PART_W;
            if (lane == 0) {
                o[0] = st[g].m;
                o[1] = st[g].l;
            }
            *reinterpret_cast<float4 *>(o + PART_ACC + 4 * lane) = st[g].a;
        }
        __syncthreads();
        merge_states(rws, W, G, rst);
    }
    cp_async_wait<0>();
    cluster.sync();  // S2: row lists (global) and their counts (shared) are published
    // ------------------------- P4: the unit's row plan for the rows kernel (CTA 0)
    for (int g = k; g < G; g += CS) {  // the unit's residual: CS states merged per head
        if (tid >= MOG_D) break;
        float mx = -INFINITY;
        for (int i = 0; i < CS; ++i) mx = fmaxf(mx, cluster.map_shared_rank(rst, i)[g * PART_W]);
        float l = 0.f, acc = 0.f;
        if (mx != -INFINITY)
            for (int i = 0; i < CS; ++i) {
                const float *r = cluster.map_shared_rank(rst, i) + g * PART_W;
                const float mi = r[0];
                if (mi == -INFINITY) continue;
                const float sc = exp2f(mi - mx);
                l += sc * r[1];
                acc += sc * r[PART_ACC + tid];
            }
        float *o = dv.partials + (((size_t)u * PART_SLOTS + MAX_SPLITS) * G + g) * PART_W;
        if (tid == 0) {
            o[0] = mx;
            o[1] = l;
        }
        o[PART_ACC + tid] = acc;
    }
    if (k == 0 && warp == W - 1) {
        int *plan = dv.slotcnt + (size_t)u * PLAN_W;  // [8 | pre[0..Uc] | coff[0..Uc)]
        int run = n_anchor;
        for (int j0 = 0; j0 < Uc; j0 += 32) {
            const int j = j0 + lane;
            int cnt = 0, coff = 0;
            if (j < Uc) {
                const int own = j % CS, s = j / CS;
                cnt = cluster.map_shared_rank(pub_cnt, own)[s];
                coff = cluster.map_shared_rank(pub_coff, own)[s];
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (j < Uc) {
                plan[PLAN_PRE + j] = run + incl - cnt;
                plan[PLAN_COFF + j] = coff;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            plan[0] = Uc;
            plan[1] = run;  // T: anchors + selected rows
            plan[2] = n_anchor;
            plan[3] = s_cnt;
            plan[4] = rlo;
            plan[PLAN_PRE + Uc] = run;
        }
    }
    cluster.sync();  // S3: the owners' counts and residual states have been read
}


constexpr int RW_SUPER = 256;                  // row positions per batch in the rows kernel
constexpr int RW_TPB = RW_SUPER / AT_ROWS;     // tiles per batch
constexpr int RW_PER = RW_SUPER / AT_THREADS;  // positions a thread fetches per batch
static_assert(RW_TPB >= AT_STAGES - 1, "the first batch must cover the pipeline's prologue");

// Kernel B: grid (P, units), 4 warps, two CTAs per SM.  Rows [p*T/P, (p+1)*T/P) of the
// unit's exact list (anchors, then the union slots' rows in slot order) through the
// 64-row tile engine.  Positions are fetched into registers one batch ahead and moved to
// shared memory when the pipeline reaches the batch, so no tile copy waits on a position
// load.  One unnormalised partial per CTA.
template <int GT>
__global__ void __launch_bounds__(AT_THREADS) k_mog_rows(DecArgs a) {
    extern __shared__ __align__(128) uint8_t tile[];
    const Dev &dv = a.dv;
    const int G = dv.G;
    __shared__ __align__(16) int s_plan[PLAN_W];
    __shared__ int s_pos[2][RW_SUPER];
    __shared__ uint32_t s_mk[2][RW_SUPER];
    const int u = blockIdx.y, p = blockIdx.x, P = gridDim.x;
    const int tid = threadIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int b = ui[UI_B], h = u % dv.h_kv;
    const uint32_t allm = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    uint32_t qa[8][4];
    load_q_frags(qa, a.q + (size_t)u * G * MOG_D, G);
    pdl_wait();  // the selection kernel's row lists and plan
    pdl_trigger();
    {
        const int *plan = dv.slotcnt + (size_t)u * PLAN_W;
        for (int q = tid; q < PLAN_W / 4; q += AT_THREADS) cp_async16(smem_u32(s_plan + 4 * q), plan + 4 * q, 16);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
    }
    const int Uc = s_plan[0], T = s_plan[1], n_anchor = s_plan[2], s_cnt = s_plan[3], rlo = s_plan[4];
    const int *s_pre = s_plan + PLAN_PRE, *s_coff = s_plan + PLAN_COFF;
    const int r0 = (int)((int64_t)T * p / P), r1 = (int)((int64_t)T * (p + 1) / P);
    const int nrow = r1 - r0, nt = (nrow + AT_ROWS - 1) / AT_ROWS;
    const uint16_t *kb = dv.K + b * dv.sb + h * dv.sh;
    const uint16_t *vb = dv.V + b * dv.sb + h * dv.sh;
    const int *rowpos = dv.rowpos + (size_t)u * dv.n_cap;
    const uint32_t *rowmask = dv.rowmask + (size_t)u * dv.n_cap;
    int pf_pos[RW_PER];
    uint32_t pf_mk[RW_PER];
    auto fetch = [&](int bt) {  // positions of batch bt into registers
#pragma unroll
        for (int jj = 0; jj < RW_PER; ++jj) {
            const int i = r0 + bt * RW_SUPER + tid + jj * AT_THREADS;
            int pp = 0;
            uint32_t mm = 0u;
            if (i < r1) {
                if (i < n_anchor) {
                    pp = i < s_cnt ? i : rlo + (i - s_cnt);
                    mm = allm;
                } else {
                    const int sl = last_le(s_pre, Uc, i);  // the slot holding row i
                    const int kk = s_coff[sl] + (i - s_pre[sl]);
                    pp = __ldcg(rowpos + kk);
                    mm = __ldcg(rowmask + kk);
                }
            }
            pf_pos[jj] = pp;
            pf_mk[jj] = mm;
        }
    };
    auto place = [&](int bt) {  // registers -> shared buffer of batch bt
#pragma unroll
        for (int jj = 0; jj < RW_PER; ++jj) {
            s_pos[bt & 1][tid + jj * AT_THREADS] = pf_pos[jj];
            s_mk[bt & 1][tid + jj * AT_THREADS] = pf_mk[jj];
        }
    };
    auto issue = [&](int t) {
        const int buf = (t / RW_TPB) & 1, rb = (t % RW_TPB) * AT_ROWS;
        issue_tile(tile + (t % AT_STAGES) * AT_STAGE_BYTES, min(AT_ROWS, nrow - t * AT_ROWS), kb, vb,
                   dv.sn, [&](int r, int64_t &pos, uint32_t &mk) {
                       int pp = s_pos[buf][rb + r];
                       uint32_t mm = s_mk[buf][rb + r];
                       if ((unsigned)pp >= (unsigned)dv.n_cap) {  // corrupt partition: flag, skip
                           flag_error(dv.status, ST_BAD_INDEX);
                           pp = 0;
                           mm = 0u;
                       }
                       pos = pp;
                       mk = mm;
                   });
    };
    WarpAcc acc;
    acc.init();
    const float scale2 = dv.tau * LOG2E;
    if (nt > 0) {
        fetch(0);
        place(0);
        if (nrow > RW_SUPER) fetch(1);
    }
    __syncthreads();
#pragma unroll
    for (int s2 = 0; s2 < AT_STAGES - 1; ++s2) {
        if (s2 < nt) issue(s2);
        cp_async_commit();
    }
    for (int t = 0; t < nt; ++t) {
        cp_async_wait<AT_STAGES - 2>();
        __syncthreads();
        const int ti = t + AT_STAGES - 1;
        if (ti < nt) {
            if (ti % RW_TPB == 0) {  // first tile of a batch: its positions go to shared memory
                const int bt = ti / RW_TPB;
                place(bt);
                __syncthreads();
                if ((bt + 1) * RW_SUPER < nrow) fetch(bt + 1);
            }
            issue(ti);
        }
        cp_async_commit();
        compute_tile(acc, qa, tile + (t % AT_STAGES) * AT_STAGE_BYTES, scale2);
    }
    cp_async_wait<0>();
    __syncthreads();
    float *st = reinterpret_cast<float *>(tile);
    warp_state_out(acc, st, G);
    __syncthreads();
    merge_states(st, AT_WARPS, G, dv.partials + ((size_t)u * PART_SLOTS + p) * G * PART_W);
}

// Kernel C: grid (G, units), 512 threads.  Merges the P row partials and the residual
// partial of one query head (running max, rescaled sums) and normalises once.  Thread
// (part, j) sums partials part, part + 4, ... for dimension j; all loads are independent.
constexpr int MG_THREADS = 4 * MOG_D;
__global__ void __launch_bounds__(MG_THREADS) k_mog_merge(const float *partials, int P, int G,
                                                          float *out) {
    const int g = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
    const int j = tid % MOG_D, part = tid / MOG_D;
    __shared__ float s_m[MAX_SPLITS + 1], s_l[MAX_SPLITS + 1], s_w[MAX_SPLITS + 1];
    __shared__ float s_acc[MG_THREADS / MOG_D][MOG_D];
    pdl_wait();
    pdl_trigger();
    const int n = P + 1;  // row partials, then the residual
    auto src = [&](int i) {
        return partials + (((size_t)u * PART_SLOTS + (i < P ? i : MAX_SPLITS)) * G + g) * PART_W;
    };
    if (tid < n) {
        s_m[tid] = __ldcg(src(tid));
        s_l[tid] = __ldcg(src(tid) + 1);
    }
    __syncthreads();
    float mx = -INFINITY;
    for (int i = 0; i < n; ++i) mx = fmaxf(mx, s_m[i]);
    if (tid < n) s_w[tid] = (s_m[tid] == -INFINITY) ? 0.f : exp2f(s_m[tid] - mx);
    __syncthreads();
    float l = 0.f;
    for (int i = 0; i < n; ++i) l += s_w[i] * s_l[i];
    float v = 0.f;
#pragma unroll 4
    for (int i = part; i < n; i += MG_THREADS / MOG_D) v += s_w[i] * __ldcg(src(i) + PART_ACC + j);
    s_acc[part][j] = v;
    __syncthreads();
    if (part == 0) {
        for (int q = 1; q < MG_THREADS / MOG_D; ++q) v += s_acc[q][j];
        out[((size_t)u * G + g) * MOG_D + j] = l > 0.f ? v / l : 0.f;
    }
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
static cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cs,
                             const DecArgs &a, const MdLay &m) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, a, m);
}

template <typename K, typename... Args>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
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

// Cluster size (CTAs per unit) and pipeline depth for a decode launch: the largest cluster
// (<= 16) such that every unit's cluster is resident at once (the occupancy query decides;
// on a 152-SM GB300 eight 12-CTA clusters of ~200 KB fit, eight 16-CTA clusters do not).
template <int GT>
static cudaError_t pick_shape(const Dev &dv, int *cs_out, MdLay *m_out) {
    const void *fn = (const void *)k_mog_decode<GT>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    const int sms = num_sms();
    for (int cs = 16; cs >= 1; --cs) {  // any size: e.g. 12-CTA clusters fit where 16 do not
        if (cs > 1 && (int64_t)cs * dv.units > 2LL * sms) continue;  // keep clusters resident
        MdLay m = md_layout(dv.G, dv.tc, dv.c_max, cs, md_warps(GT));
        if (m.total > MD_SMEM_MAX) continue;
        if ((e = ensure_smem(fn, (size_t)m.total)) != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs, dv.units);
        cfg.blockDim = dim3(md_warps(GT) * 32);
        cfg.dynamicSmemBytes = m.total;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = cs;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int ncl = 0;
        e = cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg);
        if (e != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (ncl >= dv.units || cs == 1) {
            *cs_out = cs;
            *m_out = m;
            return cudaSuccess;
        }
    }
    return cudaErrorInvalidConfiguration;
}

template <int GT>
static cudaError_t launch_steps(const DecArgs &a, cudaStream_t s, cudaEvent_t const *events) {
    const Dev &dv = a.dv;
    cudaError_t e;
    // the shape depends only on the plan: cache it per (units, G, tc, c_max, l_max)
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int>, std::pair<int, MdLay>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, dv.units, dv.G, dv.tc, dv.c_max, dv.l_max);
    int cs;
    MdLay m;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it == cache.end()) {
            if ((e = pick_shape<GT>(dv, &cs, &m)) != cudaSuccess) return e;
            cache[key] = std::make_pair(cs, m);
        } else {
            cs = it->second.first;
            m = it->second.second;
        }
    }
    if ((e = ensure_smem((const void *)k_mog_decode<GT>, (size_t)m.total)) != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[0], s)) != cudaSuccess) return e;
    if ((e = launch_ex(k_mog_decode<GT>, dim3(cs, dv.units), dim3(md_warps(GT) * 32), m.total, s, cs, a, m)) !=
        cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[1], s)) != cudaSuccess) return e;
    if ((e = ensure_smem((const void *)k_mog_rows<GT>, AT_SMEM)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_mog_rows<GT>, dim3(dv.P, dv.units), dim3(AT_THREADS), AT_SMEM, s, a)) !=
        cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[2], s)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_mog_merge, dim3(dv.G, dv.units), dim3(MG_THREADS), 0, s,
                        (const float *)dv.partials, dv.P, dv.G, a.out)) != cudaSuccess)
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

size_t slot_smem_bytes(int G, int c_max, int tc) {  // the smallest layout (16-CTA clusters)
    return (size_t)md_layout(G, tc, c_max, 16, md_warps(G <= 4 ? 4 : 16)).total;
}

cudaError_t launch_append(const Dev &dv, const Plan &pl, const void *k_new, const void *v_new,
                          cudaStream_t s) {
    k_append<<<pl.batch, 128, 0, s>>>(dv, static_cast<const uint16_t *>(k_new),
                                      static_cast<const uint16_t *>(v_new));
    return cudaGetLastError();
}

}  // namespace mog
