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
constexpr int POSCH = 1024;  // row positions staged per pass of the row phase
// dynamic shared memory of the decode kernel: the 227 KB block limit less its static arrays
constexpr int MD_SMEM_MAX = 226 * 1024;

__host__ __device__ constexpr int md_warps(int GT) { return GT <= 4 ? 12 : 8; }

// Shared-memory layout of the decode kernel (byte offsets).
struct MdLay {
    int CS, SL, KC, NSLOT, SPC, warps, rwarps, nbuf;  // KC: candidates per slice and head;
                                                      // rwarps x nbuf row buffers
    int cand_s, cand_i, pub_cnt, pub_coff, pub_state;                // read by other CTAs
    int w, csl, crs, cnn, allc_s, allc_i, selc, bm, ucl, ucoff, pre;  // local
    int sres, ssl, snn, sso, spref, smask, rst, posb, area;
    int total;
};

// area: the per-warp row buffers in P4; before that the staged value means and the
// residual warp states of P3; after P4 the warp states of the merge.
__host__ __device__ inline MdLay md_layout_rw(int G, int tc, int c_max, int l_max, int CS, int warps,
                                             int rwarps, int nbuf) {
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
    m.rwarps = rwarps;
    m.nbuf = nbuf;
    m.SL = (c_max + CS - 1) / CS;
    m.KC = m.SL < tcc ? m.SL : tcc;
    m.NSLOT = tc > 0 ? (c_max < G * tc ? c_max : G * tc) : 1;
    m.SPC = (m.NSLOT + CS - 1) / CS;
    m.cand_s = take(4 * G * m.KC, 16);
    m.cand_i = take(4 * G * m.KC, 16);
    m.pub_cnt = take(4 * m.SPC, 16);
    m.pub_coff = take(4 * m.SPC, 16);
    m.pub_state = take(4 * G * PART_W, 16);
    m.w = take(16 * 64 * G, 16);
    m.csl = take(4 * G * m.SL, 16);
    m.crs = take(4 * G * m.SL, 16);
    m.cnn = take(4 * m.SL, 16);
    m.allc_s = take(4 * CS * G * m.KC, 16);
    m.allc_i = take(4 * CS * G * m.KC, 16);
    m.selc = take(4 * G * tcc, 16);
    m.bm = take(4 * ((c_max + 31) / 32), 16);
    m.ucl = take(4 * m.NSLOT, 16);
    m.ucoff = take(4 * m.NSLOT, 16);
    m.pre = take(4 * (m.NSLOT + 1), 16);
    m.sres = take(4 * m.SPC * G * MOG_MAX_L, 16);
    m.ssl = take(4 * m.SPC * G * MOG_MAX_L, 16);
    m.snn = take(4 * m.SPC * MOG_MAX_L, 16);
    m.sso = take(4 * m.SPC * (MOG_MAX_L + 1), 16);
    m.spref = take(4 * m.SPC * (MOG_MAX_L + 1), 16);
    m.smask = take(4 * m.SPC * MOG_MAX_L, 16);
    m.rst = take(4 * G * PART_W, 16);
    m.posb = take(2 * 2 * POSCH * 4, 16);  // [2 buffers][pos | mask][POSCH]
    const int rows = rwarps * nbuf * WB_BYTES;
    const int p3 = (PCH + RCH) * MOG_D * 4 + warps * G * PART_W * 4;
    const int mrg = (warps + 1) * G * PART_W * 4;
    int a = rows > p3 ? rows : p3;
    a = a > mrg ? a : mrg;
    m.area = take(a, 128);
    m.total = (o + 15) & ~15;
    return m;
}

// Row pipeline shape: the most 16-row blocks in flight while a block is computed,
// rwarps * (nbuf - 1), over nbuf in {2, 3} and rwarps <= warps, within a CTA's shared memory.
__host__ __device__ inline MdLay md_layout(int G, int tc, int c_max, int l_max, int CS, int warps) {
    MdLay best = md_layout_rw(G, tc, c_max, l_max, CS, warps, 1, 2);
    int score = -1;
    for (int nbuf = 2; nbuf <= 3; ++nbuf)
        for (int rw = warps; rw >= 1; --rw) {
            MdLay m = md_layout_rw(G, tc, c_max, l_max, CS, warps, rw, nbuf);
            if (m.total > MD_SMEM_MAX) continue;
            const int sc = rw * (nbuf - 1) * 64 + rw;  // blocks in flight, then warps
            if (sc > score) {
                score = sc;
                best = m;
            }
            break;
        }
    return best;
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
    float *pub_state = reinterpret_cast<float *>(sm + m.pub_state);
    float4 *w = reinterpret_cast<float4 *>(sm + m.w);
    float *csl = reinterpret_cast<float *>(sm + m.csl);
    float *crs = reinterpret_cast<float *>(sm + m.crs);
    int *cnn = reinterpret_cast<int *>(sm + m.cnn);
    float *allc_s = reinterpret_cast<float *>(sm + m.allc_s);
    int *allc_i = reinterpret_cast<int *>(sm + m.allc_i);
    int *selc = reinterpret_cast<int *>(sm + m.selc);
    uint32_t *bm = reinterpret_cast<uint32_t *>(sm + m.bm);
    int *ucl = reinterpret_cast<int *>(sm + m.ucl);
    int *ucoff = reinterpret_cast<int *>(sm + m.ucoff);
    int *pre = reinterpret_cast<int *>(sm + m.pre);
    float *sres = reinterpret_cast<float *>(sm + m.sres);
    float *ssl = reinterpret_cast<float *>(sm + m.ssl);
    int *snn = reinterpret_cast<int *>(sm + m.snn);
    int *sso = reinterpret_cast<int *>(sm + m.sso);
    int *spref = reinterpret_cast<int *>(sm + m.spref);
    uint32_t *smask = reinterpret_cast<uint32_t *>(sm + m.smask);
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
    for (int e = tid; e < G * tc; e += NT)
        if (selc[e] >= 0) atomicOr(&bm[selc[e] >> 5], 1u << (selc[e] & 31));
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
    __syncthreads();
    // top-ts subclusters of every head that chose a slot's cluster
    for (int e = warp; e < nmy * G; e += W) {
        const int s = e / G, g = e % G;
        const int c = ucl[k + s * CS];
        int rk = -1;
        for (int r = 0; r < tc; ++r)
            if (selc[g * tc + r] == c) { rk = r; break; }
        if (rk < 0) continue;
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
    {  // member rows of the chosen subclusters -> the unit's row list (perm order)
        const int *perm = dv.perm + (size_t)u * dv.n_cap;
        int *rowpos = dv.rowpos + (size_t)u * dv.n_cap;
        uint32_t *rowmask = dv.rowmask + (size_t)u * dv.n_cap;
        for (int s = 0; s < nmy; ++s) {
            const int *sp = spref + s * (MOG_MAX_L + 1);
            const int *so = sso + s * (MOG_MAX_L + 1);
            const int tot = sp[L];
            for (int i = tid; i < tot; i += NT) {
                int kk = 0;
                while (sp[kk + 1] <= i) ++kk;
                rowpos[so[0] + i] = perm[so[kk] + (i - sp[kk])];
                rowmask[so[0] + i] = smask[s * MOG_MAX_L + kk];
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
                    const int c = ucl[k + s * CS];
                    uint32_t hm = 0u;  // heads that chose c
                    for (int q = 0; q < G * tc; ++q)
                        if (selc[q] == c) hm |= 1u << (q / tc);
                    const uint32_t need = hm & ~smask[s * MOG_MAX_L + l];
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
                    uint32_t chose = 0u;
                    for (int q = 0; q < G * tc; ++q)
                        if (selc[q] == c0 + cl) chose |= 1u << (q / tc);
                    const uint32_t need = allm & ~chose;
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

    // -------------------------------------------- P4: exact rows, split evenly
    if (warp == 0) {  // slot prefix from the owners' counts
        int run = n_anchor;
        for (int j0 = 0; j0 < Uc; j0 += 32) {
            const int j = j0 + lane;
            int cnt = 0;
            if (j < Uc) {
                const int own = j % CS, s = j / CS;
                cnt = cluster.map_shared_rank(pub_cnt, own)[s];
                ucoff[j] = cluster.map_shared_rank(pub_coff, own)[s];
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (j < Uc) pre[j] = run + incl - cnt;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) pre[Uc] = run;
    }
    __syncthreads();
    const int T = pre[Uc];
    const int r0 = (int)((int64_t)T * k / CS), r1 = (int)((int64_t)T * (k + 1) / CS);
    const uint16_t *kb = dv.K + b * dv.sb + h * dv.sh;
    const uint16_t *vb = dv.V + b * dv.sb + h * dv.sh;
    const int *rowpos = dv.rowpos + (size_t)u * dv.n_cap;
    const uint32_t *rowmask = dv.rowmask + (size_t)u * dv.n_cap;
    WarpAcc acc;
    acc.init();
    const float scale2 = dv.tau * LOG2E;
    {
        // Rows are taken POSCH at a time; the positions and head masks of the next POSCH rows
        // are copied into shared memory (cp.async) while the current ones are attended, so
        // no copy of a K/V row waits on a global load of its position.  Inside a pass each
        // row warp runs its own pipeline over 16-row blocks w, w+RW, ... with NB buffers.
        const int RW = m.rwarps, NB = m.nbuf;
        uint8_t *wbuf = area + (size_t)warp * NB * WB_BYTES;
        int *posb = reinterpret_cast<int *>(sm + m.posb);  // [2][2][POSCH]
        auto stage_pos = [&](int c0p, int buf) {  // rows c0p .. c0p + POSCH of [r0, r1)
            int *pp = posb + buf * 2 * POSCH;
            uint32_t *mm = reinterpret_cast<uint32_t *>(pp + POSCH);
            const int n = min(POSCH, r1 - c0p);
            for (int t = tid; t < n; t += NT) {
                const int i = c0p + t;
                if (i < n_anchor) {
                    pp[t] = i < s_cnt ? i : rlo + (i - s_cnt);
                    mm[t] = allm;
                } else {
                    int lo = 0, hi = Uc - 1;  // last slot with pre[slot] <= i
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (pre[mid] <= i) lo = mid;
                        else hi = mid - 1;
                    }
                    const int kk = ucoff[lo] + (i - pre[lo]);
                    cp_async4(smem_u32(pp + t), rowpos + kk);
                    cp_async4(smem_u32(mm + t), rowmask + kk);
                }
            }
            cp_async_commit();
        };
        if (r0 < r1) stage_pos(r0, 0);
        int pb = 0;
        for (int c0p = r0; c0p < r1; c0p += POSCH, pb ^= 1) {
            const int nrow = min(POSCH, r1 - c0p);
            cp_async_wait<0>();  // this pass's positions
            __syncthreads();
            if (c0p + POSCH < r1) stage_pos(c0p + POSCH, pb ^ 1);  // next pass's, in flight
            const int *pp = posb + pb * 2 * POSCH;
            const uint32_t *mm = reinterpret_cast<const uint32_t *>(pp + POSCH);
            const int nblk = (int)ceil_div64(nrow, WB_ROWS);
            auto rowinfo = [&](int bi, int &pos, uint32_t &mk) {  // lane's row of block bi
                pos = 0;
                mk = 0u;
                const int t = bi * WB_ROWS + lane;
                if (bi >= nblk || lane >= WB_ROWS || t >= nrow) return;
                pos = pp[t];
                mk = mm[t];
                if ((unsigned)pos >= (unsigned)dv.n_cap) {  // corrupt partition: flag, skip
                    flag_error(dv.status, ST_BAD_INDEX);
                    pos = 0;
                    mk = 0u;
                }
            };
            auto nrows_of = [&](int bi) { return min(WB_ROWS, nrow - bi * WB_ROWS); };
            const int b0 = warp < RW ? warp : nblk;  // warps without row buffers take no blocks
            int pos;
            uint32_t mk;
            for (int j = 0; j < NB - 1; ++j) {  // prologue: the first NB-1 blocks
                const int bi = b0 + j * RW;
                rowinfo(bi, pos, mk);
                if (bi < nblk) warp_issue_block(wbuf + (size_t)j * WB_BYTES, nrows_of(bi), pos, mk, kb, vb, dv.sn);
                cp_async_commit();
            }
            for (int t = 0; b0 + t * RW < nblk; ++t) {
                const int bn = b0 + (t + NB - 1) * RW;  // block entering the pipeline
                rowinfo(bn, pos, mk);
                if (bn < nblk)
                    warp_issue_block(wbuf + (size_t)((t + NB - 1) % NB) * WB_BYTES, nrows_of(bn), pos, mk,
                                     kb, vb, dv.sn);
                cp_async_commit();
                // the next pass's position copies (if any) were committed before this loop:
                // they are older than every block group, so waiting for block t covers them
                cp_async_wait_dyn(NB - 1);
                __syncwarp();
                const uint8_t *cur = wbuf + (size_t)(t % NB) * WB_BYTES;
                const uint32_t sk = smem_u32(cur);
                compute_rows16(acc, qa, sk, sk + WB_KV, reinterpret_cast<const uint32_t *>(cur + 2 * WB_KV), 0,
                               scale2);
                __syncwarp();
            }
            cp_async_wait<0>();
            __syncthreads();  // the pass's buffers and positions are free
        }
    }
    __syncthreads();
    float *wst = reinterpret_cast<float *>(area);  // [W][G][PART_W] + residual state after it
    warp_state_out(acc, wst, G);
    for (int e = tid; e < G * PART_W; e += NT) wst[(size_t)W * G * PART_W + e] = rst[e];
    __syncthreads();
    merge_states(wst, W + 1, G, pub_state);
    cluster.sync();  // S3: every CTA's partial is published

    // ------------------------------------- P5: this CTA's slice of the output
    {
        const int tot = G * MOG_D;
        const int e0 = (int)((int64_t)tot * k / CS), e1 = (int)((int64_t)tot * (k + 1) / CS);
        for (int e = e0 + tid; e < e1; e += NT) {
            const int g = e / MOG_D, j = e % MOG_D;
            float M = -INFINITY;
            for (int src = 0; src < CS; ++src)
                M = fmaxf(M, cluster.map_shared_rank(pub_state, src)[g * PART_W]);
            float lsum = 0.f, asum = 0.f;
            if (M != -INFINITY)
                for (int src = 0; src < CS; ++src) {
                    const float *ps = cluster.map_shared_rank(pub_state, src) + g * PART_W;
                    const float mi = ps[0];
                    if (mi == -INFINITY) continue;
                    const float sc = exp2f(mi - M);
                    lsum += sc * ps[1];
                    asum += sc * ps[PART_ACC + j];
                }
            a.out[(size_t)u * G * MOG_D + e] = lsum > 0.f ? asum / lsum : 0.f;
        }
    }
    cluster.sync();  // S4: keep this CTA's shared memory alive for the other readers
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
        MdLay m = md_layout(dv.G, dv.tc, dv.c_max, dv.l_max, cs, md_warps(GT));
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
    if (events)
        for (int i = 1; i < 4; ++i)
            if ((e = cudaEventRecord(events[i], s)) != cudaSuccess) return e;
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
    return (size_t)md_layout(G, tc, c_max, MOG_MAX_L, 16, md_warps(G <= 4 ? 4 : 16)).total;
}

cudaError_t launch_append(const Dev &dv, const Plan &pl, const void *k_new, const void *v_new,
                          cudaStream_t s) {
    k_append<<<pl.batch, 128, 0, s>>>(dv, static_cast<const uint16_t *>(k_new),
                                      static_cast<const uint16_t *>(v_new));
    return cudaGetLastError();
}

}  // namespace mog
