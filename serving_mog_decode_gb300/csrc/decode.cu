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
// Three kernels per decode step, launched back to back on one stream with programmatic
// dependent launch (each starts while its predecessor drains and waits with
// griddepcontrol.wait before its first dependent read):
//  k_mog_decode  selection: one thread-block cluster of CS CTAs per KV head ("unit").
//                Cluster scores for the G query heads, each head's top-tc clusters, their
//                union, the subcluster scores and each head's top-ts inside every chosen
//                cluster, the exponents of the Gaussian residual terms, and the row
//                segments and split plan of the next kernel.  Hand-offs between the CTAs
//                go through distributed shared memory behind cluster barriers.
//  k_mog_rows    exact attention: grid (P, units).  Each CTA streams its share of the
//                unit's exact rows (anchors, then the chosen subclusters' rows gathered
//                through the partition) and then its share of the residual terms through
//                the same mma.sync tile pipeline, and writes one unnormalised partial
//                (max, sum, acc).
//  k_mog_merge   grid (G, units): folds the P partials of one query head with one running
//                maximum and normalises once.
// k_append writes the new key and value of each sequence and advances its length.
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
    int warm;  // 1: the rows and merge kernels run their warm-up pass before the wait
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
// the chunks k = q + 4i (dimensions 4k..4k+3) of the mean and of the variance, from the
// fp32 summary ms or, when ms16 (ms8) is given, from its bf16 (fp8 e4m3) copy.  For every
// head g < G (G <= GT), emit(g, res, sel) is called on all 4 lanes with the log-mass
// exponent res (the residual's) and the selection score sel.
template <int GT, class Emit>
__device__ __forceinline__ void quad_scores(const float *ms, const uint16_t *ms16, const uint8_t *ms8, int n,
                                            bool valid, const float4 *w, int G, int mode, Emit &&emit) {
    const int q = threadIdx.x & 3;
    float4 mu[8], va[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (valid && ms8) {
            mu[i] = e4m3x4_to_float4(*reinterpret_cast<const uint32_t *>(ms8 + 4 * (q + 4 * i)));
            va[i] = e4m3x4_to_float4(*reinterpret_cast<const uint32_t *>(ms8 + MOG_D + 4 * (q + 4 * i)));
        } else if (valid && ms16) {
            const uint2 a = *reinterpret_cast<const uint2 *>(ms16 + 4 * (q + 4 * i));
            const uint2 b = *reinterpret_cast<const uint2 *>(ms16 + MOG_D + 4 * (q + 4 * i));
            mu[i] = make_float4(bf_lo(a.x), bf_hi(a.x), bf_lo(a.y), bf_hi(a.y));
            va[i] = make_float4(bf_lo(b.x), bf_hi(b.x), bf_lo(b.y), bf_hi(b.y));
        } else if (valid) {
            mu[i] = *reinterpret_cast<const float4 *>(ms + 4 * (q + 4 * i));
            va[i] = *reinterpret_cast<const float4 *>(ms + MOG_D + 4 * (q + 4 * i));
        } else {
            mu[i] = va[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    const float ln = n > 0 ? logf((float)n) : 0.f;
    const bool ok = valid && n > 0;
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
        const float res = ok ? ln + dm + dq : -INFINITY;
        emit(g, res, !ok ? -INFINITY : (mode == 0 ? res : dm));
    }
}

// Running log-sum-exp over the heads' selection scores, the group score of the
// group-shared selection: the log of the sum over the G heads of exp(selection score)
// (-inf when every score is -inf).
struct LogSumExp {
    float mx = -INFINITY, sum = 0.f;
    __device__ __forceinline__ void add(float x) {
        if (x == -INFINITY) return;
        if (x > mx) {
            sum = sum * expf(mx - x) + 1.f;
            mx = x;
        } else {
            sum += expf(x - mx);
        }
    }
    __device__ __forceinline__ float value() const { return mx == -INFINITY ? -INFINITY : mx + logf(sum); }
};

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}

// dynamic shared memory of the decode kernel: the 227 KB block limit less its static arrays
constexpr int MD_SMEM_MAX = 226 * 1024;

__host__ __device__ constexpr int md_warps(int GT) { return GT <= 4 ? 12 : 8; }
// CTAs per SM the selection kernel is compiled for (register budget): two for G > 4, so
// that a batch of many KV heads gets 8-CTA clusters
__host__ __device__ constexpr int md_min_blocks(int GT) { return GT <= 4 ? 1 : 2; }

// Shared-memory layout of the selection kernel (byte offsets).
struct MdLay {
    int CS, SL, SLp, KC, NPOOL, NSLOT, SPC, warps;  // KC: candidates per slice and head;
                                                    // NPOOL: CS*KC padded
    int cand_k, allc_k, selc, gpre, gseg;  // allc_k, selc, gpre, gseg receive other CTAs' pushes
    int w, ckey, crs, cnn, slm, bm, ucl;
    int sres, ssl, snn, sso, spref, smask, shm;
    int total;
};

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
    m.SLp = (m.SL + 7) & ~7;
    m.KC = m.SL < tcc ? m.SL : tcc;
    m.NPOOL = (CS * m.KC + 7) & ~7;
    m.NSLOT = tc > 0 ? (c_max < G * tc ? c_max : G * tc) : 1;
    m.SPC = (m.NSLOT + CS - 1) / CS;
    m.cand_k = take(8 * G * m.KC, 16);
    m.allc_k = take(8 * G * m.NPOOL, 16);
    m.selc = take(4 * G * tcc, 16);
    m.gpre = take(4 * (m.NSLOT + 1), 16);
    m.gseg = take(4 * (m.NSLOT + 1), 16);
    m.w = take(16 * 64 * G, 16);
    m.ckey = take(8 * G * m.SLp, 16);
    m.crs = take(4 * G * m.SL, 16);
    m.cnn = take(4 * m.SL, 16);
    m.slm = take(4 * m.SL, 16);
    m.bm = take(4 * ((c_max + 31) / 32), 16);
    m.ucl = take(4 * m.NSLOT, 16);
    m.sres = take(4 * m.SPC * G * MOG_MAX_L, 16);
    m.ssl = take(4 * m.SPC * G * MOG_MAX_L, 16);
    m.snn = take(4 * m.SPC * MOG_MAX_L, 16);
    m.sso = take(4 * m.SPC * (MOG_MAX_L + 1), 16);
    m.spref = take(4 * m.SPC * (MOG_MAX_L + 1), 16);
    m.smask = take(4 * m.SPC * MOG_MAX_L, 16);
    m.shm = take(4 * m.SPC, 16);
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

// Selection order as one integer: a larger key ranks first (score descending, then index
// ascending); 0 for a candidate that is never chosen (score -inf or NaN, index < 0).
__device__ __forceinline__ unsigned long long rank_key(float sc, int idx) {
    if (!(sc > -INFINITY) || idx < 0) return 0ull;
    uint32_t bits = __float_as_uint(sc == 0.f ? 0.f : sc);  // -0 ranks as +0
    bits = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    return ((unsigned long long)bits << 32) | (uint32_t)(0x7fffffff - idx);
}
__device__ __forceinline__ int key_index(unsigned long long key) {
    return 0x7fffffff - (int)(uint32_t)key;
}
// Rank of key x among keys[0 .. n) (n a multiple of 8, zero padded): how many are larger,
// counted up to `cap` (the result is >= cap once the key is out of the selection).
__device__ __forceinline__ int key_rank(const unsigned long long *keys, int n, unsigned long long x,
                                        int cap) {
    int rank = 0;
    for (int j0 = 0; j0 < n && rank < cap; j0 += 8) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) rank += keys[j0 + jj] > x;
    }
    return rank;
}

// Kernel A: one thread-block cluster of CS CTAs per unit.  Selection, the Gaussian
// residual and the rows kernel's plan.  Hand-offs between the CTAs are pushed (stores
// into the other CTAs' shared memory) and made visible by a cluster barrier:
//  P1  CTA k scores its slice of clusters for the G query heads and pushes the slice's
//      top-KC keys per head into every CTA's candidate pool;
//  P2  CTA k ranks its share of each head's pool and pushes the winners into every CTA's
//      top-tc list; each CTA then forms the union over the heads (ascending index);
//  P3  CTA k takes union slots k, k+CS, ...: subcluster scores, the top-ts subclusters of
//      every head that chose the slot's cluster, the slot's row and segment counts
//      (pushed), and the exponents of the residual terms: the unchosen subclusters of those
//      heads and its slice clusters no head chose;
//  P4  the unit's row segments (one per chosen subcluster, in slot order) and the first
//      segment of every rows-kernel CTA.
template <int GT>
__global__ void __launch_bounds__(md_warps(GT) * 32, md_min_blocks(GT)) k_mog_decode(DecArgs a, MdLay m) {
    namespace cg = cooperative_groups;
    constexpr int W = md_warps(GT), NT = W * 32;
    extern __shared__ __align__(128) uint8_t sm[];
    cg::cluster_group cluster = cg::this_cluster();
    const Dev &dv = a.dv;
    const int G = dv.G, tc = dv.tc, ts = dv.ts, tcc = max(tc, 1);
    const int CS = m.CS, k = (int)cluster.block_rank();
    const int u = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned long long *cand_k = reinterpret_cast<unsigned long long *>(sm + m.cand_k);
    unsigned long long *allc_k = reinterpret_cast<unsigned long long *>(sm + m.allc_k);  // [g][r][src]
    int *selc = reinterpret_cast<int *>(sm + m.selc);
    int *gpre = reinterpret_cast<int *>(sm + m.gpre);  // rows of union slot j, then its first row
    int *gseg = reinterpret_cast<int *>(sm + m.gseg);  // segments of slot j, then its first one
    float4 *w = reinterpret_cast<float4 *>(sm + m.w);
    unsigned long long *ckey = reinterpret_cast<unsigned long long *>(sm + m.ckey);  // slice keys
    float *crs = reinterpret_cast<float *>(sm + m.crs);
    int *cnn = reinterpret_cast<int *>(sm + m.cnn);
    uint32_t *slm = reinterpret_cast<uint32_t *>(sm + m.slm);  // heads that chose slice cluster
    uint32_t *bm = reinterpret_cast<uint32_t *>(sm + m.bm);
    int *ucl = reinterpret_cast<int *>(sm + m.ucl);
    float *sres = reinterpret_cast<float *>(sm + m.sres);
    float *ssl = reinterpret_cast<float *>(sm + m.ssl);  // subcluster selection scores
    int *snn = reinterpret_cast<int *>(sm + m.snn);
    int *sso = reinterpret_cast<int *>(sm + m.sso);
    int *spref = reinterpret_cast<int *>(sm + m.spref);
    uint32_t *smask = reinterpret_cast<uint32_t *>(sm + m.smask);
    uint32_t *shm = reinterpret_cast<uint32_t *>(sm + m.shm);  // heads that chose slot s
    __shared__ int s_wsum[W], s_uc;

    // Build-time constants of the unit (never rewritten after the build) may be read
    // before the wait; the window start and the current length are advanced by the append
    // and slide kernels and are read after it, where they are used.
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int b = ui[UI_B], C = ui[UI_C], L = ui[UI_L], S = ui[UI_S];
    const size_t ug = (size_t)u * dv.c_max;               // cluster index base
    const size_t usg = (size_t)u * dv.c_max * dv.l_max;   // subcluster index base
    const uint16_t *qg = a.q + (size_t)u * G * MOG_D;
    int *selu = dv.sel + (size_t)u * G * a.SW;
    const bool resid = dv.residual == 1;  // the Gaussian residual's terms (not the feature map's)
    const bool uex = dv.union_exact != 0;  // every head attends the union's subclusters
    const bool grp = dv.group_select != 0;  // one selection per KV head, by log-sum-exp
    const int GS = grp ? 1 : G;             // selection lists
    const uint32_t allg = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    const bool pooled = tc > 0 && !a.sel_in;  // selection from the scores (not given)

    // Every CTA of the cluster must have started before any pushes into its shared memory:
    // arrive now, wait before the first push.
    cluster_arrive_relaxed();
    const int c0 = k * m.SL;
    const int ns = max(0, min(C - c0, m.SL));
    const int KC = m.KC, npool = CS * KC;
    // this CTA's own shared arrays (nothing global is read before the wait)
    for (int e = tid; e < G * (m.SLp - ns); e += NT)  // padding keys
        ckey[(e / (m.SLp - ns)) * m.SLp + ns + e % (m.SLp - ns)] = 0ull;
    for (int e = tid; e < m.SL; e += NT) slm[e] = 0u;
    for (int e = tid; e < G * tcc; e += NT) selc[e] = -1;
    for (int e = tid; e < (dv.c_max + 31) / 32; e += NT) bm[e] = 0u;
    for (int e = tid; e < G * KC; e += NT) cand_k[e] = 0ull;
    for (int e = tid; e < G * (m.NPOOL - npool); e += NT)  // this CTA's own pool padding
        allc_k[(e / (m.NPOOL - npool)) * m.NPOOL + npool + e % (m.NPOOL - npool)] = 0ull;

    // ------------------------------------------------------------ P0: query, weights
    // The query may be written by the kernel just before this one, so it is read only
    // after the dependency wait too.  The slice's summaries and counts are requested into
    // L2 first, so that their latency overlaps the query's.
    pdl_wait();
    pdl_trigger();
    {
        const char *ms0 = dv.cl_ms8    ? reinterpret_cast<const char *>(dv.cl_ms8 + (ug + c0) * 2 * MOG_D)
                          : dv.cl_ms16 ? reinterpret_cast<const char *>(dv.cl_ms16 + (ug + c0) * 2 * MOG_D)
                                       : reinterpret_cast<const char *>(dv.cl_ms + (ug + c0) * 2 * MOG_D);
        const int lines = ns * (dv.cl_ms8 ? 2 : dv.cl_ms16 ? 4 : 8);  // 128-byte lines of the slice's summaries
        for (int e = tid; e < lines; e += NT) prefetch_l2(ms0 + 128 * (size_t)e);
        const char *n0 = reinterpret_cast<const char *>(dv.cl_n + ug + c0);
        if (tid * 128 < ns * 4) prefetch_l2(n0 + 128 * tid);
        if (tid == 0 && ns > 0) prefetch_l2(n0 + 4 * (ns - 1));
    }
    load_weights(w, qg, G, dv.tau);
    __syncthreads();

    // ------------------------------------------------- P1: score this CTA's clusters
    for (int base = 0; base < ns; base += NT / 4) {
        const int cl = base + (tid >> 2);
        const bool valid = cl < ns;
        const int c = c0 + (valid ? cl : 0);
        const int n = valid ? dv.cl_n[ug + c] : 0;
        const bool wr = valid && (tid & 3) == 0;
        LogSumExp gsc;
        quad_scores<GT>(dv.cl_ms + (ug + c) * 2 * MOG_D,
                        dv.cl_ms16 ? dv.cl_ms16 + (ug + c) * 2 * MOG_D : nullptr,
                        dv.cl_ms8 ? dv.cl_ms8 + (ug + c) * 2 * MOG_D : nullptr, n, valid, w, G, dv.score_mode,
                    [&](int g, float res, float sl) {
                        if (wr) {
                            ckey[g * m.SLp + cl] = rank_key(sl, c);
                            crs[g * m.SL + cl] = res;
                        }
                        gsc.add(sl);
                    });
        if (wr) {
            if (grp) ckey[cl] = rank_key(gsc.value(), c);
            cnn[cl] = n;
        }
    }
    __syncthreads();
    cluster_wait();
    if (pooled) {
        // this slice's top-KC per head (KC = min(slice, tc)) by rank, 0 padded ...
        for (int e = tid; e < GS * ns; e += NT) {
            const int g = e / ns, i = e % ns;
            const unsigned long long x = ckey[g * m.SLp + i];
            if (x == 0ull) continue;
            const int rank = key_rank(ckey + g * m.SLp, m.SLp, x, KC);
            if (rank < KC) cand_k[g * KC + rank] = x;
        }
        __syncthreads();
        // ... pushed into every CTA's pool, rank-major: pool[g][r][k]
        for (int e = tid; e < CS * GS * KC; e += NT) {
            const int dst = e / (GS * KC), q = e % (GS * KC), g = q / KC, r = q % KC;
            cluster.map_shared_rank(allc_k, dst)[g * m.NPOOL + r * CS + k] = cand_k[q];
        }
    }
    cluster.sync();  // S1: every CTA's pool is complete

    // ------------------------------------------------------- P2: selection and union
    if (pooled) {  // every CTA ranks the whole pool: each head's top-tc, in rank order
        for (int e = tid; e < GS * npool; e += NT) {
            const int g = e / npool;
            const unsigned long long x = allc_k[g * m.NPOOL + e % npool];
            if (x == 0ull) continue;
            const int rank = key_rank(allc_k + g * m.NPOOL, m.NPOOL, x, tc);
            if (rank < tc) selc[g * tc + rank] = key_index(x);
        }
    } else if (tc > 0) {
        for (int e = tid; e < GS * tc; e += NT) {  // (group mode: head 0's row)
            const int g = e / tc, r = e % tc;
            const int cc = a.sel_in[((size_t)u * G + g) * a.SW + r];
            selc[e] = (cc >= 0 && cc < C && dv.cl_n[ug + cc] > 0) ? cc : -1;
        }
    }
    __syncthreads();  // this CTA holds the full top-tc lists
    for (int e = tid; e < GS * tc; e += NT) {
        const int c = selc[e];
        if (c < 0) continue;
        atomicOr(&bm[c >> 5], 1u << (c & 31));
        if (c >= c0 && c < c0 + ns) atomicOr(&slm[c - c0], grp ? allg : 1u << (e / tc));
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
            const int cs = selc[(grp ? 0 : g) * tc + r];
            selu[(size_t)g * a.SW + r] = cs;
            if (cs < 0)
                for (int kk = 0; kk < ts; ++kk) selu[(size_t)g * a.SW + tc + r * ts + kk] = -1;
        }
    }

    // ----------------------------------------- P3: this CTA's union slots, residual
    const int nmy = Uc > k ? (Uc - k + CS - 1) / CS : 0;  // slots k, k+CS, ...
    const int npair = nmy * L;                              // (slot, subcluster) pairs
    // offsets and sizes of the slots' subclusters, in flight while their scores are computed
    for (int e = tid; e < nmy * (L + 1); e += NT) {
        const int s = e / (L + 1), i = e % (L + 1);
        const size_t c = (size_t)ucl[k + s * CS];
        cp_async4(smem_u32(sso + s * (MOG_MAX_L + 1) + i), dv.sub_off + (size_t)u * dv.sub_off_stride + c * L + i);
        if (i < L) cp_async4(smem_u32(snn + s * MOG_MAX_L + i), dv.sub_n + usg + c * L + i);
    }
    cp_async_commit();
    for (int base = 0; base < npair; base += NT / 4) {  // subcluster scores, 4 lanes a pair
        const int pr = base + (tid >> 2);
        const bool valid = pr < npair;
        const int s = valid ? pr / L : 0, l = valid ? pr % L : 0;
        const size_t gi = usg + (valid ? (size_t)ucl[k + s * CS] * L + l : 0);
        const bool wr = valid && (tid & 3) == 0;
        LogSumExp gsc;
        quad_scores<GT>(dv.sub_ms + gi * 2 * MOG_D, dv.sub_ms16 ? dv.sub_ms16 + gi * 2 * MOG_D : nullptr,
                        dv.sub_ms8 ? dv.sub_ms8 + gi * 2 * MOG_D : nullptr, valid ? dv.sub_n[gi] : 0, valid, w, G,
                    dv.score_mode, [&](int g, float res, float sl) {
                        if (wr) {
                            sres[(s * G + g) * MOG_MAX_L + l] = res;
                            ssl[(s * G + g) * MOG_MAX_L + l] = sl;
                        }
                        gsc.add(sl);
                    });
        if (wr && grp) ssl[(s * G) * MOG_MAX_L + l] = gsc.value();
    }
    for (int e = tid; e < nmy * MOG_MAX_L; e += NT) smask[e] = 0u;
    for (int e = tid; e < nmy; e += NT) shm[e] = 0u;
    cp_async_wait<0>();
    __syncthreads();
    // top-ts subclusters of every head that chose a slot's cluster
    for (int e = warp; e < nmy * G; e += W) {
        const int s = e / G, g = e % G, gs = grp ? 0 : g;  // gs: the selection head g follows
        const int c = ucl[k + s * CS];
        int rk = -1;  // the rank at which head g chose c
        for (int r0 = 0; r0 < tc && rk < 0; r0 += 32) {
            const uint32_t hit = __ballot_sync(0xffffffffu, r0 + lane < tc && selc[gs * tc + r0 + lane] == c);
            if (hit) rk = r0 + __ffs(hit) - 1;
        }
        if (rk < 0) continue;
        if (lane == 0) atomicOr(&shm[s], 1u << g);
        int *subs = selu + (size_t)g * a.SW + tc + (size_t)rk * ts;
        const int *nn = snn + s * MOG_MAX_L;
        if (a.sel_in) {
            const int32_t *si = a.sel_in + ((size_t)u * G + gs) * a.SW + tc + (size_t)rk * ts;
            for (int r = lane; r < ts; r += 32) {
                const int l2 = si[r];
                const bool ok = l2 >= 0 && l2 < L && nn[l2] > 0;
                subs[r] = ok ? l2 : -1;
                if (ok) atomicOr(&smask[s * MOG_MAX_L + l2], 1u << g);
            }
        } else {
            const float *sc = ssl + (s * G + gs) * MOG_MAX_L;
            const unsigned long long x = lane < L ? rank_key(sc[lane], lane) : 0ull;
            int rank = 0;
#pragma unroll 2
            for (int j = 0; j < L; ++j) rank += rank_key(sc[j], j) > x;
            if (x != 0ull && rank < ts) {
                subs[rank] = lane;
                atomicOr(&smask[s * MOG_MAX_L + lane], 1u << g);
            }
            const int nvalid = __popc(__ballot_sync(0xffffffffu, x != 0ull));
            for (int r = nvalid + lane; r < ts; r += 32) subs[r] = -1;
        }
    }
    __syncthreads();
    for (int s = warp; s < nmy; s += W) {  // chosen subclusters: prefix of sizes, counts
        const int *so = sso + s * (MOG_MAX_L + 1);
        const bool ch = lane < L && smask[s * MOG_MAX_L + lane] != 0u;
        const int cnt = ch ? so[lane + 1] - so[lane] : 0;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int nseg = __popc(__ballot_sync(0xffffffffu, ch));
        const int rows = __shfl_sync(0xffffffffu, incl, 31);
        if (lane < L) spref[s * (MOG_MAX_L + 1) + lane + 1] = incl;
        if (lane == 0) spref[s * (MOG_MAX_L + 1)] = 0;
        const int j = k + s * CS;  // the slot's counts, pushed to every CTA
        for (int dst = lane; dst < CS; dst += 32) {
            cluster.map_shared_rank(gpre, dst)[j] = rows;
            cluster.map_shared_rank(gseg, dst)[j] = nseg;
        }
    }
    // Gaussian residual terms, attended by the rows kernel: for the heads that chose slot s
    // but not its subcluster l, and for the heads that did not choose slice cluster c, the
    // exponent (log2) of the term; -inf where the head does not take it.  In the
    // union-exact mode every head takes the subclusters no head chose and the clusters
    // outside the union instead.  Items: the union pairs (slot j, subcluster l) at
    // j*L + l, then the clusters at Uc*L + c; rows of G exponents padded to a multiple of 4.
    __syncthreads();
    {
        float *rx = dv.resx + (size_t)u * dv.resx_stride;
        const int GP = (G + 3) & ~3;  // 16-byte rows
        for (int e = tid; e < npair * GP; e += NT) {
            const int p = e / GP, g = e - p * GP, s = p / L, l = p - s * L;
            const uint32_t takers = uex ? (smask[s * MOG_MAX_L + l] ? 0u : allg)
                                        : (shm[s] & ~smask[s * MOG_MAX_L + l]);
            const bool need = resid && g < G && snn[s * MOG_MAX_L + l] > 0 && ((takers >> g) & 1u);
            rx[((size_t)(k + s * CS) * L + l) * GP + g] = need ? sres[(s * G + g) * MOG_MAX_L + l] * LOG2E : -INFINITY;
        }
        for (int e = tid; e < ns * GP; e += NT) {
            const int cl = e / GP, g = e - cl * GP;
            const uint32_t takers = uex ? (slm[cl] ? 0u : allg) : ~slm[cl];
            const bool need = resid && g < G && cnn[cl] > 0 && ((takers >> g) & 1u);
            rx[((size_t)Uc * L + c0 + cl) * GP + g] = need ? crs[g * m.SL + cl] * LOG2E : -INFINITY;
        }
    }
    cluster.sync();  // S2: every slot's counts have been pushed

    // ------------------------------------- P4: row segments and the rows-kernel plan
    const int rlo = __ldcg(ui + UI_RLO), nnow = __ldcg(dv.n_now + b);
    const int s_cnt = min(S, nnow), n_anchor = s_cnt + max(0, nnow - rlo);
    if (warp == 0) {  // exclusive prefixes: rows after the anchors, segments from 0
        int rrun = n_anchor, srun = 0;
        for (int j0 = 0; j0 < Uc; j0 += 32) {
            const int j = j0 + lane;
            const int rc = j < Uc ? gpre[j] : 0, sc = j < Uc ? gseg[j] : 0;
            int ri = rc, si = sc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ri, o);
                const int z = __shfl_up_sync(0xffffffffu, si, o);
                if (lane >= o) {
                    ri += y;
                    si += z;
                }
            }
            if (j < Uc) {
                gpre[j] = rrun + ri - rc;
                gseg[j] = srun + si - sc;
            }
            rrun += __shfl_sync(0xffffffffu, ri, 31);
            srun += __shfl_sync(0xffffffffu, si, 31);
        }
        if (lane == 0) {
            gpre[Uc] = rrun;
            gseg[Uc] = srun;
        }
    }
    __syncthreads();
    const int T = gpre[Uc], P = dv.P;
    int *plan = dv.plan + (size_t)u * PLAN_W;
    const size_t useg = (size_t)u * dv.nseg_max;
    for (int s = warp; s < nmy; s += W) {  // this CTA's slots: segments and rows-CTA starts
        const int j = k + s * CS;
        const uint32_t chosen = __ballot_sync(0xffffffffu, lane < L && smask[s * MOG_MAX_L + lane] != 0u);
        if (lane < L && ((chosen >> lane) & 1u)) {
            const size_t sg = useg + gseg[j] + __popc(chosen & lanemask_lt());
            dv.segrow[sg] = gpre[j] + spref[s * (MOG_MAX_L + 1) + lane];
            dv.segoff[sg] = sso[s * (MOG_MAX_L + 1) + lane];
            dv.segmask[sg] = uex ? allg : smask[s * MOG_MAX_L + lane];
        }
        const int ra = gpre[j], rb = gpre[j + 1];
        if (ra < rb) {  // rows-kernel CTAs p whose first row floor(T p / P) lies in [ra, rb)
            const int pa = (int)(((int64_t)ra * P + T - 1) / T);
            const int pb = (int)(((int64_t)rb * P + T - 1) / T);
            for (int p = pa + lane; p < pb; p += 32) {
                const int rr = (int)((int64_t)T * p / P) - ra;
                const int l = last_le(spref + s * (MOG_MAX_L + 1), L, rr);  // a chosen subcluster
                plan[PLAN_START + p] = gseg[j] + __popc(chosen & ((1u << l) - 1u));
            }
        }
    }
    if (k == 0) {
        if (tid == 0) {
            plan[0] = gseg[Uc];  // segments
            plan[1] = T;
            plan[2] = n_anchor;
            plan[3] = s_cnt;
            plan[4] = rlo;
            plan[5] = Uc;
            plan[6] = L;
            plan[7] = C;
        }
        for (int j = tid; j < Uc; j += NT) plan[PLAN_UCL + j] = ucl[j];
        // CTAs that start among the anchors (or in an empty list) start at segment 0
        const int pe = T > 0 ? (int)(((int64_t)n_anchor * P + T - 1) / T) : P;
        for (int p = tid; p < min(pe, P); p += NT) plan[PLAN_START + p] = 0;
    }
}

constexpr int RW_SUPER = 256;                  // row positions per batch in the rows kernel
constexpr int RW_TPB = RW_SUPER / AT_ROWS;     // tiles per batch
constexpr int RW_PER = RW_SUPER / AT_THREADS;  // positions a thread fetches per batch
constexpr int RW_SEGW = 256;                   // row segments held in shared memory
// Two tile stages (one copy in flight while the other is computed) keep a CTA at 74.6 KB
// of shared memory, so three CTAs fit on an SM: more warps to hide the tile computation's
// latencies, and more copies in flight per SM than two CTAs with three stages.
constexpr int RW_STAGES = 2;
constexpr int RW_SMEM = RW_STAGES * AT_STAGE_BYTES;
static_assert(RW_TPB >= RW_STAGES - 1, "the first batch must cover the pipeline's prologue");

// Kernel B: grid (P, units), 4 warps, three CTAs per SM.  Rows [p*T/P, (p+1)*T/P) of the
// unit's exact list (anchors, then the chosen subclusters' rows, segment by segment)
// through the 64-row tile engine.  A window of segments sits in shared memory; a row's
// position is read from the partition (perm) at its segment's offset.  Positions are
// fetched into registers two batches ahead and moved to shared memory when the pipeline
// reaches the batch, so no tile copy waits on a position load.  After its rows, the CTA
// streams its share of the Gaussian residual terms through the same pipeline.  One
// unnormalised partial per CTA.
template <int GT, bool PAGED>
__global__ void __launch_bounds__(AT_THREADS) k_mog_rows(DecArgs a) {
    extern __shared__ __align__(128) uint8_t tile[];
    const Dev &dv = a.dv;
    const int G = dv.G;
    __shared__ __align__(16) int s_plan[PLAN_W];
    __shared__ int s_pos[2][RW_SUPER];
    __shared__ uint32_t s_mk[2][RW_SUPER];
    __shared__ int s_segrow[RW_SEGW + 1], s_segoff[RW_SEGW];
    __shared__ uint32_t s_segmask[RW_SEGW];
    const int u = blockIdx.y, p = blockIdx.x, P = gridDim.x;
    const int tid = threadIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int b = ui[UI_B], h = u % dv.h_kv;
    const uint32_t allm = (G >= 32) ? 0xffffffffu : ((1u << G) - 1u);
    constexpr int NB = GT <= 8 ? 1 : 2;  // blocks of 8 query heads
    QFrags<NB> qf;
    load_q_frags(qf, a.q + (size_t)u * G * MOG_D, G);
    // Two passes through the same code.  Pass 0 runs before the dependency wait, mostly
    // while the selection kernel is still working (this kernel is launched early): one
    // zero-filled tile of 64 masked rows and one empty tile of residual terms, into an
    // accumulator that is then discarded.  It brings the tile loop's instructions into the
    // caches, so that the real pass does not stall on instruction fetch between its memory
    // waits.  Pass 1 waits for the selection kernel and does the work.
#pragma unroll 1
    for (int pass = a.warm ? 0 : 1; pass < 2; ++pass) {
    const bool dry = pass == 0;
    if (dry) {  // a plan of 64 anchor rows (T, anchors, sinks), no segments, no terms, L = 1
        for (int q = tid; q < PLAN_W; q += AT_THREADS)
            s_plan[q] = (q >= 1 && q <= 3) ? AT_ROWS : (q == 6 ? 1 : 0);
        __syncthreads();
    } else {
        pdl_wait();  // the selection kernel's segments and plan
        pdl_trigger();
        const int *plan = dv.plan + (size_t)u * PLAN_W;
        for (int q = tid; q < PLAN_W / 4; q += AT_THREADS) cp_async16(smem_u32(s_plan + 4 * q), plan + 4 * q, 16);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
    }
    const int NS = s_plan[0], T = s_plan[1], n_anchor = s_plan[2], s_cnt = s_plan[3], rlo = s_plan[4];
    const int r0 = dry ? 0 : (int)((int64_t)T * p / P), r1 = dry ? T : (int)((int64_t)T * (p + 1) / P);
    const int nrow = r1 - r0, nt = (nrow + AT_ROWS - 1) / AT_ROWS;
    // a paged cache: positions become physical rows (page << pshift | row) when fetched
    const uint16_t *kb = dv.K + (PAGED ? 0 : b * dv.sb) + h * dv.sh;
    const uint16_t *vb = dv.V + (PAGED ? 0 : b * dv.sb) + h * dv.sh;
    const RowAddr<PAGED> ra{(uint32_t)(dv.sn * 2), dv.pshift, dv.sb * 2};
    const int *btb = PAGED ? dv.bt + (int64_t)b * dv.pps : nullptr;
    const int *perm = dv.perm + (size_t)u * dv.n_cap;
    const size_t useg = (size_t)u * dv.nseg_max;
    int wfirst = 0, wn = 0;  // the window: segments wfirst .. wfirst + wn
    auto load_window = [&](int w0) {  // all threads; the caller synchronises
        wfirst = w0;
        wn = max(0, min(RW_SEGW, NS - w0));
        for (int t = tid; t <= wn; t += AT_THREADS) {
            const int sg = w0 + t;
            s_segrow[t] = sg < NS ? __ldcg(dv.segrow + useg + sg) : T;
            if (t < wn) {
                s_segoff[t] = __ldcg(dv.segoff + useg + sg);
                s_segmask[t] = __ldcg(dv.segmask + useg + sg);
            }
        }
    };
    // positions of batch bt into registers; two batches in flight (even / odd sets)
    int pf_pos[2][RW_PER];
    uint32_t pf_mk[2][RW_PER];
    auto fetch_into = [&](int bt, int (&pp)[RW_PER], uint32_t (&mm)[RW_PER]) {
        const int first = r0 + bt * RW_SUPER, last = min(r1, first + RW_SUPER) - 1;
        if (last >= n_anchor && last >= s_segrow[wn]) {  // past the window: move it
            const int f = max(first, n_anchor);
            const int w0 = f < s_segrow[wn] ? wfirst + last_le(s_segrow, wn, f) : wfirst + wn;
            __syncthreads();
            load_window(w0);
            __syncthreads();
        }
#pragma unroll
        for (int jj = 0; jj < RW_PER; ++jj) {
            const int i = first + tid + jj * AT_THREADS;
            int q = 0;
            uint32_t mk = 0u;
            if (i <= last) {
                if (i < n_anchor) {
                    q = dry ? 0 : (i < s_cnt ? i : rlo + (i - s_cnt));
                    mk = dry ? 0u : allm;
                } else {
                    const int sg = last_le(s_segrow, wn, i);  // the segment holding row i
                    const int pi = s_segoff[sg] + (i - s_segrow[sg]);
                    q = (unsigned)pi < (unsigned)dv.n_cap ? __ldg(perm + pi) : -1;
                    mk = s_segmask[sg];
                }
            }
            pp[jj] = q;
            mm[jj] = mk;
        }
    };
    auto fetch = [&](int bt) {
        if (bt & 1) fetch_into(bt, pf_pos[1], pf_mk[1]);
        else fetch_into(bt, pf_pos[0], pf_mk[0]);
    };
    // registers -> shared buffer of batch bt (the loads have landed by now: the values are
    // first used here, so that fetching them never stalls); a paged cache's positions become
    // physical rows, an invalid one -1
    auto place = [&](int bt) {
#pragma unroll
        for (int jj = 0; jj < RW_PER; ++jj) {
            int v = (bt & 1) ? pf_pos[1][jj] : pf_pos[0][jj];
            if (PAGED)
                v = (unsigned)v < (unsigned)dv.n_cap
                        ? (__ldg(btb + (v >> dv.pshift)) << dv.pshift) | (v & ((1 << dv.pshift) - 1))
                        : -1;
            s_pos[bt & 1][tid + jj * AT_THREADS] = v;
            s_mk[bt & 1][tid + jj * AT_THREADS] = (bt & 1) ? pf_mk[1][jj] : pf_mk[0][jj];
        }
    };
    auto issue = [&](int t) {  // (the warm-up tile is zero-filled: no rows are read)
        const int buf = (t / RW_TPB) & 1, rb = (t % RW_TPB) * AT_ROWS;
        issue_tile(tile + (t % RW_STAGES) * AT_STAGE_BYTES, dry ? 0 : min(AT_ROWS, nrow - t * AT_ROWS), kb, vb,
                   ra, [&](int r, int64_t &pos, uint32_t &mk) {
                       int pp = s_pos[buf][rb + r];
                       uint32_t mm = s_mk[buf][rb + r];
                       if (PAGED ? pp < 0 : (unsigned)pp >= (unsigned)dv.n_cap) {  // corrupt partition: flag, skip
                           flag_error(dv.status, ST_BAD_INDEX);
                           pp = 0;
                           mm = 0u;
                       }
                       pos = pp;
                       mk = mm;
                   });
    };
    // The Gaussian residual terms follow the rows as 64-row tiles of given logits: items
    // [ia, ib) of the unit's list (union pairs, then clusters), 32 per tile, each as two
    // rows (bf16 high and low parts of its value mean) with its exponents from the
    // selection kernel.
    const int Uc = s_plan[5], L = s_plan[6], C = s_plan[7];
    const int npi = Uc * L, I = dv.residual == 1 ? npi + C : 0;
    const int ia = (int)((int64_t)I * p / P), ib = (int)((int64_t)I * (p + 1) / P);
    const int nr = dry ? 1 : (ib - ia + AT_ROWS / 2 - 1) / (AT_ROWS / 2);
    const float *rx = dv.resx + (size_t)u * dv.resx_stride;
    const size_t ug = (size_t)u * dv.c_max, usg = ug * dv.l_max;
    auto issue_terms = [&](int t, int tr) {  // tile t of the stream = terms tile tr
        uint8_t *stg = tile + (t % RW_STAGES) * AT_STAGE_BYTES;
        const int i0 = ia + tr * (AT_ROWS / 2), cnt = min(AT_ROWS / 2, ib - i0);
        const uint32_t sv = smem_u32(stg) + AT_TILE_BYTES;
        uint32_t *smk = reinterpret_cast<uint32_t *>(stg + 2 * AT_TILE_BYTES);
        const int ch = tid & 15;
#pragma unroll
        for (int i = 0; i < AT_ROWS / 8; ++i) {
            const int r = (tid >> 4) + 8 * i, it = r >> 1;
            const bool ok = it < cnt;
            const uint16_t *src = dv.cl_vhl;
            if (ok) {
                const int item = i0 + it;
                src = item < npi ? dv.sub_vhl + (usg + (size_t)s_plan[PLAN_UCL + item / L] * L + item % L) * 2 * MOG_D
                                 : dv.cl_vhl + (ug + (item - npi)) * 2 * MOG_D;
                src += (r & 1) * MOG_D + ch * 8;
            }
            // with bf16 or fp8 summaries a term's value mean is its high part alone (for fp8 the
            // build writes the e4m3-rounded mean there, exact in bf16): the low row is zero
            cp_async16(sv + swz(r, ch), src, ok && !((dv.bf16s | dv.fp8s) && (r & 1)) ? 16 : 0);
            if (ch == 0) smk[r] = ok ? allm : 0u;
        }
        float *E = reinterpret_cast<float *>(stg);  // [item][MOG_MAX_G] exponents
        const int G4 = (G + 3) >> 2;
        for (int e = tid; e < cnt * G4; e += AT_THREADS) {
            const int it = e / G4, q = e - it * G4;
            cp_async16(smem_u32(E + it * MOG_MAX_G + 4 * q), rx + (size_t)(i0 + it) * 4 * G4 + 4 * q, 16);
        }
    };
    WarpAcc<NB> acc;
    acc.init();
    const float scale2 = dv.tau * LOG2E;
    if (nt > 0) {
        load_window(s_plan[PLAN_START + p]);
        __syncthreads();
        fetch(0);
        place(0);
        if (nrow > RW_SUPER) fetch(1);
        if (nrow > 2 * RW_SUPER) fetch(2);
    }
    __syncthreads();
#pragma unroll
    for (int s2 = 0; s2 < RW_STAGES - 1; ++s2) {
        if (s2 < nt) issue(s2);
        cp_async_commit();
    }
    for (int t = 0; t < nt; ++t) {
        cp_async_wait<RW_STAGES - 2>();
        __syncthreads();
        const int ti = t + RW_STAGES - 1;
        int next = -1;  // batch whose positions are fetched after this tile's compute
        if (ti < nt) {
            if (ti % RW_TPB == 0) {  // first tile of a batch: its positions go to shared memory
                const int bt = ti / RW_TPB;
                place(bt);
                __syncthreads();
                if ((bt + 2) * RW_SUPER < nrow) next = bt + 2;  // into the set place() freed
            }
            issue(ti);
        }
        cp_async_commit();
        compute_tile(acc, qf, tile + (t % RW_STAGES) * AT_STAGE_BYTES, scale2);
        if (next >= 0) fetch(next);
    }
    cp_async_wait<0>();
    __syncthreads();
    // the residual terms: the same pipeline over nr tiles of given logits
#pragma unroll
    for (int s2 = 0; s2 < RW_STAGES - 1; ++s2) {
        if (s2 < nr) issue_terms(s2, s2);
        cp_async_commit();
    }
    for (int t = 0; t < nr; ++t) {
        cp_async_wait<RW_STAGES - 2>();
        __syncthreads();
        if (t + RW_STAGES - 1 < nr) issue_terms(t + RW_STAGES - 1, t + RW_STAGES - 1);
        cp_async_commit();
        compute_tile<NB, true>(acc, qf, tile + (t % RW_STAGES) * AT_STAGE_BYTES, scale2);
    }
    cp_async_wait<0>();
    __syncthreads();
    if (dry) {  // keep the discarded pass from being optimised away
        if (acc.l[0][0] == 1.5f && acc.m[0][0] == -1.5f) flag_error(dv.status, ST_BAD_SIZE);
        continue;
    }
    float *st = reinterpret_cast<float *>(tile);
    warp_state_out(acc, st, G);
    __syncthreads();
    merge_states(st, AT_WARPS, G, dv.partials + ((size_t)u * PART_SLOTS + p) * G * PART_W);
    }
}

// Kernel C: grid (G, units), 512 threads.  Merges the P partials of one query head
// (running max, rescaled sums) and normalises once.  Thread (part, j) owns partials part,
// part + 4, ... for dimension j; every load is issued before the maximum is known.
constexpr int MG_THREADS = 4 * MOG_D;
constexpr int MG_PARTS = MG_THREADS / MOG_D;
__global__ void __launch_bounds__(MG_THREADS) k_mog_merge(const float *partials, int P, int G,
                                                          float *out, int warm, const float *fmv,
                                                          const float *fmm) {
    const int g = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
    const int j = tid % MOG_D, part = tid / MOG_D;
    __shared__ float s_m[MAX_SPLITS], s_l[MAX_SPLITS];
    __shared__ float s_acc[MG_PARTS][MOG_D];
    auto src = [&](int i) { return partials + (((size_t)u * PART_SLOTS + i) * G + g) * PART_W; };
    // Pass 0 runs the same code on whatever the partials hold before the rows kernel has
    // finished (this kernel is launched early) and writes nothing: it brings the code into
    // the caches.  Pass 1 waits for the rows kernel and merges.
#pragma unroll 1
    for (int pass = warm ? 0 : 1; pass < 2; ++pass) {
    if (pass == 1) {
        pdl_wait();
        pdl_trigger();
    }
    float av[MAX_SPLITS / MG_PARTS];
#pragma unroll
    for (int q = 0; q < MAX_SPLITS / MG_PARTS; ++q) {
        const int i = part + q * MG_PARTS;
        av[q] = i < P ? __ldcg(src(i) + PART_ACC + j) : 0.f;
    }
    if (tid < P) {
        s_m[tid] = __ldcg(src(tid));
        s_l[tid] = __ldcg(src(tid) + 1);
    }
    // the feature-map residual (fmv non-null): one more state, T's vector minus the vectors
    // of the head's chosen subclusters, at the head's largest feature exponent
    float fden = 0.f, fnum = 0.f, fm2 = -INFINITY;
    if (fmv) {
        const float *fv = fmv + ((size_t)u * G + g) * (FM_NCH + 1) * FM_W;
        fden = __ldcg(fv + FM_NCH * FM_W + MOG_D);
        fnum = __ldcg(fv + FM_NCH * FM_W + j);
#pragma unroll 8
        for (int c = 0; c < FM_NCH; ++c) {
            fden -= __ldcg(fv + c * FM_W + MOG_D);
            fnum -= __ldcg(fv + c * FM_W + j);
        }
        if (fden > 0.f) fm2 = __ldcg(fmm + (size_t)u * G + g) * LOG2E;
    }
    __syncthreads();
    float mx = fm2;
    for (int i = 0; i < P; ++i) mx = fmaxf(mx, s_m[i]);
    float l = 0.f, v = 0.f;
    if (mx != -INFINITY) {
        for (int i = 0; i < P; ++i)
            if (s_m[i] != -INFINITY) l += exp2f(s_m[i] - mx) * s_l[i];
#pragma unroll
        for (int q = 0; q < MAX_SPLITS / MG_PARTS; ++q) {
            const int i = part + q * MG_PARTS;
            if (i < P && s_m[i] != -INFINITY) v += exp2f(s_m[i] - mx) * av[q];
        }
        if (fm2 != -INFINITY) {
            l += exp2f(fm2 - mx) * fden;
            if (part == 0) v += exp2f(fm2 - mx) * fnum;
        }
    }
    s_acc[part][j] = v;
    __syncthreads();
    if (part == 0) {
        for (int q = 1; q < MG_PARTS; ++q) v += s_acc[q][j];
        if (pass == 1) out[((size_t)u * G + g) * MOG_D + j] = l > 0.f ? v / l : 0.f;
    }
    }
}

// Append one token per sequence at position n_now[b], then advance n_now[b].
__global__ void k_append(Dev dv, const uint16_t *kn, const uint16_t *vn) {
    const int b = blockIdx.x;
    const int pos = dv.n_now[b];
    for (int e = threadIdx.x; e < dv.h_kv * 16; e += blockDim.x) {
        const int h = e / 16, ch = e % 16;
        const size_t src = ((size_t)b * dv.h_kv + h) * MOG_D + ch * 8;
        const int64_t ro = dv.row_off(b, h, pos);
        uint16_t *kd = dv.Kw + ro + ch * 8;
        uint16_t *vd = dv.Vw + ro + ch * 8;
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
    const bool fm = dv.residual == MOG_RESIDUAL_FEATURE_MAP;
    if (fm && (e = launch_fm_resid(dv, a.q, a.SW, s)) != cudaSuccess) return e;  // (timed with the rows)
    const void *rows_fn = dv.bt ? (const void *)k_mog_rows<GT, true> : (const void *)k_mog_rows<GT, false>;
    if ((e = ensure_smem(rows_fn, RW_SMEM)) != cudaSuccess) return e;
    if (dv.bt)
        e = launch_pdl(k_mog_rows<GT, true>, dim3(dv.P, dv.units), dim3(AT_THREADS), RW_SMEM, s, a);
    else
        e = launch_pdl(k_mog_rows<GT, false>, dim3(dv.P, dv.units), dim3(AT_THREADS), RW_SMEM, s, a);
    if (e != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[2], s)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_mog_merge, dim3(dv.G, dv.units), dim3(MG_THREADS), 0, s,
                        (const float *)dv.partials, dv.P, dv.G, a.out, a.warm,
                        (const float *)(fm ? dv.fm_vec : nullptr), (const float *)(fm ? dv.fm_mref : nullptr))) !=
        cudaSuccess)
        return e;
    if (events && (e = cudaEventRecord(events[3], s)) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_decode(const Dev &dv, const Plan &pl, const void *q, float *out,
                          const int32_t *sel_in, int32_t *sel_out, cudaStream_t s,
                          cudaEvent_t const *events) {
    DecArgs a;
    a.dv = dv;
    // with events between the kernels none starts before its predecessor ends, so the
    // warm-up passes would only add time
    a.warm = events ? 0 : 1;
    a.q = static_cast<const uint16_t *>(q);
    a.out = out;
    a.sel_in = sel_in;
    a.SW = dv.tc + dv.tc * dv.ts;
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

size_t slot_smem_bytes(int G, int c_max, int l_max, int tc) {  // the smallest layout (16-CTA clusters)
    return (size_t)md_layout(G, tc, c_max, 16, md_warps(G <= 4 ? 4 : 16)).total;
}

cudaError_t launch_append(const Dev &dv, const Plan &pl, const void *k_new, const void *v_new,
                          cudaStream_t s) {
    k_append<<<pl.batch, 128, 0, s>>>(dv, static_cast<const uint16_t *>(k_new),
                                      static_cast<const uint16_t *>(v_new));
    return cudaGetLastError();
}

}  // namespace mog
