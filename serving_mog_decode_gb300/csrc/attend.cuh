// attend.cuh -- split-KV online-softmax attention over 64-row tiles of a bf16 KV cache,
// shared by the full-scan kernel and the MoG exact-attention kernel.
//
// One CTA = 4 warps.  Rows (keys) are copied into shared memory with 16-byte cp.async,
// three stages deep, in a layout whose 16-byte chunks are XOR-swizzled by (row & 7) so
// that ldmatrix reads are bank-conflict free.  Warp w owns rows 16w..16w+15 of every
// tile and keeps its own running (max, sum, output) for the G query heads of the KV head.
// The keys sit in the M dimension of an m16n8k16 bf16 mma and the heads in N (8 per
// block), so no MMA row is padding:
//  - logits S^T = K Q^T: A = K tile, B = Q^T (bf16, exact), fp32 accumulate;
//  - weights P = 2^(S*tau*log2e - m), split into bf16 hi + lo parts (16-bit precision)
//    so the product O^T += V^T P^T (fp32 accumulate) keeps ~2^-17 relative weight error;
//  - a per-row head mask removes heads for which a row is not selected (logit -inf).
#pragma once

#include "common.cuh"

namespace mog {

constexpr int AT_WARPS = 4;
constexpr int AT_THREADS = AT_WARPS * 32;
constexpr int AT_ROWS = 64;
constexpr int AT_STAGES = 3;
constexpr int AT_ROW_BYTES = MOG_D * 2;               // 256
constexpr int AT_TILE_BYTES = AT_ROWS * AT_ROW_BYTES;  // 16 KB (K or V)
constexpr int AT_STAGE_BYTES = 2 * AT_TILE_BYTES + AT_ROWS * 4;
constexpr int AT_SMEM = AT_STAGES * AT_STAGE_BYTES;
constexpr float LOG2E = 1.4426950408889634f;

// Per-warp running state for the G query heads of a KV head, in the transposed layout of
// the P.V product: O^T (dimensions x heads) = V^T (dimensions x keys) . P^T (keys x heads).
// NB blocks of 8 heads (N = 8 per mma).  Lane l holds, for head block nb and dimension
// tile mt (16 dimensions), dimensions mt*16 + l/4 (+8) of heads nb*8 + (l%4)*2 (+1).
template <int NB>
struct WarpAcc {
    float o[NB][8][4];
    float m[NB][2];  // running max (log2 domain) of heads nb*8 + (l%4)*2, +1
    float l[NB][2];  // this lane's share of their running sums
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[nb][t][e] = 0.f;
            m[nb][0] = m[nb][1] = -INFINITY;
            l[nb][0] = l[nb][1] = 0.f;
        }
    }
};

// Q^T as mma B fragments (k = dimensions, n = heads) for the 8 k-steps of d = 128:
// b[nb][ks] = {Q[h][k0], Q[h][k0+1]}, {Q[h][k0+8], Q[h][k0+9]} with h = nb*8 + l/4,
// k0 = 16ks + (l%4)*2; heads >= G are zero.
template <int NB>
struct QFrags {
    uint32_t b[NB][8][2];
};
template <int NB>
__device__ __forceinline__ void load_q_frags(QFrags<NB> &qf, const uint16_t *q, int G) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int h = nb * 8 + (lane >> 2);
        const uint32_t *qr = reinterpret_cast<const uint32_t *>(q + (size_t)h * MOG_D);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int k0 = ks * 16 + (lane & 3) * 2;
            qf.b[nb][ks][0] = h < G ? qr[k0 / 2] : 0u;
            qf.b[nb][ks][1] = h < G ? qr[(k0 + 8) / 2] : 0u;
        }
    }
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * AT_ROW_BYTES + ((chunk ^ (row & 7)) << 4));
}

// Row addressing of the tile engine.  Contiguous (PAGED = false): row `pos` of a head's
// slab is at byte pos * row_bytes from the slab base (a 32-bit offset: the slab is below
// 4 GB).  Paged: `pos` is a physical row, (page << pshift) | row-in-page, at
// page * page_bytes + row * row_bytes from the base (64-bit).
template <bool PAGED>
struct RowAddr {
    uint32_t row_bytes;
    int pshift;
    int64_t page_bytes;
    __device__ __forceinline__ uint64_t off(int64_t pos) const {
        if (!PAGED) return (uint32_t)pos * row_bytes;
        return (uint64_t)(pos >> pshift) * (uint64_t)page_bytes +
               (uint32_t)(pos & ((1 << pshift) - 1)) * row_bytes;
    }
};

// Issue the copies of one tile: rows r < nrows come from krow/vrow(pos(r)); others are
// zero-filled with mask 0.  `posf(r, &pos, &mask)` supplies row positions.
template <bool PAGED, typename RowFn>
__device__ __forceinline__ void issue_tile(uint8_t *stage, int nrows, const uint16_t *kbase,
                                           const uint16_t *vbase, const RowAddr<PAGED> &ra, RowFn posf) {
    uint32_t *smask = reinterpret_cast<uint32_t *>(stage + 2 * AT_TILE_BYTES);
    const uint32_t sk = smem_u32(stage), sv = sk + AT_TILE_BYTES;
    const int tid = threadIdx.x;
    // each thread: rows tid/16 + 8i, chunk tid%16
    const int ch = tid & 15;
#pragma unroll
    for (int i = 0; i < AT_ROWS / 8; ++i) {
        const int r = (tid >> 4) + 8 * i;
        int64_t pos = 0;
        uint32_t mk = 0;
        const bool ok = r < nrows;
        if (ok) posf(r, pos, mk);
        const uint64_t off = ok ? ra.off(pos) + ch * 16 : 0u;
        const uint16_t *ks = reinterpret_cast<const uint16_t *>(reinterpret_cast<const char *>(kbase) + off);
        const uint16_t *vs = reinterpret_cast<const uint16_t *>(reinterpret_cast<const char *>(vbase) + off);
        cp_async16(sk + swz(r, ch), ks, ok ? 16 : 0);
        cp_async16(sv + swz(r, ch), vs, ok ? 16 : 0);
        if (ch == 0) smask[r] = ok ? mk : 0u;
    }
}

// Consume 16 rows (keys) rbase..rbase+15 of a shared-memory K/V block into this warp's
// accumulator.  sk, sv: shared addresses of the swizzled K and V rows; smask: per-row head
// masks (bit g set: head g attends to the row).
//  - logits S^T = K Q^T: keys in M (16), heads in N (8 per block), fp32 accumulate;
//  - weights P = 2^(S*tau*log2e - m), split into bf16 high + low parts; each 8 x 8 block
//    is transposed in registers (movmatrix) into the B operand of O^T += V^T P^T.
// GIVEN: the block holds precomputed terms instead of keys: row pairs (2i, 2i+1) are the
// bf16 high and low parts of a value vector, and `given` holds their log2-domain logits
// E[i][16] (16 heads per item), used as they are.
template <int NB, bool GIVEN = false>
__device__ __forceinline__ void compute_rows16(WarpAcc<NB> &acc, const QFrags<NB> &qf, uint32_t sk,
                                               uint32_t sv, const uint32_t *smask, int rbase,
                                               float scale2, const float *given = nullptr) {
    const int lane = threadIdx.x & 31;
    const int mat = lane >> 3, r8 = lane & 7;
    float s[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nb][e] = 0.f;
    if (!GIVEN) {
        const int key = rbase + (mat & 1) * 8 + r8;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t a[4];
            ldsm_x4(sk + swz(key, 2 * ks + (mat >> 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16(s[nb], a, qf.b[nb][ks][0], qf.b[nb][ks][1]);
        }
    }
    const int kA = rbase + (lane >> 2), kB = kA + 8;  // this lane's keys
    const uint32_t mkA = smask[kA], mkB = smask[kB];
    uint32_t bhi[NB][2], blo[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int hh = nb * 8 + (lane & 3) * 2;  // this lane's heads hh, hh + 1
        if (GIVEN) {
            s[nb][0] = ((mkA >> hh) & 1u) ? given[(kA >> 1) * MOG_MAX_G + hh] : -INFINITY;
            s[nb][1] = ((mkA >> (hh + 1)) & 1u) ? given[(kA >> 1) * MOG_MAX_G + hh + 1] : -INFINITY;
            s[nb][2] = ((mkB >> hh) & 1u) ? given[(kB >> 1) * MOG_MAX_G + hh] : -INFINITY;
            s[nb][3] = ((mkB >> (hh + 1)) & 1u) ? given[(kB >> 1) * MOG_MAX_G + hh + 1] : -INFINITY;
        } else {
            s[nb][0] = ((mkA >> hh) & 1u) ? s[nb][0] * scale2 : -INFINITY;
            s[nb][1] = ((mkA >> (hh + 1)) & 1u) ? s[nb][1] * scale2 : -INFINITY;
            s[nb][2] = ((mkB >> hh) & 1u) ? s[nb][2] * scale2 : -INFINITY;
            s[nb][3] = ((mkB >> (hh + 1)) & 1u) ? s[nb][3] * scale2 : -INFINITY;
        }
        // per-head maximum over the 16 keys: the 8 lanes that share l%4
        float mx0 = fmaxf(s[nb][0], s[nb][2]), mx1 = fmaxf(s[nb][1], s[nb][3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(acc.m[nb][0], mx0), mn1 = fmaxf(acc.m[nb][1], mx1);
        const float al0 = mn0 == -INFINITY ? 1.f : ex2(acc.m[nb][0] - mn0);
        const float al1 = mn1 == -INFINITY ? 1.f : ex2(acc.m[nb][1] - mn1);
        acc.m[nb][0] = mn0;
        acc.m[nb][1] = mn1;
        const float p0 = mn0 == -INFINITY ? 0.f : ex2(s[nb][0] - mn0);
        const float p1 = mn1 == -INFINITY ? 0.f : ex2(s[nb][1] - mn1);
        const float p2 = mn0 == -INFINITY ? 0.f : ex2(s[nb][2] - mn0);
        const float p3 = mn1 == -INFINITY ? 0.f : ex2(s[nb][3] - mn1);
        // a given term's low-part row (odd key) adds no weight of its own
        const bool wA = !GIVEN || !(kA & 1);
        acc.l[nb][0] = acc.l[nb][0] * al0 + (wA ? p0 + p2 : 0.f);
        acc.l[nb][1] = acc.l[nb][1] * al1 + (wA ? p1 + p3 : 0.f);
        if (al0 != 1.f || al1 != 1.f) {  // the running max moved: rescale the output
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                acc.o[nb][t][0] *= al0;
                acc.o[nb][t][1] *= al1;
                acc.o[nb][t][2] *= al0;
                acc.o[nb][t][3] *= al1;
            }
        }
        const uint32_t hA = cvt_bf2(p0, p1), hB = cvt_bf2(p2, p3);
        const uint32_t lA = cvt_bf2(p0 - bf_lo(hA), p1 - bf_hi(hA));
        const uint32_t lB = cvt_bf2(p2 - bf_lo(hB), p3 - bf_hi(hB));
        bhi[nb][0] = movmatrix_t(hA);
        bhi[nb][1] = movmatrix_t(hB);
        blo[nb][0] = movmatrix_t(lA);
        blo[nb][1] = movmatrix_t(lB);
    }
    {
        const int key = rbase + (mat >> 1) * 8 + r8;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(sv + swz(key, 2 * mt + (mat & 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                mma_bf16(acc.o[nb][mt], a, bhi[nb][0], bhi[nb][1]);
                mma_bf16(acc.o[nb][mt], a, blo[nb][0], blo[nb][1]);
            }
        }
    }
}

// Consume one 64-row tile (already in shared memory): warp w takes rows 16w..16w+15.
// GIVEN: the tile holds precomputed terms whose logits sit at the start of the stage.
template <int NB, bool GIVEN = false>
__device__ __forceinline__ void compute_tile(WarpAcc<NB> &acc, const QFrags<NB> &qf,
                                             const uint8_t *stage, float scale2) {
    const uint32_t sk = smem_u32(stage);
    compute_rows16<NB, GIVEN>(acc, qf, sk, sk + AT_TILE_BYTES,
                              reinterpret_cast<const uint32_t *>(stage + 2 * AT_TILE_BYTES),
                              (threadIdx.x >> 5) * 16, scale2, reinterpret_cast<const float *>(stage));
}

// Partial result layout: per head, [0] = m (log2 domain), [1] = l, [2], [3] unused,
// [4 .. 4+d) = acc; 528 bytes, so that every partial is a whole number of 16-byte chunks.
constexpr int PART_W = MOG_D + 4;
constexpr int PART_ACC = 4;

// Write this warp's state for heads < G into st[w][g][PART_W] (shared memory).
template <int NB>
__device__ __forceinline__ void warp_state_out(const WarpAcc<NB> &acc, float *st, int G) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float *b = st + (size_t)w * G * PART_W;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        float l0 = acc.l[nb][0], l1 = acc.l[nb][1];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        }
        const int hh = nb * 8 + (lane & 3) * 2, d0 = lane >> 2;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = hh + e;
            if (h >= G) continue;
            float *r = b + h * PART_W;
            if (d0 == 0) {
                r[0] = acc.m[nb][e];
                r[1] = e ? l1 : l0;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                r[PART_ACC + t * 16 + d0] = acc.o[nb][t][e];
                r[PART_ACC + t * 16 + d0 + 8] = acc.o[nb][t][e + 2];
            }
        }
    }
}

// Merge n states st[i][g][PART_W] held in shared memory (stride per state G*PART_W
// floats) into dst[g][PART_W] (shared or global).  Called by all threads of the CTA.
__device__ __forceinline__ void merge_states(const float *st, int n, int G, float *dst) {
    for (int e = threadIdx.x; e < G * MOG_D; e += blockDim.x) {
        const int g = e / MOG_D, j = e % MOG_D;
        float m = -INFINITY;
        for (int i = 0; i < n; ++i) m = fmaxf(m, st[((size_t)i * G + g) * PART_W]);
        float l = 0.f, a = 0.f;
        if (m != -INFINITY) {
            for (int i = 0; i < n; ++i) {
                const float *r = st + ((size_t)i * G + g) * PART_W;
                if (r[0] == -INFINITY) continue;
                const float sc = exp2f(r[0] - m);
                l += sc * r[1];
                a += sc * r[PART_ACC + j];
            }
        }
        float *o = dst + (size_t)g * PART_W;
        if (j == 0) {
            o[0] = m;
            o[1] = l;
        }
        o[PART_ACC + j] = a;
    }
}

// Merge n partials part[i][g][PART_W] from global memory and write the normalised
// result out[g][d] (= acc / l).  The partials are staged into shared memory `sm`
// (sm_floats floats, >= G*PART_W + G*(n_chunk+2)) with cp.async, all copies of a chunk in
// flight at once, and folded into a running (max, sum, acc) per head.
__device__ __forceinline__ void merge_global_out(const float *part, int n, int G, float *sm,
                                                 int sm_floats, float *out) {
    const int per = G * PART_W;
    int ch = (sm_floats - 3 * MOG_MAX_G) / (per + G);
    ch = ch < 1 ? 1 : ch;
    float *stage = sm;                        // [ch][G][PART_W]
    float *sS = stage + (size_t)ch * per;     // [ch][G] per-partial scales
    float *sM = sS + (size_t)ch * G;          // [G] running max
    float *sL = sM + MOG_MAX_G;               // [G] running sum
    float *sA = sL + MOG_MAX_G;               // [G] rescale of the running acc
    if (threadIdx.x < (unsigned)G) {
        sM[threadIdx.x] = -INFINITY;
        sL[threadIdx.x] = 0.f;
    }
    float acc[MOG_MAX_G * MOG_D / 128];  // elements e = tid + k*blockDim, blockDim >= 128
    const int ept = (G * MOG_D + blockDim.x - 1) / blockDim.x;
    for (int k = 0; k < ept; ++k) acc[k] = 0.f;
    for (int c0 = 0; c0 < n; c0 += ch) {
        const int cnt = min(ch, n - c0);
        const int q4 = cnt * per / 4;
        const float *src = part + (size_t)c0 * per;
        for (int q = threadIdx.x; q < q4; q += blockDim.x) cp_async16(smem_u32(stage + 4 * q), src + 4 * q, 16);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        if (threadIdx.x < (unsigned)G) {
            const int g = threadIdx.x;
            float mn = sM[g];
            for (int i = 0; i < cnt; ++i) mn = fmaxf(mn, stage[(size_t)i * per + g * PART_W]);
            float lsum = 0.f;
            for (int i = 0; i < cnt; ++i) {
                const float mi = stage[(size_t)i * per + g * PART_W];
                const float sc = (mi == -INFINITY) ? 0.f : exp2f(mi - mn);
                sS[i * G + g] = sc;
                lsum += sc * stage[(size_t)i * per + g * PART_W + 1];
            }
            const float so = (sM[g] == -INFINITY) ? 0.f : exp2f(sM[g] - mn);
            sA[g] = so;
            sL[g] = sL[g] * so + lsum;
            sM[g] = mn;
        }
        __syncthreads();
        for (int k = 0; k < ept; ++k) {
            const int e = threadIdx.x + k * blockDim.x;
            if (e >= G * MOG_D) break;
            const int g = e / MOG_D, j = e % MOG_D;
            float a = acc[k] * sA[g];
            for (int i = 0; i < cnt; ++i) a += sS[i * G + g] * stage[(size_t)i * per + g * PART_W + PART_ACC + j];
            acc[k] = a;
        }
        __syncthreads();
    }
    for (int k = 0; k < ept; ++k) {
        const int e = threadIdx.x + k * blockDim.x;
        if (e >= G * MOG_D) break;
        const int g = e / MOG_D;
        out[e] = sL[g] > 0.f ? acc[k] / sL[g] : 0.f;
    }
}

}  // namespace mog
