// dense.cu -- full-scan exact decode attention, the comparison path: every query head
// attends to all N_b keys of its KV head (softmax(tau q.K^T) V, tau = 1/sqrt(d)).
// "Iceberg Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians",
// Abstract: decoding over a long context normally scans the whole KV cache; this is that
// scan.  Split-KV: each (KV head, split) CTA streams a contiguous key range through the
// attention engine and writes a partial (max, sum, acc); a second kernel merges them.
#include <cuda.h>
#include <stdio.h>

#include <map>
#include <mutex>

#include "attend.cuh"
#include "internal.h"

namespace mog {
// Two tile stages (74.6 KB of shared memory a CTA) and three CTAs per SM, as the MoG rows
// kernel: measured 1.7% faster at 1M and 6% at 128K than three stages at two per SM.
constexpr int DN_STAGES = 2;
constexpr int DN_SMEM = DN_STAGES * AT_STAGE_BYTES;

struct DenseArgs {
    const uint16_t *K, *V;
    int64_t sb, sh, sn;
    const int *bt;  // block table of a paged cache, or null
    int pshift, pps;
    const int32_t *lengths;
    int h_kv, G, splits;
    const uint16_t *q;
    float *out, *part;  // part: [units][splits][G][PART_W]
    float scale2;
};

// NB: blocks of 8 query heads per KV head (1 for G <= 8, else 2); PAGED: a block-table cache
template <int NB, bool PAGED>
__global__ void __launch_bounds__(AT_THREADS) k_dense_split(DenseArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    const int u = blockIdx.y, p = blockIdx.x;
    const int b = u / a.h_kv, h = u % a.h_kv;
    const int n = a.lengths[b];
    // contiguous split of [0, n) into `splits` ranges of whole tiles
    const int64_t ntile = ceil_div64(n, AT_ROWS);
    const int64_t t0 = ntile * p / a.splits, t1 = ntile * (p + 1) / a.splits;
    const int64_t lo = t0 * AT_ROWS, hi = min((int64_t)n, t1 * AT_ROWS);
    const int nt = (int)(t1 - t0);
    const uint16_t *kb = a.K + (PAGED ? 0 : b * a.sb) + h * a.sh;
    const uint16_t *vb = a.V + (PAGED ? 0 : b * a.sb) + h * a.sh;
    const RowAddr<PAGED> ra{(uint32_t)(a.sn * 2), a.pshift, a.sb * 2};
    const int *btb = PAGED ? a.bt + (int64_t)b * a.pps : nullptr;
    const uint32_t allm = a.G >= 32 ? 0xffffffffu : ((1u << a.G) - 1u);
    QFrags<NB> qf;
    load_q_frags(qf, a.q + ((int64_t)b * a.h_kv * a.G + (int64_t)h * a.G) * MOG_D, a.G);
    WarpAcc<NB> acc;
    acc.init();
    auto issue = [&](int t) {
        const int64_t r0 = lo + (int64_t)t * AT_ROWS;
        const int nr = (int)min((int64_t)AT_ROWS, hi - r0);
        issue_tile(dsm + (t % DN_STAGES) * AT_STAGE_BYTES, nr, kb, vb, ra,
                   [&](int r, int64_t &pos, uint32_t &mk) {
                       pos = r0 + r;
                       if (PAGED)  // physical row: (page << pshift) | row in page
                           pos = ((int64_t)__ldg(btb + (pos >> a.pshift)) << a.pshift) |
                                 (pos & ((1 << a.pshift) - 1));
                       mk = allm;
                   });
    };
#pragma unroll
    for (int s = 0; s < DN_STAGES - 1; ++s) {
        if (s < nt) issue(s);
        cp_async_commit();
    }
    for (int t = 0; t < nt; ++t) {
        cp_async_wait<DN_STAGES - 2>();
        __syncthreads();
        if (t + DN_STAGES - 1 < nt) issue(t + DN_STAGES - 1);
        cp_async_commit();
        compute_tile(acc, qf, dsm + (t % DN_STAGES) * AT_STAGE_BYTES, a.scale2);
    }
    cp_async_wait<0>();
    __syncthreads();
    float *st = reinterpret_cast<float *>(dsm);
    warp_state_out(acc, st, a.G);
    __syncthreads();
    merge_states(st, AT_WARPS, a.G, a.part + ((int64_t)u * a.splits + p) * a.G * PART_W);
}

constexpr int MERGE_THREADS = 256;
constexpr int MERGE_SMEM = 96 * 1024;

__global__ void __launch_bounds__(MERGE_THREADS) k_dense_merge(DenseArgs a) {
    extern __shared__ __align__(16) float mg[];
    const int u = blockIdx.x;
    merge_global_out(a.part + (int64_t)u * a.splits * a.G * PART_W, a.splits, a.G, mg,
                     MERGE_SMEM / 4, a.out + (int64_t)u * a.G * MOG_D);
}

int dense_splits(int units, int n_max) {
    // enough CTAs for two per SM, no split shorter than 8 tiles
    const int want = (int)ceil_div64(3 * num_sms(), units);
    const int64_t bl = ceil_div64(n_max, 8 * AT_ROWS);
    const int by_len = bl < 1 ? 1 : (int)bl;
    return max(1, min(want, by_len));
}

cudaError_t launch_dense(const mog_kv *kv, const int32_t *lengths, int n_max, int batch, int h_kv,
                         int G, const void *q, float *out, float *scratch, int splits,
                         cudaStream_t s) {
    const bool pg = kv->block_table != nullptr;
    const void *split_fn = G <= 8 ? (pg ? (const void *)k_dense_split<1, true> : (const void *)k_dense_split<1, false>)
                                  : (pg ? (const void *)k_dense_split<2, true> : (const void *)k_dense_split<2, false>);
    cudaError_t e = ensure_smem(split_fn, DN_SMEM);
    if (e == cudaSuccess) e = ensure_smem((const void *)k_dense_merge, MERGE_SMEM);
    if (e != cudaSuccess) return e;
    DenseArgs a{static_cast<const uint16_t *>(kv->k), static_cast<const uint16_t *>(kv->v),
                kv->stride_b, kv->stride_h, kv->stride_n, kv->block_table,
                kv->block_table ? log2_exact(kv->page_rows) : 0, kv->block_table ? kv->pages_per_seq : 0,
                lengths, h_kv, G, splits, static_cast<const uint16_t *>(q), out, scratch,
                (float)(LOG2E / sqrt((double)MOG_D))};
    const int U = batch * h_kv;
    if (G <= 8 && !pg) k_dense_split<1, false><<<dim3(splits, U), AT_THREADS, DN_SMEM, s>>>(a);
    else if (G <= 8) k_dense_split<1, true><<<dim3(splits, U), AT_THREADS, DN_SMEM, s>>>(a);
    else if (!pg) k_dense_split<2, false><<<dim3(splits, U), AT_THREADS, DN_SMEM, s>>>(a);
    else k_dense_split<2, true><<<dim3(splits, U), AT_THREADS, DN_SMEM, s>>>(a);
    k_dense_merge<<<U, MERGE_THREADS, MERGE_SMEM, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// dense_decode_noalloc: dense_decode with its partial results in a fixed device array that
// the library owns, for callers that cannot allocate device memory.
// ------------------------------------------------------------------------------------

// Scratch for the split partials of dense_decode_noalloc.  Every GPU that loads the library
// keeps this array until the process exits.
constexpr size_t DENSE_STATIC_BYTES = 4u << 20;
static __device__ __align__(256) float g_dense_static[DENSE_STATIC_BYTES / sizeof(float)];

// The CUDA context current on the calling thread, as a process-unique id, through the
// runtime's driver entry points (false if there is none or the driver cannot say).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
static bool current_context_id(unsigned long long *id) {
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
    });
    CUcontext c = nullptr;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c) return false;
    return get_id(c, id) == CUDA_SUCCESS;
}

// Device address of g_dense_static in the current context.  In host code the symbol is
// only a stand-in, never an address a kernel may use.  The address belongs to the module
// loaded in one context: it is asked for once per context (the first call on a device,
// with that device current, and again after a device reset makes a new context) and
// cached under the context's id.  If the context cannot be identified the address is
// asked for on every call.
cudaError_t dense_static_scratch(float **ptr, size_t *bytes) {
    static std::mutex mu;
    static std::map<unsigned long long, float *> addr;
    *bytes = DENSE_STATIC_BYTES;
    unsigned long long id = 0;
    std::lock_guard<std::mutex> lk(mu);
    if (current_context_id(&id)) {
        auto it = addr.find(id);
        if (it != addr.end()) {
            *ptr = it->second;
            return cudaSuccess;
        }
    }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_dense_static);  // makes the context if needed
    if (e != cudaSuccess) return e;
    *ptr = static_cast<float *>(p);
    if (current_context_id(&id)) addr[id] = *ptr;
    return cudaSuccess;
}

}  // namespace mog
