// api.cu -- the C ABI of libmog (declared in mog.h): argument validation, the arena
// layout, and the launch sequences.  No entry point allocates device memory.
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace mog;

struct mog_handle {
    Plan plan;
    Dev dev;
    mog_kv kv;
    char *arena;
    std::vector<int32_t> lengths;
    std::vector<int32_t> info;  // host copy of unit_info
    int appended;
    bool fm_ready;  // mog_feature_map has run (the feature-map residual can decode)
};

static thread_local char g_err[256] = "";

static int cuda_fail(cudaError_t e, const char *where) {
    snprintf(g_err, sizeof g_err, "%s: %s", where, cudaGetErrorString(e));
    return MOG_ERR_CUDA;
}
#define CK(call)                                              \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);   \
    } while (0)

namespace mog {

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

// The attribute is an upper bound, so it only ever grows: a launch that needs less than
// the largest value set so far for (kernel, device) needs no call.
cudaError_t ensure_smem(const void *fn, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> top;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    size_t &cur = top[std::make_pair(fn, dev)];
    if (bytes <= cur) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) cur = bytes;
    return e;
}

static int isqrt_round(int64_t n) {
    int64_t c = (int64_t)sqrt((double)n);
    while (c * c > n) --c;
    while ((c + 1) * (c + 1) <= n) ++c;
    return (int)(n - c * c > c ? c + 1 : c);  // round(sqrt(n)); a tie cannot occur
}
static int ceil_log2(int64_t n) {
    int l = 0;
    while (((int64_t)1 << l) < n) ++l;
    return l;
}

void unit_clusters(const mog_params *p, int n, int *C, int *L) {
    *C = std::max(1, p->n_clusters > 0 ? p->n_clusters : isqrt_round(n));
    *L = std::max(1, p->n_sub > 0 ? p->n_sub : ceil_log2(n));
}

static int64_t al(int64_t x) { return (x + 255) & ~(int64_t)255; }

int make_plan(const mog_params *p, const int32_t *lengths_host, Plan *pl) {
    if (!p || !lengths_host || !pl) return MOG_ERR_INVALID_ARG;
    const int known_flags = MOG_FLAG_UNION_EXACT | MOG_FLAG_SLIDING | MOG_FLAG_GROUP_SELECT |
                            MOG_FLAG_BF16_SUMMARIES | MOG_FLAG_FP8_SUMMARIES | MOG_FLAG_KMEANSPP;
    if ((p->flags & MOG_FLAG_BF16_SUMMARIES) && (p->flags & MOG_FLAG_FP8_SUMMARIES))
        return MOG_ERR_INVALID_ARG;
    if ((p->flags & ~known_flags) != 0 || p->batch <= 0 || p->h_kv <= 0 || p->h_q <= 0 || p->n_cap <= 0 ||
        p->top_c < 0 || p->top_s < 0 || p->n_sink < 0 || p->n_recent < 0 || p->iters_l1 < 0 ||
        p->iters_l2 < 0 || p->n_clusters < 0 || p->n_sub < 0 ||
        (p->score_mode != 0 && p->score_mode != 1) || p->residual < 0 || p->residual > 2)
        return MOG_ERR_INVALID_ARG;
    // the feature-map residual subtracts each head's own chosen subclusters from fixed sums:
    // neither the union's rows nor keys moved by the sliding window are in those sums
    if (p->residual == MOG_RESIDUAL_FEATURE_MAP && (p->flags & (MOG_FLAG_UNION_EXACT | MOG_FLAG_SLIDING)))
        return MOG_ERR_INVALID_ARG;
    if (p->d != MOG_D || p->h_q % p->h_kv != 0 || p->h_q / p->h_kv > MOG_MAX_G)
        return MOG_ERR_SHAPE;
    Plan &P = *pl;
    memset(&P, 0, sizeof P);
    P.batch = p->batch;
    P.h_kv = p->h_kv;
    P.h_q = p->h_q;
    P.G = p->h_q / p->h_kv;
    P.d = p->d;
    P.n_cap = p->n_cap;
    P.units = p->batch * p->h_kv;
    P.tc = p->top_c;
    P.ts = p->top_s;
    P.T1 = p->iters_l1 > 0 ? p->iters_l1 : 10;
    P.T2 = p->iters_l2 > 0 ? p->iters_l2 : 10;
    P.score_mode = p->score_mode;
    P.residual = p->residual;
    P.union_exact = (p->flags & MOG_FLAG_UNION_EXACT) ? 1 : 0;
    P.sliding = (p->flags & MOG_FLAG_SLIDING) ? 1 : 0;
    P.group_select = (p->flags & MOG_FLAG_GROUP_SELECT) ? 1 : 0;
    P.bf16s = (p->flags & MOG_FLAG_BF16_SUMMARIES) ? 1 : 0;
    P.fp8s = (p->flags & MOG_FLAG_FP8_SUMMARIES) ? 1 : 0;
    P.kpp = (p->flags & MOG_FLAG_KMEANSPP) ? 1 : 0;
    P.R = p->n_recent;
    P.c_max = P.l_max = 1;
    P.n_mid_max = 0;
    for (int b = 0; b < p->batch; ++b) {
        const int n = lengths_host[b];
        if (n < 1 || n > p->n_cap) return MOG_ERR_SHAPE;
        int C, L;
        unit_clusters(p, n, &C, &L);
        P.c_max = std::max(P.c_max, C);
        P.l_max = std::max(P.l_max, L);
        P.n_mid_max = std::max(P.n_mid_max, std::max(0, n - p->n_recent - p->n_sink));
    }
    if (P.l_max > MOG_MAX_L || P.c_max > MAX_C || P.ts > MOG_MAX_L) return MOG_ERR_SHAPE;
    if (std::min(P.c_max, P.G * P.tc) > MOG_MAX_UNION || P.tc > MOG_MAX_UNION) return MOG_ERR_SHAPE;
    if (slot_smem_bytes(P.G, P.c_max, P.l_max, P.tc) > 226 * 1024) return MOG_ERR_SHAPE;  // decode shared memory
    const int sms = num_sms();
    // rows kernel: one wave of three CTAs per SM; with so many units that a wave gives each
    // fewer than four CTAs, four per unit over several waves, which the CTA scheduler
    // balances across units of different lengths
    P.P = std::min(MAX_SPLITS, std::max(4, 3 * sms / P.units));
    // the sort workspace covers the longest mid region a later re-clustering can see
    P.nchunks = std::max(1, (int)ceil_div64(std::max(P.n_mid_max, p->n_cap - p->n_recent - p->n_sink),
                                            SORT_CHUNK));
    P.sub_off_stride = (P.c_max * P.l_max + 1 + 3) & ~3;
    const int64_t U = P.units, G = P.G, cm = P.c_max, lm = P.l_max, nc = P.n_cap;
    const int64_t SW = P.tc + P.tc * P.ts;
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        const int64_t r = o;
        o += al(std::max<int64_t>(bytes, 4));
        return r;
    };
    P.o_status = take(64);
    P.o_unit_info = take(4 * U * UI_STRIDE);
    P.o_n_now = take(4 * P.batch);
    P.o_perm = take(4 * U * nc);
    P.o_sub_off = take(4 * U * P.sub_off_stride);
    P.o_cl_n = take(4 * U * cm);
    P.o_cl_ms = take(4 * U * cm * 2 * MOG_D);
    P.o_cl_vbar = take(4 * U * cm * MOG_D);
    P.o_sub_n = take(4 * U * cm * lm);
    P.o_sub_ms = take(4 * U * cm * lm * 2 * MOG_D);
    P.o_sub_vbar = take(4 * U * cm * lm * MOG_D);
    P.o_cl_vhl = take(2 * U * cm * 2 * MOG_D);
    P.o_sub_vhl = take(2 * U * cm * lm * 2 * MOG_D);
    P.o_cl_ms16 = P.bf16s ? take(2 * U * cm * 2 * MOG_D) : 0;
    P.o_sub_ms16 = P.bf16s ? take(2 * U * cm * lm * 2 * MOG_D) : 0;
    P.o_cl_ms8 = P.fp8s ? take(U * cm * 2 * MOG_D) : 0;
    P.o_sub_ms8 = P.fp8s ? take(U * cm * lm * 2 * MOG_D) : 0;
    P.o_l1_assign = take(4 * U * nc);
    P.o_l1_steps = take(4 * U);
    P.o_cent = take(4 * U * cm * MOG_D);
    P.o_permA = take(4 * U * nc);
    P.o_changed = take(4 * U * P.T1);
    P.o_fb_list = take(4 * U * nc);
    P.o_fb_cnt = take(4 * U * P.T1);
    P.o_rc_list = take(4 * U * nc);
    P.o_rc_cnt = take(4 * U * P.T1);
    P.cimg_ustride = (int64_t)ceil_div64(cm, KM_CHUNK) * KM_IMG_CHUNK;
    P.cn_ustride = (int64_t)ceil_div64(cm, KM_CHUNK) * KM_CHUNK;
    P.o_cimg = take(2 * U * P.cimg_ustride);
    P.o_cnorm = take(4 * U * P.cn_ustride);
    P.o_hist = take(4 * U * P.nchunks * cm);
    P.o_offs = take(4 * U * P.nchunks * cm);
    P.o_ctot = take(4 * U * cm);
    P.o_coff = take(4 * U * (cm + 1));
    P.o_sub_assign = take(4 * U * nc);
    P.nseg_max = (int)std::max<int64_t>(1, std::min<int64_t>(cm, G * P.tc) * lm);  // union x subclusters
    P.o_partials = take(4 * U * PART_SLOTS * G * (MOG_D + 4));
    P.o_sel = take(4 * U * G * std::max<int64_t>(SW, 1));
    P.o_plan = take(4 * U * PLAN_W);
    P.o_segrow = take(4 * U * P.nseg_max);
    P.o_segoff = take(4 * U * P.nseg_max);
    P.o_segmask = take(4 * U * P.nseg_max);
    // residual items per unit: union pairs, then clusters; G exponents each (16-byte rows)
    P.resx_stride = (std::min<int64_t>(cm, G * std::max(P.tc, 1)) * lm + cm) * ((G + 3) & ~3LL);
    P.o_resx = take(4 * U * P.resx_stride);
    // k-means++ seeding: one CTA per PP_ROWS mid keys of the longest mid region a
    // re-clustering can see
    P.pp_nblk = P.kpp ? (int)ceil_div64(std::max<int64_t>(1, nc), PP_ROWS) : 0;
    P.o_pp_draw = P.kpp ? take(8 * U * cm) : 0;
    P.o_pp_idx = P.kpp ? take(4 * U * cm) : 0;
    P.o_pp_d2 = P.kpp ? take(4 * 2 * U * nc) : 0;
    P.o_pp_part = P.kpp ? take(8 * 2 * U * (int64_t)P.pp_nblk) : 0;
    const bool fm = P.residual == MOG_RESIDUAL_FEATURE_MAP;
    P.o_fm_omega = fm ? take(4 * FM_M * MOG_D) : 0;
    P.o_fm_mi = fm ? take(4 * FM_M) : 0;
    P.o_fm_z = fm ? take(4 * U * cm * lm * FM_M * FM_W) : 0;
    P.o_fm_zc = fm ? take(4 * U * cm * FM_M * FM_W) : 0;
    P.o_fm_t = fm ? take(4 * U * FM_M * FM_W) : 0;
    P.o_fm_vec = fm ? take(4 * U * G * (FM_NCH + 1) * FM_W) : 0;
    P.o_fm_mref = fm ? take(4 * U * G) : 0;
    P.total = o;
    return MOG_OK;
}

void trace_layout(const Plan &P, mog_trace_layout *t) {
    memset(t, 0, sizeof *t);
    t->units = P.units;
    t->iters_l1 = P.T1;
    t->iters_l2 = P.T2;
    t->c_max = P.c_max;
    t->l_max = P.l_max;
    t->d = MOG_D;
    t->n_mid = std::max(P.n_mid_max, 1);
    const int64_t U = P.units;
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        const int64_t r = o;
        o += al(std::max<int64_t>(bytes, 4));
        return r;
    };
    t->l1_cent = take(4 * U * P.T1 * P.c_max * MOG_D);
    t->l1_assign = take(4 * U * P.T1 * t->n_mid);
    t->l2_cent = take(4 * U * P.c_max * P.T2 * P.l_max * MOG_D);
    t->l2_assign = take(4 * U * P.T2 * t->n_mid);
    t->l2_steps = take(4 * U * P.c_max);
    t->bytes = o;
}

Dev make_dev(const Plan &P, void *arena, const mog_kv *kv) {
    Dev d;
    memset(&d, 0, sizeof d);
    char *a = static_cast<char *>(arena);
    d.K = static_cast<const uint16_t *>(kv->k);
    d.V = static_cast<const uint16_t *>(kv->v);
    d.Kw = static_cast<uint16_t *>(kv->k);
    d.Vw = static_cast<uint16_t *>(kv->v);
    d.sb = kv->stride_b;
    d.sh = kv->stride_h;
    d.sn = kv->stride_n;
    d.bt = kv->block_table;
    d.pshift = kv->block_table ? log2_exact(kv->page_rows) : 0;
    d.pps = kv->block_table ? kv->pages_per_seq : 0;
    d.batch = P.batch;
    d.h_kv = P.h_kv;
    d.G = P.G;
    d.units = P.units;
    d.n_cap = P.n_cap;
    d.c_max = P.c_max;
    d.l_max = P.l_max;
    d.tc = P.tc;
    d.ts = P.ts;
    d.T1 = P.T1;
    d.T2 = P.T2;
    d.score_mode = P.score_mode;
    d.residual = P.residual;
    d.union_exact = P.union_exact;
    d.group_select = P.group_select;
    d.bf16s = P.bf16s;
    d.fp8s = P.fp8s;
    d.kpp = P.kpp;
    d.pp_nblk = P.pp_nblk;
    d.P = P.P;
    d.nseg_max = P.nseg_max;
    d.cimg_ustride = P.cimg_ustride;
    d.cn_ustride = P.cn_ustride;
    d.resx_stride = P.resx_stride;
    d.nchunks = P.nchunks;
    d.sub_off_stride = P.sub_off_stride;
    d.tau = (float)(1.0 / sqrt((double)P.d));
#define PTR(name, T) d.name = reinterpret_cast<T *>(a + P.o_##name)
    PTR(unit_info, int);
    PTR(n_now, int);
    PTR(perm, int);
    PTR(sub_off, int);
    PTR(cl_n, int);
    PTR(sub_n, int);
    PTR(l1_assign, int);
    PTR(status, int);
    PTR(l1_steps, int);
    PTR(cl_ms, float);
    PTR(cl_vbar, float);
    PTR(sub_ms, float);
    PTR(sub_vbar, float);
    PTR(cl_vhl, uint16_t);
    PTR(sub_vhl, uint16_t);
    if (P.bf16s) {
        PTR(cl_ms16, uint16_t);
        PTR(sub_ms16, uint16_t);
    }
    if (P.fp8s) {
        PTR(cl_ms8, uint8_t);
        PTR(sub_ms8, uint8_t);
    }
    if (P.residual == MOG_RESIDUAL_FEATURE_MAP) {
        PTR(fm_omega, float);
        PTR(fm_mi, float);
        PTR(fm_z, float);
        PTR(fm_zc, float);
        PTR(fm_t, float);
        PTR(fm_vec, float);
        PTR(fm_mref, float);
    }
    if (P.kpp) {
        PTR(pp_draw, double);
        PTR(pp_idx, int);
        PTR(pp_d2, float);
        PTR(pp_part, double);
    }
    PTR(cent, float);
    PTR(permA, int);
    PTR(changed, int);
    PTR(fb_list, int);
    PTR(fb_cnt, int);
    PTR(rc_list, int);
    PTR(rc_cnt, int);
    PTR(cimg, uint16_t);
    PTR(cnorm, float);
    PTR(hist, int);
    PTR(offs, int);
    PTR(ctot, int);
    PTR(coff, int);
    PTR(sub_assign, int);
    PTR(partials, float);
    PTR(sel, int);
    PTR(plan, int);
    PTR(segrow, int);
    PTR(segoff, int);
    PTR(segmask, uint32_t);
    PTR(resx, float);
#undef PTR
    return d;
}

}  // namespace mog

// Partition sanity check for mog_build_from_partition: offsets monotone and complete,
// positions inside the unit's mid region.  Bad input sets the status word; the
// statistics kernel then skips the unit.
__global__ void k_check_partition(Dev dv) {
    const int u = blockIdx.x;
    const int *ui = dv.unit_info + u * UI_STRIDE;
    const int C = ui[UI_C], L = ui[UI_L], nm = ui[UI_NMID], S = ui[UI_S];
    const int *so = dv.sub_off + (size_t)u * dv.sub_off_stride;
    const int *pm = dv.perm + (size_t)u * dv.n_cap;
    bool bad = false;
    for (int g = threadIdx.x; g < C * L; g += blockDim.x)
        if (so[g] > so[g + 1]) bad = true;
    if (threadIdx.x == 0 && (so[0] != 0 || so[C * L] != nm)) bad = true;
    for (int i = threadIdx.x; i < nm; i += blockDim.x)
        if (pm[i] < S || pm[i] >= S + nm) bad = true;
    if (bad) flag_error(dv.status, ST_BAD_INDEX);
}

// ------------------------------------------------------------------------------- ABI

static const char *kNames[] = {"MOG_OK", "MOG_ERR_INVALID_ARG", "MOG_ERR_SHAPE",
                               "MOG_ERR_ARENA_TOO_SMALL", "MOG_ERR_CUDA", "MOG_ERR_DEVICE_CHECK",
                               "MOG_ERR_TIMEOUT", "MOG_ERR_NOT_IMPLEMENTED", "MOG_ERR_CAPACITY"};

extern "C" const char *mog_status_string(int status) {
    if (status < 0 || status >= (int)(sizeof kNames / sizeof kNames[0])) return "MOG_UNKNOWN_STATUS";
    return kNames[status];
}

extern "C" const char *mog_last_error(void) { return g_err; }

static bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

namespace mog {
int log2_exact(int x) {
    if (x <= 0 || (x & (x - 1))) return -1;
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}
}  // namespace mog

static int check_kv(const mog_kv *kv, int batch, int h_kv, int n_cap) {
    if (!kv || !kv->k || !kv->v) return MOG_ERR_INVALID_ARG;
    if (!aligned16(kv->k) || !aligned16(kv->v)) return MOG_ERR_INVALID_ARG;
    if (kv->stride_n < MOG_D || kv->stride_b < 0 || kv->stride_h < 0) return MOG_ERR_SHAPE;
    if ((kv->stride_n | kv->stride_b | kv->stride_h) & 7) return MOG_ERR_SHAPE;
    (void)batch;
    (void)h_kv;
    if (kv->block_table) {  // paged: whole pages of a power-of-two number of rows
        const int sh = log2_exact(kv->page_rows);
        if (sh < 4 || sh > 20 || kv->pages_per_seq <= 0) return MOG_ERR_SHAPE;
        if ((int64_t)kv->pages_per_seq * kv->page_rows < n_cap) return MOG_ERR_SHAPE;
        return MOG_OK;
    }
    // the attention kernels address a row inside its head's slab with a 32-bit byte offset
    if ((int64_t)n_cap * kv->stride_n * 2 >= (1LL << 32)) return MOG_ERR_SHAPE;
    return MOG_OK;
}

extern "C" int mog_arena_bytes(const mog_params *p, const int32_t *lengths_host, size_t *bytes) {
    if (!bytes) return MOG_ERR_INVALID_ARG;
    Plan pl;
    int st = make_plan(p, lengths_host, &pl);
    if (st != MOG_OK) return st;
    *bytes = (size_t)pl.total;
    return MOG_OK;
}

// One unit's row of unit_info for a build over the first n keys of its sequence.
static void set_unit_info(int32_t *r, int C, int L, int n, int S, int R, int b) {
    r[UI_C] = C;
    r[UI_L] = L;
    r[UI_NBUILD] = n;
    r[UI_NMID] = std::max(0, n - R - S);
    r[UI_S] = S;
    r[UI_RLO] = std::max(S, n - R);
    r[UI_B] = b;
}

// Upload the handle's unit_info and clear what a build accumulates into.
static cudaError_t reset_build_state(mog_handle *h, cudaStream_t s) {
    const Plan &pl = h->plan;
    char *a = h->arena;
    cudaError_t e = cudaMemcpyAsync(a + pl.o_unit_info, h->info.data(), h->info.size() * 4,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a + pl.o_changed, 0, 4 * (size_t)pl.units * pl.T1, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a + pl.o_fb_cnt, 0, 4 * (size_t)pl.units * pl.T1, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a + pl.o_rc_cnt, 0, 4 * (size_t)pl.units * pl.T1, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a + pl.o_coff, 0, 4 * (size_t)pl.units * (pl.c_max + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a + pl.o_l1_assign, 0xff, 4 * (size_t)pl.units * pl.n_cap, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a + pl.o_l1_steps, 0, 4 * (size_t)pl.units, s);
    // groups beyond a unit's C / L keep count 0 (the decode scores every c < c_max)
    if (e == cudaSuccess) e = cudaMemsetAsync(a + pl.o_cl_n, 0, 4 * (size_t)pl.units * pl.c_max, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(a + pl.o_sub_n, 0, 4 * (size_t)pl.units * pl.c_max * pl.l_max, s);
    if (e == cudaSuccess && pl.kpp)  // seeds past a unit's C stay -1
        e = cudaMemsetAsync(a + pl.o_pp_idx, 0xff, 4 * (size_t)pl.units * pl.c_max, s);
    return e;
}

static int common_build(const mog_kv *kv, const int32_t *lengths_dev,
                        const int32_t *lengths_host, const mog_params *p, void *arena,
                        size_t arena_bytes, cudaStream_t s, mog_handle **out, mog_handle **hh) {
    if (!out || !lengths_dev || !arena) return MOG_ERR_INVALID_ARG;
    *out = nullptr;
    Plan pl;
    int st = make_plan(p, lengths_host, &pl);
    if (st != MOG_OK) return st;
    if ((st = check_kv(kv, p->batch, p->h_kv, p->n_cap)) != MOG_OK) return st;
    if (((uintptr_t)arena & 255) != 0) return MOG_ERR_INVALID_ARG;
    if (arena_bytes < (size_t)pl.total) return MOG_ERR_ARENA_TOO_SMALL;
    mog_handle *h = new mog_handle;
    h->plan = pl;
    h->kv = *kv;
    h->arena = static_cast<char *>(arena);
    h->dev = make_dev(pl, arena, kv);
    h->lengths.assign(lengths_host, lengths_host + p->batch);
    h->appended = 0;
    h->fm_ready = false;
    h->info.assign((size_t)pl.units * UI_STRIDE, 0);
    for (int u = 0; u < pl.units; ++u) {
        const int b = u / p->h_kv;
        int C, L;
        unit_clusters(p, lengths_host[b], &C, &L);
        set_unit_info(&h->info[(size_t)u * UI_STRIDE], C, L, lengths_host[b], p->n_sink, p->n_recent, b);
    }
    cudaError_t e = cudaMemcpyAsync(h->arena + pl.o_n_now, lengths_dev, 4 * (size_t)pl.batch,
                                    cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->arena + pl.o_status, 0, 64, s);
    if (e == cudaSuccess) e = reset_build_state(h, s);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "mog_build set-up");
    }
    *hh = h;
    return MOG_OK;
}

extern "C" int mog_build(const mog_kv *kv, const int32_t *lengths_dev, const int32_t *lengths_host,
                         const mog_params *p, void *arena_dev, size_t arena_bytes, void *stream,
                         mog_handle **out) {
    if (p && (p->flags & MOG_FLAG_KMEANSPP)) return MOG_ERR_INVALID_ARG;  // draws: mog_build_seeded
    mog_handle *h = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = common_build(kv, lengths_dev, lengths_host, p, arena_dev, arena_bytes, s, out, &h);
    if (st != MOG_OK) return st;
    cudaError_t e = launch_build(h->dev, h->plan, s);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "mog_build launch");
    }
    *out = h;
    return MOG_OK;
}

extern "C" int mog_trace_layout_of(const mog_params *p, const int32_t *lengths_host,
                                   mog_trace_layout *out) {
    if (!out) return MOG_ERR_INVALID_ARG;
    Plan pl;
    int st = make_plan(p, lengths_host, &pl);
    if (st != MOG_OK) return st;
    trace_layout(pl, out);
    return MOG_OK;
}

static int build_traced_or_seeded(const mog_kv *kv, const int32_t *lengths_dev,
                                  const int32_t *lengths_host, const mog_params *p,
                                  const double *draws, void *arena_dev, size_t arena_bytes,
                                  void *trace_dev, size_t trace_bytes, void *stream, mog_handle **out);

extern "C" int mog_build_traced(const mog_kv *kv, const int32_t *lengths_dev,
                                const int32_t *lengths_host, const mog_params *p, void *arena_dev,
                                size_t arena_bytes, void *trace_dev, size_t trace_bytes,
                                void *stream, mog_handle **out) {
    if (!trace_dev) return MOG_ERR_INVALID_ARG;
    if (p && (p->flags & MOG_FLAG_KMEANSPP)) return MOG_ERR_INVALID_ARG;  // draws: mog_build_seeded
    return build_traced_or_seeded(kv, lengths_dev, lengths_host, p, nullptr, arena_dev, arena_bytes,
                                  trace_dev, trace_bytes, stream, out);
}

extern "C" int mog_build_seeded(const mog_kv *kv, const int32_t *lengths_dev,
                                const int32_t *lengths_host, const mog_params *p,
                                const double *draws_dev, void *arena_dev, size_t arena_bytes,
                                void *trace_dev, size_t trace_bytes, void *stream, mog_handle **out) {
    if (!p || !(p->flags & MOG_FLAG_KMEANSPP) || !draws_dev || ((uintptr_t)draws_dev & 7))
        return MOG_ERR_INVALID_ARG;
    return build_traced_or_seeded(kv, lengths_dev, lengths_host, p, draws_dev, arena_dev, arena_bytes,
                                  trace_dev, trace_bytes, stream, out);
}

static int build_traced_or_seeded(const mog_kv *kv, const int32_t *lengths_dev,
                                  const int32_t *lengths_host, const mog_params *p,
                                  const double *draws, void *arena_dev, size_t arena_bytes,
                                  void *trace_dev, size_t trace_bytes, void *stream, mog_handle **out) {
    if (trace_dev && !aligned16(trace_dev)) return MOG_ERR_INVALID_ARG;
    if (out) *out = nullptr;
    mog_trace_layout tl;
    int st = mog_trace_layout_of(p, lengths_host, &tl);
    if (st != MOG_OK) return st;
    if (trace_dev && trace_bytes < (size_t)tl.bytes) return MOG_ERR_ARENA_TOO_SMALL;
    mog_handle *h = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = common_build(kv, lengths_dev, lengths_host, p, arena_dev, arena_bytes, s, out, &h);
    if (st != MOG_OK) return st;
    TraceDev td{};
    cudaError_t e = cudaSuccess;
    if (trace_dev) {
        char *tr = static_cast<char *>(trace_dev);
        td.l1c = reinterpret_cast<float *>(tr + tl.l1_cent);
        td.l1a = reinterpret_cast<int *>(tr + tl.l1_assign);
        td.l2c = reinterpret_cast<float *>(tr + tl.l2_cent);
        td.l2a = reinterpret_cast<int *>(tr + tl.l2_assign);
        td.l2s = reinterpret_cast<int *>(tr + tl.l2_steps);
        td.nm = tl.n_mid;
        e = cudaMemsetAsync(trace_dev, 0, (size_t)tl.bytes, s);
    }
    if (e == cudaSuccess && draws)
        e = cudaMemcpyAsync(h->dev.pp_draw, draws, 8 * (size_t)h->plan.units * h->plan.c_max,
                            cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = launch_build(h->dev, h->plan, s, td);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "mog_build launch");
    }
    *out = h;
    return MOG_OK;
}

extern "C" int mog_sub_off_stride(const mog_params *p, const int32_t *lengths_host, int64_t *stride) {
    if (!stride) return MOG_ERR_INVALID_ARG;
    Plan pl;
    int st = make_plan(p, lengths_host, &pl);
    if (st != MOG_OK) return st;
    *stride = pl.sub_off_stride;
    return MOG_OK;
}

extern "C" int mog_build_from_partition(const mog_kv *kv, const int32_t *lengths_dev,
                                        const int32_t *lengths_host, const mog_params *p,
                                        const int32_t *perm_dev, const int32_t *sub_off_dev,
                                        void *arena_dev, size_t arena_bytes, void *stream,
                                        mog_handle **out) {
    if (!perm_dev || !sub_off_dev) return MOG_ERR_INVALID_ARG;
    mog_handle *h = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = common_build(kv, lengths_dev, lengths_host, p, arena_dev, arena_bytes, s, out, &h);
    if (st != MOG_OK) return st;
    const Plan &pl = h->plan;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(h->arena + pl.o_perm, perm_dev, 4 * (size_t)pl.units * pl.n_cap,
                             cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(h->arena + pl.o_sub_off, sub_off_dev,
                             4 * (size_t)pl.units * pl.sub_off_stride, cudaMemcpyDeviceToDevice,
                             s)) != cudaSuccess) {
        delete h;
        return cuda_fail(e, "mog_build_from_partition copy");
    }
    k_check_partition<<<pl.units, 256, 0, s>>>(h->dev);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_stats_only(h->dev, pl, s);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "mog_build_from_partition launch");
    }
    *out = h;
    return MOG_OK;
}

extern "C" int mog_decode_ex(mog_handle *h, const void *q_dev, float *out_dev,
                             const int32_t *sel_in_dev, int32_t *sel_out_dev, void *stream) {
    if (!h || !q_dev || !out_dev) return MOG_ERR_INVALID_ARG;
    if (h->plan.residual == MOG_RESIDUAL_FEATURE_MAP && !h->fm_ready) return MOG_ERR_INVALID_ARG;
    if (!aligned16(q_dev) || !aligned16(out_dev)) return MOG_ERR_INVALID_ARG;
    cudaError_t e = launch_decode(h->dev, h->plan, q_dev, out_dev, sel_in_dev, sel_out_dev,
                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "mog_decode launch");
    return MOG_OK;
}

extern "C" int mog_decode_phased(mog_handle *h, const void *q_dev, float *out_dev,
                                 const int32_t *sel_in_dev, int32_t *sel_out_dev,
                                 void *const *events, void *stream) {
    if (!h || !q_dev || !out_dev || !events) return MOG_ERR_INVALID_ARG;
    if (h->plan.residual == MOG_RESIDUAL_FEATURE_MAP && !h->fm_ready) return MOG_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
        if (!events[i]) return MOG_ERR_INVALID_ARG;
    if (!aligned16(q_dev) || !aligned16(out_dev)) return MOG_ERR_INVALID_ARG;
    cudaEvent_t ev[4];
    for (int i = 0; i < 4; ++i) ev[i] = static_cast<cudaEvent_t>(events[i]);
    cudaError_t e = launch_decode(h->dev, h->plan, q_dev, out_dev, sel_in_dev, sel_out_dev,
                                  static_cast<cudaStream_t>(stream), ev);
    if (e != cudaSuccess) return cuda_fail(e, "mog_decode_phased launch");
    return MOG_OK;
}

extern "C" int mog_decode(mog_handle *h, const void *q_dev, float *out_dev, void *stream) {
    return mog_decode_ex(h, q_dev, out_dev, nullptr, nullptr, stream);
}

extern "C" int mog_append(mog_handle *h, const void *k_new_dev, const void *v_new_dev, void *stream) {
    if (!h || !k_new_dev || !v_new_dev) return MOG_ERR_INVALID_ARG;
    if (!aligned16(k_new_dev) || !aligned16(v_new_dev)) return MOG_ERR_INVALID_ARG;
    const int nmax = *std::max_element(h->lengths.begin(), h->lengths.end());
    if ((int64_t)nmax + h->appended + 1 > h->plan.n_cap) return MOG_ERR_CAPACITY;
    cudaError_t e = launch_append(h->dev, h->plan, k_new_dev, v_new_dev, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "mog_append launch");
    if (h->plan.sliding) {
        e = launch_slide(h->dev, h->plan, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "mog_append slide launch");
    }
    h->appended += 1;
    return MOG_OK;
}

extern "C" int mog_recluster(mog_handle *h, void *stream) {
    if (!h) return MOG_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Plan &pl = h->plan;
    // every sequence has taken the same number of appends since the last build
    int nmid = 0;
    for (int b = 0; b < pl.batch; ++b) h->lengths[b] += h->appended;
    h->appended = 0;
    for (int u = 0; u < pl.units; ++u) {
        int32_t *r = &h->info[(size_t)u * UI_STRIDE];
        set_unit_info(r, r[UI_C], r[UI_L], h->lengths[r[UI_B]], r[UI_S], pl.R, r[UI_B]);
        nmid = std::max(nmid, r[UI_NMID]);
    }
    h->plan.n_mid_max = nmid;
    cudaError_t e = reset_build_state(h, s);
    if (e == cudaSuccess) e = launch_build(h->dev, h->plan, s);
    if (e == cudaSuccess && h->fm_ready) e = launch_fm_build(h->dev, h->plan, s);  // the new partition's sums
    if (e != cudaSuccess) return cuda_fail(e, "mog_recluster");
    return MOG_OK;
}

extern "C" int mog_feature_map(mog_handle *h, const float *omega_dev, void *stream) {
    if (!h || !omega_dev || ((uintptr_t)omega_dev & 3)) return MOG_ERR_INVALID_ARG;
    if (h->plan.residual != MOG_RESIDUAL_FEATURE_MAP) return MOG_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(h->dev.fm_omega, omega_dev, 4 * (size_t)FM_M * MOG_D,
                                    cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = launch_fm_build(h->dev, h->plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "mog_feature_map");
    h->fm_ready = true;
    return MOG_OK;
}

extern "C" int mog_get_layout(const mog_handle *h, mog_layout *o) {
    if (!h || !o) return MOG_ERR_INVALID_ARG;
    const Plan &P = h->plan;
    memset(o, 0, sizeof *o);
    o->units = P.units;
    o->c_max = P.c_max;
    o->l_max = P.l_max;
    o->n_cap = P.n_cap;
    o->d = P.d;
    o->group = P.G;
    o->top_c = P.tc;
    o->top_s = P.ts;
    o->unit_info = P.o_unit_info;
    o->n_now = P.o_n_now;
    o->perm = P.o_perm;
    o->sub_off = P.o_sub_off;
    o->sub_off_stride = P.sub_off_stride;
    o->cl_n = P.o_cl_n;
    o->cl_ms = P.o_cl_ms;
    o->cl_vbar = P.o_cl_vbar;
    o->sub_n = P.o_sub_n;
    o->sub_ms = P.o_sub_ms;
    o->sub_vbar = P.o_sub_vbar;
    o->l1_assign = P.o_l1_assign;
    o->status = P.o_status;
    o->l1_steps = P.o_l1_steps;
    o->fallback = P.o_fb_cnt;
    o->cl_ms16 = P.o_cl_ms16;
    o->sub_ms16 = P.o_sub_ms16;
    o->cl_ms8 = P.o_cl_ms8;
    o->sub_ms8 = P.o_sub_ms8;
    o->pp_idx = P.o_pp_idx;
    o->fm_z = P.o_fm_z;
    o->fm_t = P.o_fm_t;
    return MOG_OK;
}

extern "C" int mog_sync_status(mog_handle *h, void *stream) {
    if (!h) return MOG_ERR_INVALID_ARG;
    CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    int st = 0;
    CK(cudaMemcpy(&st, h->arena + h->plan.o_status, 4, cudaMemcpyDeviceToHost));
    if (st & (1 << ST_TIMEOUT)) return MOG_ERR_TIMEOUT;
    return st ? MOG_ERR_DEVICE_CHECK : MOG_OK;
}

extern "C" int mog_decode_splits(const mog_handle *h, int32_t *splits) {
    if (!h || !splits) return MOG_ERR_INVALID_ARG;
    *splits = h->plan.P;
    return MOG_OK;
}

extern "C" void mog_destroy(mog_handle *h) { delete h; }

// ---------------------------------------------------------------------- dense_decode

extern "C" int dense_decode_scratch_bytes(int32_t batch, int32_t h_kv, int32_t h_q, int32_t d,
                                          int32_t n_max, size_t *bytes) {
    if (!bytes || batch <= 0 || h_kv <= 0 || h_q <= 0 || n_max <= 0) return MOG_ERR_INVALID_ARG;
    if (d != MOG_D || h_q % h_kv != 0 || h_q / h_kv > MOG_MAX_G) return MOG_ERR_SHAPE;
    const int units = batch * h_kv, G = h_q / h_kv;
    *bytes = (size_t)units * dense_splits(units, n_max) * G * (MOG_D + 4) * sizeof(float);
    return MOG_OK;
}

extern "C" int dense_decode(const mog_kv *kv, const int32_t *lengths_dev, int32_t n_max,
                            int32_t batch, int32_t h_kv, int32_t h_q, int32_t d, const void *q_dev,
                            float *out_dev, void *scratch_dev, size_t scratch_bytes, void *stream) {
    size_t need = 0;
    int st = dense_decode_scratch_bytes(batch, h_kv, h_q, d, n_max, &need);
    if (st != MOG_OK) return st;
    if ((st = check_kv(kv, batch, h_kv, n_max)) != MOG_OK) return st;
    if (!lengths_dev || !q_dev || !out_dev || !scratch_dev) return MOG_ERR_INVALID_ARG;
    if (!aligned16(q_dev) || !aligned16(out_dev) || !aligned16(scratch_dev)) return MOG_ERR_INVALID_ARG;
    if (scratch_bytes < need) return MOG_ERR_ARENA_TOO_SMALL;
    const int units = batch * h_kv;
    cudaError_t e = launch_dense(kv, lengths_dev, n_max, batch, h_kv, h_q / h_kv, q_dev, out_dev,
                                 static_cast<float *>(scratch_dev), dense_splits(units, n_max),
                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dense_decode launch");
    return MOG_OK;
}

extern "C" int dense_decode_noalloc(const mog_kv *kv, const int32_t *lengths_dev, int32_t n_max,
                                    int32_t batch, int32_t h_kv, int32_t h_q, int32_t d,
                                    const void *q_dev, float *out_dev, void *stream) {
    size_t need = 0;
    int st = dense_decode_scratch_bytes(batch, h_kv, h_q, d, n_max, &need);
    if (st != MOG_OK) return st;
    if ((st = check_kv(kv, batch, h_kv, n_max)) != MOG_OK) return st;
    if (!lengths_dev || !q_dev || !out_dev) return MOG_ERR_INVALID_ARG;
    if (!aligned16(q_dev) || !aligned16(out_dev)) return MOG_ERR_INVALID_ARG;
    float *scratch = nullptr;
    size_t cap = 0;
    CK(dense_static_scratch(&scratch, &cap));  // set-up on the first call on a device
    if (need > cap) {
        snprintf(g_err, sizeof g_err,
                 "dense_decode_noalloc: this shape needs %zu bytes of scratch, the static "
                 "array holds %zu",
                 need, cap);
        return MOG_ERR_CAPACITY;
    }
    const int units = batch * h_kv;
    cudaError_t e = launch_dense(kv, lengths_dev, n_max, batch, h_kv, h_q / h_kv, q_dev, out_dev,
                                 scratch, dense_splits(units, n_max), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dense_decode_noalloc launch");
    return MOG_OK;
}

// ----------------------------------------------------------------- parity exports

// scratch of mog_kmeans_assign: counters (256 B), the fallback and recheck row lists,
// the centroid images and norms of the tensor-core pass
static size_t km_off_lists() { return 256; }
static size_t km_list_bytes(int n) { return ((4 * (size_t)std::max(n, 1)) + 255) & ~(size_t)255; }
static size_t km_img_bytes(int k) { return 2 * (size_t)ceil_div64(k, KM_CHUNK) * KM_IMG_CHUNK; }

extern "C" int mog_kmeans_assign_scratch_bytes(int32_t n, int32_t k, int32_t d, size_t *bytes) {
    if (!bytes || n < 0 || k <= 0) return MOG_ERR_INVALID_ARG;
    if (d != MOG_D) return MOG_ERR_SHAPE;
    if (k > MAX_C) return MOG_ERR_SHAPE;
    *bytes = km_off_lists() + 2 * km_list_bytes(n) + km_img_bytes(k) + 4 * (size_t)ceil_div64(k, KM_CHUNK) * KM_CHUNK;
    return MOG_OK;
}

extern "C" int mog_kmeans_assign(const void *x_dev, int64_t ld, int32_t n, const float *cent_dev,
                                 int32_t k, int32_t d, int32_t *assign_out_dev, void *scratch_dev,
                                 size_t scratch_bytes, void *stream, int32_t *counts_host) {
    size_t need = 0;
    int st = mog_kmeans_assign_scratch_bytes(n, k, d, &need);
    if (st != MOG_OK) return st;
    if (!x_dev || !cent_dev || !assign_out_dev || !scratch_dev) return MOG_ERR_INVALID_ARG;
    if (!aligned16(x_dev) || !aligned16(cent_dev) || ld < MOG_D || (ld & 7)) return MOG_ERR_SHAPE;
    if (scratch_bytes < need || !aligned16(scratch_dev)) return MOG_ERR_ARENA_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(scratch_dev);
    int *sc = reinterpret_cast<int *>(base);
    KmScratch ks;
    ks.changed = sc;
    ks.fb_cnt = sc + 32;
    ks.rc_cnt = sc + 40;
    ks.status = sc + 48;
    ks.fb_list = reinterpret_cast<int *>(base + km_off_lists());
    ks.rc_list = reinterpret_cast<int *>(base + km_off_lists() + km_list_bytes(n));
    ks.cimg = reinterpret_cast<uint16_t *>(base + km_off_lists() + 2 * km_list_bytes(n));
    ks.cnorm = reinterpret_cast<float *>(base + km_off_lists() + 2 * km_list_bytes(n) + km_img_bytes(k));
    CK(cudaMemsetAsync(sc, 0, 256, s));
    CK(launch_assign_l1(static_cast<const uint16_t *>(x_dev), ld, n, cent_dev, k, assign_out_dev, ks, s));
    if (counts_host) {
        int32_t c[3];
        CK(cudaMemcpyAsync(&c[0], ks.fb_cnt, 4, cudaMemcpyDeviceToHost, s));
        CK(cudaMemcpyAsync(&c[1], ks.rc_cnt, 4, cudaMemcpyDeviceToHost, s));
        CK(cudaMemcpyAsync(&c[2], ks.status, 4, cudaMemcpyDeviceToHost, s));
        CK(cudaStreamSynchronize(s));
        counts_host[0] = c[0];
        counts_host[1] = c[1];
        if (c[2]) return (c[2] & (1 << ST_TIMEOUT)) ? MOG_ERR_TIMEOUT : MOG_ERR_DEVICE_CHECK;
    }
    return MOG_OK;
}

extern "C" int mog_kmeans_assign_segments(const void *x_dev, int64_t ld, const int32_t *rows_dev,
                                          const int32_t *seg_off_dev, int32_t n_seg,
                                          const float *cent_dev, int32_t k, int32_t d,
                                          int32_t *assign_out_dev, void *stream) {
    if (!x_dev || !rows_dev || !seg_off_dev || !cent_dev || !assign_out_dev || n_seg < 0)
        return MOG_ERR_INVALID_ARG;
    if (d != MOG_D || k <= 0 || k > MOG_MAX_L || ld < MOG_D || (ld & 7) || !aligned16(x_dev))
        return MOG_ERR_SHAPE;
    CK(launch_assign_segments(static_cast<const uint16_t *>(x_dev), ld, rows_dev, seg_off_dev, n_seg,
                              cent_dev, k, assign_out_dev, static_cast<cudaStream_t>(stream)));
    return MOG_OK;
}

extern "C" int mog_check_bounded_wait(int32_t limit, int32_t arrive, int32_t *scratch_dev,
                                      void *stream) {
    if (!scratch_dev || limit <= 0) return MOG_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = 0;
    CK(cudaMemsetAsync(scratch_dev, 0, sizeof(int32_t), s));
    CK(launch_wait_check(limit, arrive, scratch_dev, s));
    CK(cudaMemcpyAsync(&st, scratch_dev, sizeof st, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if (st & (1 << ST_TIMEOUT)) return MOG_ERR_TIMEOUT;
    return st ? MOG_ERR_DEVICE_CHECK : MOG_OK;
}
