// internal.h -- host/device shared structures of libmog (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mog.h"

namespace mog {

// per-unit table, int32 x 8 (mirrors mog_layout.unit_info)
enum { UI_C = 0, UI_L, UI_NBUILD, UI_NMID, UI_S, UI_RLO, UI_B, UI_STRIDE = 8 };

constexpr int SORT_CHUNK = 1024;   // rows per stable-sort chunk (one warp)
// First-level assignment on the tensor cores: centroids in chunks of KM_CHUNK, each chunk
// an image of KM_IMG_CHUNK bf16 ({high, low} x two 64-column halves x KM_CHUNK rows).
constexpr int KM_CHUNK = 128;
constexpr int64_t KM_IMG_CHUNK = 4LL * KM_CHUNK * 64;
constexpr int MAX_SPLITS = 64;     // partials per unit in the exact-attention kernel
constexpr int PART_SLOTS = MAX_SPLITS;  // partials per unit: one per rows-kernel CTA
// Rows-kernel plan per unit, written by the selection kernel: [0] segments NS, [1] rows T,
// [2] anchors, [3] sink rows, [4] first recent position, [5] union size Uc, [6] subclusters
// per cluster L, [7] clusters C, [PLAN_START + p] the segment holding the first row of
// rows-kernel CTA p (0 while that row is an anchor), [PLAN_UCL + j] the cluster of union
// slot j.
constexpr int PLAN_START = 8;
constexpr int PLAN_UCL = PLAN_START + MAX_SPLITS;
constexpr int PLAN_W = PLAN_UCL + MOG_MAX_UNION;  // ints, whole 16-byte chunks
constexpr int MAX_C = 4096;        // clusters per unit supported
constexpr int PP_THREADS = 256, PP_PER = 4;  // k-means++ seeding: keys per thread
constexpr int PP_ROWS = PP_THREADS * PP_PER;  // ... and per CTA
constexpr int FM_M = MOG_FM_FEATURES;  // feature-map residual: features
constexpr int FM_W = MOG_D + 4;        // floats per feature row of a sum: d values, the plain sum, padding
constexpr int FM_NCH = 32;             // decode: CTAs per head over its chosen subclusters

// Typed view of an arena, passed by value to every kernel.
struct Dev {
    // cache
    const uint16_t *K, *V;
    uint16_t *Kw, *Vw;  // writable views (append)
    int64_t sb, sh, sn;
    const int *bt;      // block table of a paged cache (null: contiguous), [batch][pps]
    int pshift, pps;    // log2(rows per page), pages per sequence
    // shape
    int batch, h_kv, G, units, n_cap, c_max, l_max, tc, ts, T1, T2, score_mode, residual;
    int union_exact;  // every head attends the union of the heads' chosen subclusters
    int group_select;  // one selection per KV head (log-sum-exp of the heads' scores)
    int bf16s;         // summaries read as bf16 (cl_ms16, sub_ms16, value means' high parts)
    int fp8s;          // summaries read as fp8 e4m3 (cl_ms8, sub_ms8; value means rounded)
    int kpp;           // first-level k-means++ seeds (pp_*)
    int P, nchunks, nseg_max;
    int64_t sub_off_stride;
    float tau;
    // persistent
    int *unit_info, *n_now, *perm, *sub_off, *cl_n, *sub_n, *l1_assign, *status, *l1_steps;
    float *cl_ms, *cl_vbar, *sub_ms, *sub_vbar;
    uint16_t *cl_vhl, *sub_vhl;  // value means as bf16 high and low parts [item][2][d]
    uint16_t *cl_ms16, *sub_ms16;  // bf16 mean and variance [item][2][d], or null
    uint8_t *cl_ms8, *sub_ms8;     // e4m3 mean and variance [item][2][d], or null
    // build workspace
    float *cent;
    int *permA, *changed, *fb_list, *fb_cnt, *hist, *offs, *ctot, *coff, *sub_assign;
    int *rc_list, *rc_cnt;  // rows the tensor-core pass leaves to the direct pass
    uint16_t *cimg;         // centroid images for the tensor cores [unit][cimg_ustride]
    float *cnorm;           // |c|^2 [unit][cn_ustride]
    int64_t cimg_ustride, cn_ustride;
    // k-means++ seeding: draws [unit][c_max], seeds [unit][c_max], D2 [2][unit][n_cap]
    // (round parity), per-CTA D2 sums [2][unit][pp_nblk]
    double *pp_draw, *pp_part;
    int *pp_idx;
    float *pp_d2;
    int pp_nblk;
    // feature-map residual: frequencies [FM_M][d], M_i [FM_M], sums per subcluster
    // [unit][c_max*l_max][FM_M][FM_W], per cluster [unit][c_max][FM_M][FM_W], per unit
    // [unit][FM_M][FM_W]; decode: per-head vectors [unit][G][FM_NCH+1][FM_W], maxima [unit][G]
    float *fm_omega, *fm_mi, *fm_z, *fm_zc, *fm_t, *fm_vec, *fm_mref;
    // decode workspace
    float *partials;  // [units][PART_SLOTS][G][PART_W]
    int *sel;         // [units][G][tc + tc*ts] selection of the last step
    int *plan;        // [units][PLAN_W]
    int *segrow, *segoff;  // [units][nseg_max] first row of a segment, its offset in perm
    uint32_t *segmask;     // [units][nseg_max] heads that attend the segment
    float *resx;           // [units][resx_stride]: residual exponents [item][G, padded to 4]
    int64_t resx_stride;

    // element offset of row pos of (b, h): through the block table when the cache is paged
    __device__ __forceinline__ int64_t row_off(int b, int h, int64_t pos) const {
        if (!bt) return b * sb + h * sh + pos * sn;
        const int64_t page = bt[(int64_t)b * pps + (pos >> pshift)];
        return page * sb + h * sh + (pos & ((1 << pshift) - 1)) * sn;
    }
    __device__ __forceinline__ const uint16_t *krow(int b, int h, int64_t pos) const {
        return K + row_off(b, h, pos);
    }
    __device__ __forceinline__ const uint16_t *vrow(int b, int h, int64_t pos) const {
        return V + row_off(b, h, pos);
    }
};

// Device pointers of a build trace (see mog_trace_layout); all null for an untraced build.
// Only the build's kernels take it, so that the decode kernels' parameters stay as they are.
struct TraceDev {
    float *l1c, *l2c;
    int *l1a, *l2a, *l2s;
    int64_t nm;  // row stride of the traced assignments
};

// Host-side plan: sizes and byte offsets of every array in the arena.
struct Plan {
    int batch, h_kv, h_q, G, d, n_cap, units, c_max, l_max, tc, ts, T1, T2;
    int score_mode, residual, union_exact, group_select, sliding, bf16s, fp8s, kpp, R, P, nchunks,
        n_mid_max, nseg_max, pp_nblk;
    int64_t sub_off_stride;
    int64_t o_unit_info, o_n_now, o_perm, o_sub_off, o_cl_n, o_cl_ms, o_cl_vbar, o_sub_n, o_sub_ms,
        o_sub_vbar, o_cl_vhl, o_sub_vhl, o_cl_ms16, o_sub_ms16, o_cl_ms8, o_sub_ms8, o_l1_assign, o_status,
        o_l1_steps;
    int64_t o_cent, o_permA, o_changed, o_fb_list, o_fb_cnt, o_hist, o_offs, o_ctot, o_coff,
        o_sub_assign, o_rc_list, o_rc_cnt, o_cimg, o_cnorm, cimg_ustride, cn_ustride;
    int64_t o_partials, o_sel, o_plan, o_segrow, o_segoff, o_segmask, o_resx, resx_stride;
    int64_t o_pp_draw, o_pp_idx, o_pp_d2, o_pp_part;
    int64_t o_fm_omega, o_fm_mi, o_fm_z, o_fm_zc, o_fm_t, o_fm_vec, o_fm_mref;
    int64_t total;
};

int num_sms();
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (function, device, size)
cudaError_t ensure_smem(const void *fn, size_t bytes);
int make_plan(const mog_params *p, const int32_t *lengths_host, Plan *pl);
void trace_layout(const Plan &pl, mog_trace_layout *t);
Dev make_dev(const Plan &pl, void *arena, const mog_kv *kv);
void unit_clusters(const mog_params *p, int n, int *C, int *L);

// launchers (return cudaError_t of the launch)
cudaError_t launch_build(const Dev &dv, const Plan &pl, cudaStream_t s, const TraceDev &tr = TraceDev{});
cudaError_t launch_stats_only(const Dev &dv, const Plan &pl, cudaStream_t s);
cudaError_t launch_decode(const Dev &dv, const Plan &pl, const void *q, float *out,
                          const int32_t *sel_in, int32_t *sel_out, cudaStream_t s,
                          cudaEvent_t const *events = nullptr);
cudaError_t launch_append(const Dev &dv, const Plan &pl, const void *k_new, const void *v_new,
                          cudaStream_t s);
cudaError_t launch_slide(const Dev &dv, const Plan &pl, cudaStream_t s);
cudaError_t launch_fm_build(const Dev &dv, const Plan &pl, cudaStream_t s);
cudaError_t launch_fm_resid(const Dev &dv, const uint16_t *q, int SW, cudaStream_t s);
cudaError_t launch_dense(const mog_kv *kv, const int32_t *lengths, int n_max, int batch, int h_kv,
                         int G, const void *q, float *out, float *scratch, int splits,
                         cudaStream_t s);
int log2_exact(int x);  // log2 of a power of two, -1 otherwise
int dense_splits(int units, int n_max);
cudaError_t dense_static_scratch(float **ptr, size_t *bytes);
size_t slot_smem_bytes(int G, int c_max, int l_max, int tc);
// Work buffers of a single-matrix first-level assignment step.
struct KmScratch {
    int *changed, *fb_cnt, *rc_cnt, *status, *fb_list, *rc_list;
    uint16_t *cimg;
    float *cnorm;
};
cudaError_t launch_assign_l1(const uint16_t *x, int64_t ld, int n, const float *cent, int k,
                             int32_t *assign, const KmScratch &ks, cudaStream_t s);
cudaError_t launch_wait_check(int limit, int arrive, int *status, cudaStream_t s);
cudaError_t launch_assign_segments(const uint16_t *x, int64_t ld, const int32_t *rows,
                                   const int32_t *seg_off, int n_seg, const float *cent, int k,
                                   int32_t *assign, cudaStream_t s);

}  // namespace mog
