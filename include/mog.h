/*
 * mog.h -- C ABI of libmog: Mixture-of-Gaussians (MoG) decode attention on one GPU
 * (NVIDIA GB300, sm_103a).
 *
 * What the library computes, and where the pages state it:
 *   [IA] "Iceberg Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians",
 *        Abstract: after prefill, each head's keys are split into O(sqrt N) clusters and
 *        O(log N) subclusters per cluster, each group summarised by a Gaussian; at decode
 *        the query is scored against the summaries, the best clusters/subclusters are
 *        attended exactly, the rest is approximated from the groups' means and variances.
 *   [RC] newx.sg paper page on retrieval-completion attention, Abstract: sink and tail
 *        anchors are attended exactly together with the retrieved keys; the estimated
 *        numerator and denominator of the rest are added in the unnormalised domain and
 *        one normalisation follows.
 * Residual form of this library (consistent with [IA]'s use of group means and variances): an
 * unselected group s (count n_s, key mean mu_s, per-dimension population variance
 * sigma2_s, value mean vbar_s) adds den_s = n_s * exp(tau q.mu_s + tau^2/2 *
 * sum_j q_j^2 sigma2_sj - m) to the denominator and den_s * vbar_s to the numerator,
 * tau = 1/sqrt(d), m the running maximum.
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are device pointers, *_host host pointers.  The caller owns all
 *    memory (KV cache, queries, outputs, the build arena, scratch).  The library never
 *    allocates device memory; a handle is a small host structure.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All
 *    device work is enqueued on it; no entry point synchronises the host unless it says so.
 *  - bf16 data are IEEE bfloat16 bit patterns (uint16).  KV caches are [B][H_kv][n_cap][d]
 *    with element strides given in mog_kv; d must be 128 and rows contiguous.
 *  - Return value: MOG_OK or a mog_status error.  Argument errors are detected before any
 *    work is enqueued.  Errors detected on the device are recorded in the handle's status
 *    word and reported by mog_sync_status.
 */
#ifndef MOG_H
#define MOG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOG_OK = 0,
    MOG_ERR_INVALID_ARG = 1,     /* null pointer, negative size, bad flag */
    MOG_ERR_SHAPE = 2,           /* unsupported shape (d != 128, G > 16, ...) */
    MOG_ERR_ARENA_TOO_SMALL = 3, /* caller buffer smaller than the size query returned */
    MOG_ERR_CUDA = 4,            /* a CUDA runtime call failed (see mog_last_error) */
    MOG_ERR_DEVICE_CHECK = 5,    /* a device-side check failed (see mog_sync_status) */
    MOG_ERR_TIMEOUT = 6,         /* reserved: a bounded device wait gave up */
    MOG_ERR_NOT_IMPLEMENTED = 7,
    MOG_ERR_CAPACITY = 8         /* appending past n_cap */
} mog_status;

/*
 * Build and decode parameters.  All counts are per KV head ("unit" = (b, h_kv)).
 *  n_clusters, n_sub : C and L; 0 selects round(sqrt(N_b)) and ceil(log2(N_b)) from each
 *                      sequence's build length N_b ([IA]: O(sqrt N) x O(log N)).
 *  top_c, top_s      : clusters selected per query head, subclusters selected inside each
 *                      selected cluster ([IA]).  min(C, top_c*G) <= 256, L <= 32.
 *  n_sink, n_recent  : anchors S and R; positions [0,S) and [N_b-R, N) are never clustered
 *                      and always attended exactly ([RC]).
 *  iters_l1, iters_l2: Lloyd assignment steps per level (0 selects 10); a level stops
 *                      early once a step changes no assignment.
 *  score_mode        : 0 = log-mass score ln n + tau q.mu + tau^2/2 sum q^2 sigma2 (the
 *                      residual's own exponent); 1 = tau q.mu only.
 *  residual          : 1 = add the Gaussian residual (default), 0 = top-only ablation,
 *                      2 = the feature-map residual (MOG_RESIDUAL_FEATURE_MAP) instead.
 *  flags             : 0, or any of MOG_FLAG_UNION_EXACT, MOG_FLAG_SLIDING,
 *                      MOG_FLAG_GROUP_SELECT, MOG_FLAG_KMEANSPP (mog_build_seeded only),
 *                      and one of MOG_FLAG_BF16_SUMMARIES, MOG_FLAG_FP8_SUMMARIES.
 *
 * MOG_FLAG_UNION_EXACT (a variant of this library; the pages select per query head and do
 * not define it): each query head still makes its own selection, but every query head of a
 * KV head attends exactly the anchors and the rows of every subcluster that any of them
 * chose (the rows are loaded once for the group anyway); the Gaussian residual then covers
 * the groups no head chose: the other non-empty subclusters of the chosen clusters and the
 * clusters no head chose.  The bytes read are those of the default mode.
 */
#define MOG_FLAG_UNION_EXACT 1
/*
 * MOG_RESIDUAL_FEATURE_MAP (mog_params.residual = 2; the retrieval-completion page on
 * newx.sg, Abstract and AI Summary: a fixed-size feature-map summary of the mid region,
 * built at prefill, estimates the numerator and denominator of the keys that are not
 * retrieved, added to the exact part unnormalised before one normalisation): instead of
 * the groups' Gaussians, every mid key that a head does not attend exactly contributes
 * phi(q~).phi(k~) [v, 1], phi_i(x) = m^(-1/2) exp(w_i.x - |x|^2/2) for the
 * m = MOG_FM_FEATURES caller-given frequencies w_i (drawn N(0, I_d); mog_feature_map),
 * q~ = sqrt(tau) q, k~ = sqrt(tau) k.  The build keeps every subcluster's feature sums;
 * a decode subtracts the head's chosen subclusters' sums from the unit's total.  Not
 * with MOG_FLAG_UNION_EXACT or MOG_FLAG_SLIDING (MOG_ERR_INVALID_ARG).
 */
#define MOG_RESIDUAL_FEATURE_MAP 2
#define MOG_FM_FEATURES 32
/*
 * MOG_FLAG_SLIDING (a variant of this library; the pages keep a recent window but do not
 * say what happens to a key leaving it): the recent anchors stay the last n_recent keys.
 * When mog_append makes a KV head's window longer, its oldest recent key joins the nearest
 * non-empty cluster and, inside it, the nearest non-empty subcluster (the build's
 * nearest-centroid rule against the groups' means), and both groups' count, mean,
 * population variance and value mean take it by Welford's update.  The key's row joins
 * its subcluster in the partition (`perm`, `sub_off`), so it is attended exactly whenever
 * that subcluster is chosen.  A head with no non-empty cluster keeps a growing window.
 */
#define MOG_FLAG_SLIDING 2
/*
 * MOG_FLAG_GROUP_SELECT (a variant of this library; the pages select per query head): the
 * G query heads of a KV head select once.  A group's score is the log of the sum over the
 * heads of exp(its per-head selection score), the log of the group's total estimated
 * attention mass; the top_c clusters and the top_s subclusters inside each are taken by
 * that score.  Every head attends the group's selection exactly and takes its own Gaussian
 * residual of every other non-empty group.  Fewer rows are read than with per-head
 * selections.  The exported selection repeats the group's lists for every head; a given
 * selection (mog_decode_ex) is taken from the group's first head.
 */
#define MOG_FLAG_GROUP_SELECT 4
/*
 * MOG_FLAG_BF16_SUMMARIES (a variant of this library; the pages do not fix the summaries'
 * precision): the selection scores and the Gaussian residual terms use every group's key
 * mean, per-dimension variance and value mean rounded from their fp32 values to bf16
 * (nearest, ties to even); counts stay exact.  The build keeps the fp32 summaries and
 * writes the bf16 copies beside them (mog_layout.cl_ms16, sub_ms16); the sliding window
 * updates both.  The decode reads half the summary bytes.
 */
#define MOG_FLAG_BF16_SUMMARIES 8
/*
 * MOG_FLAG_FP8_SUMMARIES (a variant of this library, exclusive with the bf16 one): the same
 * with the summaries rounded from fp32 to fp8 e4m3 (nearest, ties to even, saturating at
 * +-448); the build writes e4m3 copies of the means and variances (mog_layout.cl_ms8,
 * sub_ms8: a quarter of the fp32 bytes) and the residual terms read the rounded value
 * means (exact in bf16).
 */
#define MOG_FLAG_FP8_SUMMARIES 16
/*
 * MOG_FLAG_KMEANSPP (a variant of this library; the pages name no seeding): the first
 * level starts from k-means++ seeds instead of strided ones.  Seed 0 of a unit is mid key
 * floor(u_0 n) (n mid keys in position order); seed r >= 1 is drawn with the uniform u_r
 * from the mid keys with probability proportional to D2, the squared distance to the
 * nearest seed so far: the first key (in position order) whose running sum of D2 exceeds
 * u_r times the total.  D2 is computed in fp32 (each difference rounded to fp32, four
 * partial sums, dimension j into sum j mod 4, by fused multiply-add in increasing j, then
 * (s0 + s1) + (s2 + s3)), the running sums in fp64; if every key sits
 * on a seed the pick is floor(u_r n).  The draws u are an input (mog_build_seeded); each
 * round reads every mid key once, so the seeding costs about C_u passes over the keys.
 * The second level keeps its strided seeds.
 */
#define MOG_FLAG_KMEANSPP 32
typedef struct mog_params {
    int32_t batch, h_kv, h_q, d;
    int32_t n_cap;
    int32_t n_clusters, n_sub;
    int32_t top_c, top_s;
    int32_t n_sink, n_recent;
    int32_t iters_l1, iters_l2;
    int32_t score_mode;
    int32_t residual;
    int32_t flags;
} mog_params;

/* A bf16 KV cache in device memory, contiguous or paged.  mog_append writes into it.
 *  Contiguous (block_table == NULL): element (b, h, n, j) of K is
 *    k[b*stride_b + h*stride_h + n*stride_n + j], and n_cap * stride_n * 2 bytes must stay
 *    below 4 GiB (one head's rows are addressed with 32-bit offsets; MOG_ERR_SHAPE
 *    otherwise).
 *  Paged (a serving engine's block table): position n of sequence b lives in page
 *    block_table[b*pages_per_seq + n / page_rows] (a device int32 array of
 *    batch*pages_per_seq entries, caller-owned), row n % page_rows of it, and element
 *    (b, h, n, j) of K is k[page*stride_b + h*stride_h + (n % page_rows)*stride_n + j]:
 *    stride_b is the stride of one page.  page_rows is a power of two >= 16,
 *    pages_per_seq * page_rows >= n_cap, and every page index p used must have
 *    p * page_rows < 2^31.  The block table must not change while a handle uses it.  The
 *    build's first-level assignment then skips its tensor-core pass (whose TMA tiles need
 *    contiguous rows) and scores every key with the direct fp32 pass; results are the same.
 *  V uses the same strides and table.  stride_n >= d, all strides multiples of 8 elements
 *  (16-byte aligned rows), base pointers 16-byte aligned. */
typedef struct mog_kv {
    void *k;
    void *v;
    int64_t stride_b, stride_h, stride_n;
    const int32_t *block_table; /* NULL: contiguous */
    int32_t page_rows;
    int32_t pages_per_seq;
} mog_kv;

typedef struct mog_handle mog_handle;

/* Byte offsets (into the arena) of the handle's device arrays, for inspection by tests.
 * u = b*h_kv + h indexes units. */
typedef struct mog_layout {
    int32_t units, c_max, l_max, n_cap, d, group, top_c, top_s;
    int64_t unit_info;  /* int32 [units][8]: C_u, L_u, N_build, N_mid, S, recent_lo, b, 0 */
    int64_t n_now;      /* int32 [batch]: current length of each sequence */
    int64_t perm;       /* int32 [units][n_cap]: mid positions ordered (cluster, sub, position) */
    int64_t sub_off;    /* int32 [units][sub_off_stride]: offsets into perm, C_u*L_u+1 used */
    int64_t sub_off_stride;
    int64_t cl_n;       /* int32 [units][c_max] */
    int64_t cl_ms;      /* f32   [units][c_max][2][d]: mean, variance */
    int64_t cl_vbar;    /* f32   [units][c_max][d] */
    int64_t sub_n;      /* int32 [units][c_max*l_max], group c*L_u + l */
    int64_t sub_ms;     /* f32   [units][c_max*l_max][2][d] */
    int64_t sub_vbar;   /* f32   [units][c_max*l_max][d] */
    int64_t l1_assign;  /* int32 [units][n_cap]: final first-level cluster of mid key S+i */
    int64_t status;     /* int32 [8]: device status word, check counters */
    int64_t l1_steps;   /* int32 [units]: assignment steps taken by the first level */
    int64_t fallback;   /* int32 [units][iters_l1]: rows decided by the exact fp64 fallback */
    int64_t cl_ms16;    /* bf16  [units][c_max][2][d]: mean, variance (MOG_FLAG_BF16_SUMMARIES; else 0) */
    int64_t sub_ms16;   /* bf16  [units][c_max*l_max][2][d] (MOG_FLAG_BF16_SUMMARIES; else 0) */
    int64_t cl_ms8;     /* e4m3  [units][c_max][2][d] (MOG_FLAG_FP8_SUMMARIES; else 0) */
    int64_t sub_ms8;    /* e4m3  [units][c_max*l_max][2][d] (MOG_FLAG_FP8_SUMMARIES; else 0) */
    int64_t pp_idx;     /* int32 [units][c_max]: seed r's mid-key index, -1 past C_u (MOG_FLAG_KMEANSPP; else 0) */
    /* MOG_RESIDUAL_FEATURE_MAP (else 0): f32 [units][c_max*l_max][MOG_FM_FEATURES][d+4]
     * feature sums of every subcluster, row i holding sum over members of
     * exp(w_i.k~ - |k~|^2/2 - M_i) v_k in [0, d) and the same sum without v at d (entries
     * d+1 .. d+3 zero), scaled by M_i = |w_i|^2/2 - 40; and f32
     * [units][MOG_FM_FEATURES][d+4] their sum per unit */
    int64_t fm_z, fm_t;
} mog_layout;

/* Human-readable name of a status code.  Never NULL. */
const char *mog_status_string(int status);

/* Text of the last CUDA error seen by this thread's calls into the library. */
const char *mog_last_error(void);

/*
 * Size of the device arena mog_build needs for these parameters and build lengths.
 * lengths_host: int32[batch] build lengths N_b (1 <= N_b <= n_cap).
 */
int mog_arena_bytes(const mog_params *p, const int32_t *lengths_host, size_t *bytes);

/*
 * MoG build ([IA], the post-prefill hierarchical partition): for every unit, first-level
 * Lloyd k-means of the mid keys [S, N_b - R) into C_u clusters, second-level k-means of
 * each cluster into L_u subclusters, then count, key mean, per-dimension population
 * variance and value mean of every cluster and subcluster.  Enqueued on `stream`; no host
 * synchronisation.
 *  kv           : the cache (read; must outlive the handle)
 *  lengths_dev  : int32[batch] N_b on the device; lengths_host the same values on the host
 *  arena_dev    : caller-owned device buffer of at least mog_arena_bytes() bytes, 256-byte
 *                 aligned; it holds every summary and all decode workspace and must
 *                 outlive the handle
 *  out          : receives a new handle (free it with mog_destroy)
 */
int mog_build(const mog_kv *kv, const int32_t *lengths_dev, const int32_t *lengths_host,
              const mog_params *p, void *arena_dev, size_t arena_bytes, void *stream,
              mog_handle **out);

/*
 * MoG decode step ([IA], decoding: score the summaries, attend the best groups exactly,
 * approximate the rest from their Gaussians; [RC]): per query head, score the
 * clusters, take the top top_c, score their subclusters, take the top top_s in each,
 * attend exactly to the members of the selected subclusters plus the anchors, add the
 * Gaussian residual of every unselected non-empty group, normalise once.
 *  q_dev   : bf16 [batch][h_q][d]; query head g*G + i belongs to KV head g
 *  out_dev : f32 [batch][h_q][d]
 * Calls on one handle must not overlap on the GPU (they share the arena's workspace).
 */
int mog_decode(mog_handle *h, const void *q_dev, float *out_dev, void *stream);

/*
 * mog_decode with the selection exposed, for parity tests.  sel layout: int32
 * [batch][h_q][top_c + top_c*top_s]: the selected cluster ids in rank order, then for
 * the i-th selected cluster its top_s subcluster indices (0..L_u-1) in rank order; -1
 * pads missing entries.  sel_in_dev (may be NULL) replaces the library's own selection;
 * sel_out_dev (may be NULL) receives the selection used.
 */
int mog_decode_ex(mog_handle *h, const void *q_dev, float *out_dev, const int32_t *sel_in_dev,
                  int32_t *sel_out_dev, void *stream);

/*
 * Append one decode token per sequence: k_new_dev, v_new_dev bf16 [batch][h_kv][d] are
 * written at position n_now[b] of the cache, then n_now[b] += 1.  Appended keys join the
 * recent anchors; without MOG_FLAG_SLIDING the summaries are unchanged and the window
 * grows.  With it, a second kernel then moves each KV head's oldest recent key into its
 * nearest cluster and subcluster once the window holds more than n_recent keys (see
 * MOG_FLAG_SLIDING), updating that head's counts, means, variances, value means,
 * partition and window start in the arena.  MOG_ERR_CAPACITY if a sequence would exceed
 * n_cap (checked on the host from the build lengths and the number of appends).  Not to
 * be run concurrently with a decode on the same handle.
 */
int mog_append(mog_handle *h, const void *k_new_dev, const void *v_new_dev, void *stream);

/*
 * The feature-map summary (MOG_RESIDUAL_FEATURE_MAP; the retrieval-completion page's
 * prefill-time summary): copies the frequencies omega_dev (f32 [MOG_FM_FEATURES][d],
 * device, 4-byte aligned; rows drawn N(0, I_d) by the caller) into the arena and computes
 * every subcluster's feature sums and the units' totals for the handle's partition.
 * Required once after the build before a decode with residual = 2 (MOG_ERR_INVALID_ARG
 * otherwise, also when the handle was built with another residual); mog_recluster redoes
 * the sums for the new partition.  Enqueued on `stream`.
 */
int mog_feature_map(mog_handle *h, const float *omega_dev, void *stream);

/*
 * Periodic re-clustering during long generation ([IA]'s post-prefill partition, redone
 * on the grown sequence): rebuilds the partition and every summary of the handle, in
 * place, over each sequence's current mid region [S, N_now - n_recent), with the numbers
 * of clusters and subclusters of the original build (the arena is sized for them).  The
 * recent window restarts as the last n_recent keys, and keys that the sliding window had
 * moved into the clusters are clustered afresh with the rest.  Equivalent to mog_build on
 * the first N_now keys with those explicit C and L.  A serving loop calls it every so many
 * appended tokens.  Enqueued on `stream`; not to overlap a decode or an append on the
 * handle.
 */
int mog_recluster(mog_handle *h, void *stream);

/*
 * mog_decode_ex that also records four caller-created cudaEvent_t (passed as void*), all
 * on `stream`: events[0] before the selection kernel (cluster and subcluster scores, top-k,
 * the Gaussian residual, the row list), events[1] after it, events[2] after the
 * exact-attention rows kernel, events[3] after the merge kernel (which normalises), so
 * that each phase of one decode step can be timed.  The events keep each kernel from
 * starting before its predecessor has finished, so the rows and merge kernels skip the
 * warm-up pass over their own code that mog_decode lets them run while they wait.  Same
 * arguments and results otherwise.
 */
int mog_decode_phased(mog_handle *h, const void *q_dev, float *out_dev,
                      const int32_t *sel_in_dev, int32_t *sel_out_dev, void *const *events,
                      void *stream);

/* Copy the arena layout of a handle. */
int mog_get_layout(const mog_handle *h, mog_layout *out);

/* Synchronise `stream`, then read the device status word: MOG_OK or the recorded error. */
int mog_sync_status(mog_handle *h, void *stream);

/* Split factor (partial results per unit) of the decode's exact-attention kernel. */
int mog_decode_splits(const mog_handle *h, int32_t *splits);

/* Free the host structure of a handle (not the caller's arena or cache).  NULL is a no-op. */
void mog_destroy(mog_handle *h);

/*
 * Full-scan exact decode attention, the comparison path ([IA]: the full KV scan that MoG
 * avoids): for every query head, softmax(tau q.K^T) V over keys [0, N_b).  Query head
 * (b, g*G + i) reads KV head (b, g).
 *  lengths_dev : int32[batch] on the device; n_max >= every length (sizes the launch)
 *  q_dev       : bf16 [batch][h_q][d];  out_dev: f32 [batch][h_q][d]
 *  scratch_dev : device buffer of at least dense_decode_scratch_bytes() bytes (partial
 *                results of the split scan); no initial contents needed
 */
int dense_decode_scratch_bytes(int32_t batch, int32_t h_kv, int32_t h_q, int32_t d,
                               int32_t n_max, size_t *bytes);
int dense_decode(const mog_kv *kv, const int32_t *lengths_dev, int32_t n_max, int32_t batch,
                 int32_t h_kv, int32_t h_q, int32_t d, const void *q_dev, float *out_dev,
                 void *scratch_dev, size_t scratch_bytes, void *stream);

/*
 * dense_decode without a scratch argument.  No counterpart in the papers: this entry point
 * exists for callers that cannot allocate device memory -- for example a serving engine
 * that has handed its whole device budget to a preallocated KV pool and forbids further
 * cudaMalloc, or code that runs where allocation is not allowed or would stall other work.
 * The split partials live in a library-owned static device array of 4 MiB (every GPU that
 * loads the library holds it until the process exits); shapes that need more return
 * MOG_ERR_CAPACITY (mog_last_error states the sizes).  Nothing is allocated, by the
 * library or any routine it calls.
 *  - The first call on a device looks up the array's device address (with that device
 *    current) and caches it under the current CUDA context; a call in a new context (after
 *    cudaDeviceReset, or under another context the caller made current) looks it up again.
 *    Make the first call in each context before any stream capture.
 *  - Every call on a device shares the one array, and each call rewrites all of it that
 *    it reads; calls that overlap on the GPU (other streams, other threads) race.
 * Arguments as dense_decode.
 */
int dense_decode_noalloc(const mog_kv *kv, const int32_t *lengths_dev, int32_t n_max,
                         int32_t batch, int32_t h_kv, int32_t h_q, int32_t d, const void *q_dev,
                         float *out_dev, void *stream);

/*
 * Test export of one first-level k-means assignment step ([IA]'s partition, computed by
 * a Lloyd step): for each of the n rows x_i (bf16, row stride ld elements),
 * assign_out_dev[i] = argmin_c sum_j (x_ij - cent_cj)^2 with the lowest index on ties,
 * decided exactly as the fp64 sum of rounded squares in index order.  The same kernels
 * as mog_build's first level: the distances are scored on the tensor cores (bf16 keys,
 * centroids as bf16 high + low parts, fp32 accumulate); a row whose best centroid is not
 * separated from the others by the scores' error bound is decided by the direct fp32
 * pass, and a row that pass cannot certify by the fp64 rule.  cent_dev: f32 [k][d],
 * k <= 4096.  scratch_dev: 16-byte aligned, at least mog_kmeans_assign_scratch_bytes()
 * bytes.  counts_host (may be NULL; int32[2]) receives the rows decided by the fp64 rule
 * and the rows the tensor-core pass left to the direct pass; with it the call
 * synchronises the stream and reports a device-side failure (MOG_ERR_TIMEOUT,
 * MOG_ERR_DEVICE_CHECK).
 */
int mog_kmeans_assign_scratch_bytes(int32_t n, int32_t k, int32_t d, size_t *bytes);
int mog_kmeans_assign(const void *x_dev, int64_t ld, int32_t n, const float *cent_dev,
                      int32_t k, int32_t d, int32_t *assign_out_dev, void *scratch_dev,
                      size_t scratch_bytes, void *stream, int32_t *counts_host);

/*
 * Test export of one second-level assignment step: n_seg segments, segment s holding
 * rows rows_dev[seg_off[s] .. seg_off[s+1]) of x, assigned among its own k centroids
 * cent_dev[s][k][d] (f32), same decision rule as above.  The same kernel as mog_build's
 * second level.  k <= 32.
 */
int mog_kmeans_assign_segments(const void *x_dev, int64_t ld, const int32_t *rows_dev,
                               const int32_t *seg_off_dev, int32_t n_seg, const float *cent_dev,
                               int32_t k, int32_t d, int32_t *assign_out_dev, void *stream);

/*
 * Build trace: the intermediate states of mog_build's two Lloyd loops ([IA]'s hierarchical
 * partition), for step-by-step comparison with a reference implementation.  Byte offsets
 * into the caller's trace buffer; u = b*h_kv + h indexes units, n_mid is the row stride of
 * the assignment arrays (the longest sequence's mid-region length); mid key i of a unit is
 * position S + i.
 *  l1_cent   f32   [units][iters_l1][c_max][d]: the centroids first-level step t assigned to
 *                  (step 0: the seeds)
 *  l1_assign int32 [units][iters_l1][n_mid]: the cluster of mid key i after step t
 *  l2_cent   f32   [units][c_max][iters_l2][l_max][d]: cluster c's second-level centroids
 *                  used by its step t
 *  l2_assign int32 [units][iters_l2][n_mid]: after second-level step t, the subcluster of
 *                  the cluster member at index j of the unit's members listed by (final
 *                  first-level cluster, position): entry cluster_start(c) + j
 *  l2_steps  int32 [units][c_max]: second-level steps taken by each cluster
 * A level stops early when a step changes no assignment; entries of later steps repeat
 * the last one (first level) or stay zero (second level).  The first level's step count
 * is mog_layout.l1_steps.
 */
typedef struct mog_trace_layout {
    int32_t units, iters_l1, iters_l2, c_max, l_max, d;
    int64_t n_mid;
    int64_t l1_cent, l1_assign, l2_cent, l2_assign, l2_steps;
    int64_t bytes;  /* size of the trace buffer */
} mog_trace_layout;

/* Layout and size of the build trace for these parameters and build lengths. */
int mog_trace_layout_of(const mog_params *p, const int32_t *lengths_host, mog_trace_layout *out);

/*
 * mog_build that also records its build trace (see mog_trace_layout) into trace_dev, a
 * caller-owned device buffer of at least mog_trace_layout_of().bytes bytes, 16-byte
 * aligned.  The clustering and the handle are exactly those of mog_build; the trace
 * costs a copy of the centroids and assignments after every step.  For parity tests.
 */
int mog_build_traced(const mog_kv *kv, const int32_t *lengths_dev, const int32_t *lengths_host,
                     const mog_params *p, void *arena_dev, size_t arena_bytes, void *trace_dev,
                     size_t trace_bytes, void *stream, mog_handle **out);

/*
 * mog_build (or, with trace_dev non-NULL, mog_build_traced) with k-means++ seeds for the
 * first level; p->flags must include MOG_FLAG_KMEANSPP, which mog_build and
 * mog_build_traced reject with MOG_ERR_INVALID_ARG.
 *  draws_dev : float64 [units][c_max] on the device, uniform draws in [0, 1); unit u's
 *              seed r takes draws_dev[u*c_max + r] (c_max = mog_trace_layout_of().c_max,
 *              the largest C_u).  Copied into the arena, so mog_recluster seeds from the
 *              same draws.  A draw outside [0, 1) is clamped into it and sets the status
 *              word (MOG_ERR_DEVICE_CHECK from mog_sync_status).
 *  trace_dev, trace_bytes : as mog_build_traced, or NULL and 0.
 * The seeds are exported in mog_layout.pp_idx.
 */
int mog_build_seeded(const mog_kv *kv, const int32_t *lengths_dev, const int32_t *lengths_host,
                     const mog_params *p, const double *draws_dev, void *arena_dev,
                     size_t arena_bytes, void *trace_dev, size_t trace_bytes, void *stream,
                     mog_handle **out);

/*
 * mog_build with the partition given instead of clustered: perm_dev int32 [units][n_cap]
 * lists each unit's mid positions ordered by (cluster, subcluster, position) and
 * sub_off_dev int32 [units][sub_off_stride] the offsets (C_u*L_u+1 used, relative to the
 * unit's perm row).  Only the summaries are computed.  For parity tests.
 */
int mog_sub_off_stride(const mog_params *p, const int32_t *lengths_host, int64_t *stride);
int mog_build_from_partition(const mog_kv *kv, const int32_t *lengths_dev,
                             const int32_t *lengths_host, const mog_params *p,
                             const int32_t *perm_dev, const int32_t *sub_off_dev,
                             void *arena_dev, size_t arena_bytes, void *stream,
                             mog_handle **out);

/*
 * Self-check of the bounded device waits (no counterpart in the papers).  Every wait of the
 * library's kernels on an mbarrier (the tensor-core assignment's pipeline) gives up after
 * a fixed number of polls, records MOG_ERR_TIMEOUT in the status word and lets the kernel
 * return, so that a lost arrival cannot hang the GPU.  This call runs that same wait on a
 * one-arrival mbarrier with `limit` polls: with arrive != 0 the arrival is made first and
 * the call returns MOG_OK; with arrive == 0 nothing completes the barrier and the call
 * returns MOG_ERR_TIMEOUT, leaving the CUDA context usable.  scratch_dev: one int32 of
 * device memory.  Synchronises `stream`.
 */
int mog_check_bounded_wait(int32_t limit, int32_t arrive, int32_t *scratch_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOG_H */
