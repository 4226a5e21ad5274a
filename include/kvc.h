/*
 * kvc.h -- C ABI of the GB300 (sm_103a) decode-time KV-cache compression event.
 *
 * The event, per unit = (layer, sequence, KV head), follows
 * "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning" (AMS),
 * Method, Key designs 1-4:
 *   1. attention usage of the cache by the W most recent decode queries of the
 *      unit's GQA group (softmax of q.k/sqrt(d), summed over queries and heads;
 *      causally unseen suffix entries filled with the window maximum);
 *      the base score is the usage max-pooled over 7 neighbours
 *      ("RefreshKV: Updating Small KV Cache During Long-form Generation",
 *      A2 prefilling stage and A6 baseline settings);
 *   2. average pool (5), clamp + eps normalisation to a mass, EMA credit mix;
 *   3. cuts at cumulative-mass multiples of Delta, split/merge to 16..256;
 *   4. exact-integer quotas (q_min + mass share), must-keep sinks and suffix;
 *   5. segment-local top-k, union with must-keep, budget fix-up;
 *   6. sort the kept slots and gather K, V and the credit into a fixed-length
 *      cache.
 *
 * Memory and layout (every tensor pointer below is DEVICE memory, caller
 * owned, C-contiguous, 16-byte aligned, with the layer dimension outermost):
 *   q       [L][B][H*G][W][d]  bf16 (raw 16-bit patterns, uint16_t);
 *                              query head h*G+g belongs to KV head h
 *                              (SkipKV, A2 Method details, 4.1 token importance: g(i)=floor(i/n))
 *   k, v    [L][B][H][T][d]    bf16; slot t of a sequence with left padding
 *                              pad[b] is valid iff t >= pad[b]
 *   credit  [L][B][H][T]       fp32 EMA credit (Key design 1)
 *   pad     [B]                int32 left padding per sequence, 0 <= pad <= T
 *   n_carry [B]                int32: slots [pad, pad+n_carry) carry credit
 *                              from the previous event; later slots are new
 *                              and start at their current mass
 *   mass, score               [L][B][H][T] fp32 (0 / -inf on padding)
 *   seg_start, seg_len, quota [L][B][H][S_max] int32, S_max from
 *                              kvc_stage_sizes; seg_start is an absolute slot
 *   n_seg, n_kept             [L][B][H] int32
 *   kept_idx                  [L][B][H][budget] int32 absolute slots, ascending,
 *                              -1 past n_kept
 *   k_out, v_out              [L][B][H][budget][d] bf16; rows past n_kept = 0
 *   credit_out                [L][B][H][budget] fp32
 * L, B, H, G, W, d come from the handle's config; T (<= max_T) is per call.
 * The window's query j sits at slot T-W+j and sees slots [pad, T-W+j].
 * n_kept = min(budget, T - pad).
 *
 * Calls.  Every entry point validates its arguments on the host and returns a
 * negative KVC_ERR_* code without launching anything if they are wrong.
 * Otherwise it enqueues its kernels on `stream` (a cudaStream_t; NULL = the
 * legacy default stream) and returns KVC_OK without synchronising; device-side
 * conditions are reported through kvc_get_device_status.  No entry point
 * allocates memory except kvc_create.  A handle is not thread-safe and must
 * not be used on two streams at once (it owns one workspace).  Outputs must
 * not alias inputs, except credit_post may alias credit_in in kvc_mass.
 * The caller keeps the logical (RoPE) positions of the kept tokens: the next
 * token's position continues the original progress (AMS, Key design 4).
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define KVC_OK 0
#define KVC_ERR_ARG (-1)         /* null pointer, bad config value           */
#define KVC_ERR_SHAPE (-2)       /* T out of range for this handle           */
#define KVC_ERR_ALIGN (-3)       /* pointer not 16-byte aligned              */
#define KVC_ERR_NOMEM (-4)       /* workspace allocation failed (create)     */
#define KVC_ERR_CUDA (-5)        /* a CUDA runtime call failed               */
#define KVC_ERR_DEVICE (-6)      /* no usable sm_103 device                  */
#define KVC_ERR_TIMEOUT (-7)     /* a bounded device wait gave up            */
#define KVC_ERR_UNSUPPORTED (-8) /* config outside what the kernels handle   */

/* ---- device status bits (kvc_get_device_status) ------------------------ */
#define KVC_STATUS_WAIT_TIMEOUT 0x1u /* an mbarrier wait hit its bound; the
                                        affected outputs are unspecified     */
#define KVC_STATUS_BAD_INDEX 0x2u    /* kvc_compact got a kept index outside
                                        [0, T): that row was written as zeros;
                                        kvc_compact_paged: an index, block or
                                        free-stack entry out of range (nothing
                                        was changed)                          */
#define KVC_STATUS_POOL_EXHAUSTED 0x4u /* kvc_compact_paged: the free stack
                                        held fewer blocks than the compacted
                                        caches need (nothing was changed)     */

/* ---- configuration ------------------------------------------------------ */
typedef struct {
  int n_layers;    /* L                                                    */
  int batch;       /* B                                                    */
  int n_kv_heads;  /* H                                                    */
  int group;       /* G query heads per KV head                            */
  int head_dim;    /* d: 64 or 128                                         */
  int max_T;       /* largest T any call will pass, <= 65536               */
  int window;      /* W: most recent decode queries (128); G*W <= 4096     */
  int budget;      /* T_keep (AMS: 256/512/1024)                           */
  int avg_pool;    /* odd, mass average pool (5)                           */
  int max_pool;    /* odd, score max pool (7)                              */
  float delta;     /* cumulative-mass step, delta >= 1/1024 (0.1)          */
  int seg_min;     /* >= 1 (16)                                            */
  int seg_max;     /* 2*seg_min <= seg_max, 16 <= seg_max <= 4096 (256)    */
  int q_min;       /* 1                                                    */
  int n_sink;      /* 4                                                    */
  int n_recent;    /* recent suffix kept                                   */
  float lambda;    /* credit EMA decay in [0,1] (0.9)                      */
  float beta;      /* current-mass weight in [0,1] (0.9)                   */
  float eps;       /* mass floor > 0 (1e-6)                                */
  float softmax_scale; /* 0 => 1/sqrt(head_dim)                            */
  /* Ablation switches ("Adaptive Mass-Segmented KV Compression for Long-Form
   * Reasoning", Experiments, ablation table: fixed-length segments, no
   * mass-weighted quota, global head-only top-k; "no EMA credit" is
   * beta = 1).  All 0 = the method.                                        */
  int seg_fixed;     /* > 0: segments of seg_fixed valid slots (>= seg_min)
                        instead of mass cut points; a shorter tail joins the
                        segment before it                                   */
  int quota_by_len;  /* 1: quotas in proportion to segment length instead of
                        segment mass (same minimums, rounding, correction)  */
  int global_topk;   /* 1: one segment over all valid slots, quota = budget:
                        per-head top-k on the score plus the must-keep set  */
  /* Second base score (SkipKV, A2 Method details, 4.1 token redundancy score, after R-KV):
   * sigma in (0, 1] selects on sigma*I - (1-sigma)*R instead of the score
   * (see kvc_redundancy_score); 0 = off.  Segments and quotas stay on the
   * attention mass.                                                         */
  float redundancy_sigma;
  /* Tensor-core kernel of step 1 (same results up to fp32 summation order):
   * 1 = one SM per MMA (M128 x N256, two accumulators per SM);
   * 2 = CTA pairs (two SMs of a TPC share each M256 x N128 MMA, four
   *     accumulators per SM, two MMA-issuing threads);
   * 0 = automatic (1: the pairs are as fast on the attention pass over
   *     slots and slower on the one over query rows, whose odd tile count
   *     leaves half of a pair idle). */
  int attn_kernel;
} kvc_config;

typedef struct kvc_handle kvc_handle;

/* Fill *cfg with the method's defaults (AMS schedule: W 128, Delta 0.1,
 * lengths 16/256, q_min 1, 4 sinks, lambda = beta = 0.9; eps 1e-6; pools 5/7)
 * and zero sizes.  The caller sets the sizes and budget. */
void kvc_default_config(kvc_config* cfg);

/* Validate `cfg`, select the current CUDA device (must be sm_103), and
 * allocate the handle and its device workspace (sized from the config's
 * maximum dimensions).  On success *out owns them; free with kvc_destroy. */
int kvc_create(const kvc_config* cfg, kvc_handle** out);

/* Free the handle and its workspace (synchronises the device first). */
void kvc_destroy(kvc_handle* h);

/* *s_max = max(1, T / seg_min): the segment-array stride for this T. */
int kvc_stage_sizes(const kvc_handle* h, int T, int* s_max);

/* Steps 1-2: attention usage, score, mass, credit.
 * Defined by AMS, Method, Key design 1 (usage of each slot by the W most
 * recent queries with the window-maximum fill; the 1-D average pool; the mass
 * equation m = (max(u,0)+eps)/sum; the EMA credit c <- lambda c + (1-lambda) m
 * and the mix m_used = normalize(beta m + (1-beta) normalize(c))), and by
 * RefreshKV, A2 and A6 (the score: usage max-pooled over 7 neighbours).
 *   mass, score, credit_post  [L][B][H][T] fp32 out; padding gets mass 0,
 *   score -inf, credit 0.  Slots at or after pad+n_carry start their credit at
 *   their current mass (the credit convention of this library).
 * Uses the handle's workspace for per-query softmax statistics and the raw
 * usage.  credit_in is read, credit_post written (they may be the same buffer).
 * Host-detectable errors (null or unaligned pointer, T outside [1, max_T])
 * return a negative code and launch nothing; a bounded wait that runs out sets
 * KVC_STATUS_WAIT_TIMEOUT in the status word. */
int kvc_mass(kvc_handle* h, const uint16_t* q, const uint16_t* k, int T,
             const int32_t* pad, const int32_t* n_carry,
             const float* credit_in, float* credit_post, float* mass,
             float* score, void* stream);

/* Steps 3-4: segmentation and quotas on the fp32 mass.
 * Defined by AMS, Method, Key design 2 (cumulative mass C(t), cut points
 * b_k = min{t : C(t) >= k Delta}, short segments merged and long ones split)
 * and Key design 3 (quota = q_min + the mass-proportional share of the rest of
 * the budget, clipped to the segment and corrected to the exact budget).
 * Bit-exact integer arithmetic (40-bit fixed-point mass, exact rational
 * comparisons).
 *   mass       [L][B][H][T] fp32 (kvc_mass's m_used);
 *   seg_start, seg_len, quota  [L][B][H][S_max] int32 out, S_max from
 *              kvc_stage_sizes; seg_start is an absolute slot; entries past
 *              n_seg are zero;
 *   n_seg      [L][B][H] int32 out (0 for an all-padding sequence).
 * A cache no longer than the budget gets quota = length everywhere. */
int kvc_segment_quota(kvc_handle* h, const float* mass, int T,
                      const int32_t* pad, int32_t* seg_start,
                      int32_t* seg_len, int32_t* quota, int32_t* n_seg,
                      void* stream);

/* Step 5 (and the index sort of step 6): kept slots per unit.
 * Defined by AMS, Method, Key design 3 (must-keep: the first n_sink valid
 * slots and the last n_recent, counted inside their own segment's quota; the
 * worked example of section "A complete example") and Key design 4 (each
 * segment keeps its best non-must-keep slots by score, up to its quota; the
 * union with must-keep, over-budget removal of the globally worst picks, kept
 * slots sorted ascending).
 *   score      [L][B][H][T] fp32 (ties go to the lower slot);
 *   seg_*      as kvc_segment_quota writes them;
 *   kept_idx   [L][B][H][budget] int32 out, ascending, -1 past n_kept;
 *   n_kept     [L][B][H] int32 out = min(budget, valid slots). */
int kvc_select(kvc_handle* h, const float* score, int T, const int32_t* pad,
               const int32_t* seg_start, const int32_t* seg_len,
               const int32_t* quota, const int32_t* n_seg, int32_t* kept_idx,
               int32_t* n_kept, void* stream);

/* Step 6: gather K, V and the post-EMA credit at the kept slots.
 * Defined by AMS, Method, Key design 4 (physical compaction into a fixed-length
 * per-head cache, not a mask) and Key design 1 (the credit stays aligned with
 * the slots it describes, so it follows the same indices).
 *   k_out, v_out  [L][B][H][budget][d] bf16 out; credit_out [L][B][H][budget]
 *   fp32 out; rows past n_kept are zero.  k_out/v_out must not alias k/v.
 * An index outside [0, T) writes a zero row and sets KVC_STATUS_BAD_INDEX. */
int kvc_compact(kvc_handle* h, const uint16_t* k, const uint16_t* v,
                const float* credit_post, int T, const int32_t* kept_idx,
                const int32_t* n_kept, uint16_t* k_out, uint16_t* v_out,
                float* credit_out, void* stream);

/* Second base score ("SkipKV: Selective Skipping of KV Generation and Storage
 * for Efficient Inference with Large Reasoning Models", A2 Method details, 4.1:
 * the token redundancy score after R-KV, and
 * the final eviction score without its sentence term), for every unit:
 *   r_i = mean over the other valid slots j != i of cos(k_i, k_j)
 *         (a zero key has cosine 0 with every key; r = 0 below two valid slots),
 *   R_i = exp(r_i) / sum over valid v of exp(r_v),
 *   I_i = score_i / sum over valid v of score_v   (0 when that sum is 0),
 *   sel_score_i = sigma * I_i - (1 - sigma) * R_i,  sigma = cfg.redundancy_sigma;
 * padding slots get sel_score = -inf and redundancy = 0.  Computed in O(T d)
 * per unit through sum_j cos(k_i, k_j) = (k_i/|k_i|) . (sum_j k_j/|k_j|) - 1,
 * fp32 arithmetic.
 *   k          [L][B][H][T][d] bf16, as for kvc_mass;
 *   score      [L][B][H][T] fp32, >= 0 on valid slots (kvc_mass's score);
 *   sel_score  [L][B][H][T] fp32 out (may alias score);
 *   redundancy [L][B][H][T] fp32 out, R; may be NULL.
 * Uses the handle's workspace as scratch (two fp32 values per slot).
 * Needs cfg.redundancy_sigma > 0 (else KVC_ERR_ARG).  kvc_event runs it between
 * steps 4 and 5 whenever redundancy_sigma > 0; segments and quotas stay on the
 * attention mass.  Device pointers, caller-owned; asynchronous on `stream`. */
int kvc_redundancy_score(kvc_handle* h, const uint16_t* k, const float* score, int T,
                         const int32_t* pad, float* sel_score, float* redundancy,
                         void* stream);

/* Steps 1-5 in one call: kvc_mass, kvc_segment_quota and kvc_select chained,
 * with every intermediate written to the caller's buffers.
 * Defined by AMS, Method, Key designs 1-4 up to the kept set (usage and mass,
 * cut points, quotas and must-keep, in-segment selection), with the RefreshKV
 * A2/A6 score, and by the overhead statement of the same section (mass
 * processing and the prefix sum are O(H_kv T) work after the attention).  For
 * T <= 4096 the mass, segmentation and selection run as one launch (one CTA
 * per unit, mass, score and segments held in shared memory between the
 * steps); every output is bit-identical to the three stage calls.  With
 * cfg.redundancy_sigma > 0, or longer units, the stage kernels run in turn and
 * score is overwritten by kvc_redundancy_score's mix before the selection.
 * For callers that compact on their own (kvc_compact_paged).
 *   q, k, pad, n_carry, credit_in, credit_post, mass, score  as for kvc_mass;
 *   seg_start, seg_len, quota, n_seg  as kvc_segment_quota writes them;
 *   kept_idx, n_kept  as kvc_select writes them.
 * Device pointers, caller-owned, 16-byte aligned; asynchronous on `stream`;
 * the errors of kvc_mass. */
int kvc_mass_select(kvc_handle* h, const uint16_t* q, const uint16_t* k, int T,
                    const int32_t* pad, const int32_t* n_carry,
                    const float* credit_in, float* credit_post, float* mass,
                    float* score, int32_t* seg_start, int32_t* seg_len,
                    int32_t* quota, int32_t* n_seg, int32_t* kept_idx,
                    int32_t* n_kept, void* stream);

/* The whole event, steps 1-6, with the intermediates in the workspace.
 * Defined by AMS, Method, Key designs 1-4 in order (usage and mass, cut points,
 * quotas and must-keep, in-segment selection and physical compaction), with the
 * RefreshKV A2/A6 score: kvc_mass_select, then kvc_compact, with the same
 * bits as the stage entry points chained; the arguments are those of kvc_mass
 * and kvc_compact.  With
 * cfg.redundancy_sigma > 0, step 5 selects on kvc_redundancy_score's mix. */
int kvc_event(kvc_handle* h, const uint16_t* q, const uint16_t* k,
              const uint16_t* v, int T, const int32_t* pad,
              const int32_t* n_carry, const float* credit_in,
              uint16_t* k_out, uint16_t* v_out, float* credit_out,
              int32_t* kept_idx, int32_t* n_kept, void* stream);

/* The whole event from host buffers, pipelined over groups of layers.
 * No counterpart in the pages: the deployment path when the caches live in
 * host memory.  The layer-major layout makes each group of layers one
 * contiguous slab of every tensor; the slabs of group g+1 are copied host ->
 * device on one of the handle's copy streams while group g's event runs on
 * `stream`, and group g-1's outputs go device -> host on two others (each
 * slab in two halves: one device -> host stream alone moves far less).  Every
 * pointer is as for kvc_event (device ones 16-byte aligned); host buffers
 * should be page-locked for the copies to overlap.  The device input and
 * output buffers are the caller's, full size ([L][...]).  layers_per_stage >= 1
 * is rounded up so that every slab starts on a 16-byte boundary (at most 64
 * stages); the last stage is kept as small as that allows, since its event and
 * copies back are all that follows the last host -> device copy.  The host
 * link bounds the whole call; small stages (1-2 layers of a 28-layer event)
 * shorten the pipeline's fill and tail and were measured fastest.  V is read only
 * at the kept rows: when v_host is page-locked and mapped into the device's
 * address space, the gather reads those rows from it directly and v_dev is
 * neither copied into nor read.  When the call returns the work is queued; everything, the last
 * host copy included, is complete once `stream` is.  Uses cudaMemcpyAsync. */
typedef struct {
  const uint16_t* q_host;      uint16_t* q_dev;       /* [L][B][H*G][W][d] */
  const uint16_t* k_host;      uint16_t* k_dev;       /* [L][B][H][T][d]   */
  const uint16_t* v_host;      uint16_t* v_dev;
  const int32_t* pad_host;     int32_t* pad_dev;      /* [B] */
  const int32_t* n_carry_host; int32_t* n_carry_dev;  /* [B] */
  const float* credit_host;    float* credit_dev;     /* [L][B][H][T] */
  uint16_t* k_out_dev;         uint16_t* k_out_host;  /* [L][B][H][budget][d] */
  uint16_t* v_out_dev;         uint16_t* v_out_host;
  float* credit_out_dev;       float* credit_out_host;  /* [L][B][H][budget] */
  int32_t* kept_idx_dev;       int32_t* kept_idx_host;  /* [L][B][H][budget] */
  int32_t* n_kept_dev;         int32_t* n_kept_host;    /* [L][B][H] */
} kvc_host_buffers;

int kvc_event_host(kvc_handle* h, const kvc_host_buffers* io, int T, int layers_per_stage,
                   void* stream);

/* Step 6 into a paged KV pool ("Adaptive Mass-Segmented KV Compression for
 * Long-Form Reasoning", Appendix E): new blocks are taken from a free stack,
 * each head's kept rows are copied from their original positions into the
 * new physical slots, the sequence's new block table is written and its old
 * blocks are pushed back onto the stack.
 *   k_pool, v_pool  [L][n_blocks][H][block_size][d] bf16, in/out: logical
 *                   token t of sequence b, layer l, head h is row t % bs of
 *                   block table[b][t / bs] (one table per sequence, shared by
 *                   all layers);
 *   seq_len [B]     tokens per sequence before the event;
 *   pad [B]         as for the other entry points: kept_idx holds dense slots,
 *                   the logical position is slot - pad[b];
 *   kept_idx, n_kept  from kvc_select / kvc_event ([L][B][H][budget], [L][B][H];
 *                   n_kept must be the same for every layer and head of a
 *                   sequence, as the method makes it);
 *   credit_post [L][B][H][T] -> credit_out [L][B][H][budget] (dense, as in
 *                   kvc_compact; slots past n_kept are 0);
 *   table_old [B][max_blocks] in, table_new [B][max_blocks] out (-1 past the
 *                   ceil(n_kept / bs) new blocks);
 *   free_list [n_blocks] and *free_top (device int32), in/out: entries
 *                   [0, *free_top) are free; sequence b takes the next
 *                   ceil(n_kept_b / bs) entries below the top in sequence
 *                   order (deterministic), and its ceil(seq_len_b / bs) old
 *                   blocks are pushed back afterwards in sequence order.
 * block_size >= 1, n_blocks >= 1, max_blocks >= 1, T as for kvc_compact.  On a
 * device-side failure nothing is changed and KVC_STATUS_POOL_EXHAUSTED or
 * KVC_STATUS_BAD_INDEX is set (kvc_get_device_status).  The pools must not be
 * used by other work on other streams during the call; asynchronous on
 * `stream`; no allocation. */
int kvc_compact_paged(kvc_handle* h, uint16_t* k_pool, uint16_t* v_pool, int n_blocks,
                      int block_size, int max_blocks, const int32_t* seq_len,
                      const int32_t* pad, const int32_t* kept_idx, const int32_t* n_kept,
                      const float* credit_post, int T, float* credit_out,
                      const int32_t* table_old, int32_t* table_new, int32_t* free_list,
                      int32_t* free_top, void* stream);

/* Query-similarity refresh trigger ("RefreshKV: Updating Small KV Cache During
 * Long-form Generation", dynamic scheduling): for every (layer, sequence), the
 * cosine similarity between the current decode token's query averaged over the
 * H*G query heads and the reference query of that layer's last full step;
 * below `threshold` a full (refresh) step is decided and the reference becomes
 * the current averaged query.  A zero reference (none yet) or a zero query
 * decides a refresh.  Called by the runtime every S-th decode step.
 *   q      [L][B][H*G][d] bf16: the current token's queries (device);
 *   q_ref  [L][B][d] fp32, in/out: reference queries, zero before any full step;
 *   flag   [L][B] int32 out: 1 = take a full step / refresh, 0 = keep decoding
 *          from the compressed cache;
 *   sim    [L][B] fp32 out: the cosine (-2 where it is undefined).
 * threshold in [-1, 1], else KVC_ERR_ARG.  Device pointers, 16-byte aligned,
 * caller-owned; asynchronous on `stream`; no allocation. */
int kvc_refresh_decision(kvc_handle* h, const uint16_t* q, float* q_ref, float threshold,
                         int32_t* flag, float* sim, void* stream);

/* ---- failure-path self-test -------------------------------------------
 * No counterpart in the pages: a check of the library's own failure path.
 * Launches one thread that waits, through the same bounded mbarrier wait the
 * pipelined kernels use, on a barrier that nothing completes.  The wait gives
 * up after its limit (about 2 s), sets KVC_STATUS_WAIT_TIMEOUT in the device
 * status word and the kernel returns normally: nothing traps or hangs and the
 * CUDA context stays usable.  kvc_get_device_status then reports the bit (and
 * clears it).  Asynchronous on `stream`. */
int kvc_wait_self_test(kvc_handle* h, void* stream);

/* ---- tracing -------------------------------------------------------------
 * While enabled, every entry point records a CUDA event on its stream after
 * each kernel it launches (and one before the first), so that the time of each
 * kernel launch is known without a profiler.  Recording costs about a
 * microsecond per kernel and never synchronises.  kvc_profile_read waits for
 * the recorded events, then reports per kernel its launch count and summed
 * duration (ms, event to event on the launch stream). */
typedef struct {
  const char* name;   /* static string owned by the library */
  int launches;
  double total_ms;
} kvc_kernel_time;

/* enable != 0 starts recording (clearing earlier totals); 0 stops. */
int kvc_profile(kvc_handle* h, int enable);

/* Copy up to `capacity` per-kernel totals into out[], the count into *n_out;
 * reset != 0 clears the totals afterwards. */
int kvc_profile_read(kvc_handle* h, kvc_kernel_time* out, int capacity,
                     int* n_out, int reset);

/* ---- no-allocation variant ----------------------------------------------
 * No counterpart in the pages: this is a deployment aid.  kvc_mass_noalloc
 * computes exactly what kvc_mass computes (same kernels, same results) for
 * callers that cannot allocate device memory when they compress -- e.g. an
 * engine that has reserved all free memory for its KV pool -- so it takes no
 * handle and never allocates.  Its scratch is a fixed device array of
 * KVC_NOALLOC_SCRATCH_FLOATS floats (4 MiB) that every GPU loading this
 * library holds until the process exits; a call needs
 * about n_layers*batch*n_kv_heads * (2*group*window + T) floats and returns
 * KVC_ERR_SHAPE (with a message on stderr) above that -- call it per layer or
 * on fewer sequences then.  The config fields kvc_mass uses are checked as in
 * kvc_create; q, k, pad, n_carry, credit_in, credit_post, mass, score are as in
 * kvc_mass.
 * status: device uint32 (required; NULL returns KVC_ERR_ARG) that the kernels
 * OR their KVC_STATUS_* bits into; the caller zeroes it and reads it after the
 * stream completes.
 * The first call on a device (with it current) looks up the scratch address
 * with cudaGetSymbolAddress and caches it per device; make that first call
 * before any stream capture.  The cached address belongs to the device's
 * primary context: after cudaDeviceReset on that device, do not call this
 * entry point on it again in the same process.
 * Every call shares the scratch: calls that overlap on the GPU race. */
#define KVC_NOALLOC_SCRATCH_FLOATS (1u << 20)
int kvc_mass_noalloc(const kvc_config* cfg, const uint16_t* q, const uint16_t* k,
                     int T, const int32_t* pad, const int32_t* n_carry,
                     const float* credit_in, float* credit_post, float* mass,
                     float* score, uint32_t* status, void* stream);

/* Synchronise `stream`, then read and clear the device status bits. */
int kvc_get_device_status(kvc_handle* h, uint32_t* bits, void* stream);

/* Human-readable text of the last error on this handle ("" if none). */
const char* kvc_last_error(const kvc_handle* h);

/* Name of a KVC_* status code. */
const char* kvc_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
