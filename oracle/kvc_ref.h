/*
 * kvc_ref.h -- the CPU oracle of the decode-time KV-cache compression event.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, fp64 restatement of the
 * method, written to check the CUDA library against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may call it; the
 * product path never does.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * Sources (page title, then section / equation):
 *  [AMS]  "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning",
 *         Method -- Key designs 1-4, the complete example, and the schedule
 *         defaults under "Loss function / training strategy".
 *  [RKV]  "RefreshKV: Updating Small KV Cache During Long-form Generation",
 *         A2 Method details (max pooling of neighbouring scores before top-K),
 *         A6 Appendix (SnapKV baseline settings: window 1, kernel 7).
 *  [SKV]  "SkipKV: Selective Skipping of KV Generation and Storage for
 *         Efficient Inference with Large Reasoning Models", A2 Method details,
 *         token importance score (query window, GQA map g(i) = floor(i/n),
 *         attention mask M).
 *
 * Conventions.  A "unit" is one (layer, sequence, KV head).  Arrays handed to
 * the batched entry points are unit-major and compact: [U, ...].  bf16 data
 * is passed as its raw 16-bit patterns (uint16_t).  Every cache has T slots;
 * slots [0, pad) are left padding and never take part; slots [pad, T) are the
 * n = T - pad valid positions.
 *
 * Parity pins: every step is pinned by tests/test_oracle_*.py against closed
 * forms, library routines, brute force or the worked example of [AMS].
 */
#ifndef KVC_REF_H
#define KVC_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int group;        /* G: query heads per KV head                         */
  int head_dim;     /* d                                                  */
  int window;       /* W: most recent decode queries                      */
  int budget;       /* T_keep                                             */
  int avg_pool;     /* odd kernel of the mass average pool (5)            */
  int max_pool;     /* odd kernel of the score max pool (7)               */
  float delta;      /* cumulative-mass step (0.1)                         */
  int seg_min;      /* 16                                                 */
  int seg_max;      /* 256                                                */
  int q_min;        /* 1                                                  */
  int n_sink;       /* 4                                                  */
  int n_recent;     /* recent suffix kept                                 */
  float lambda;     /* EMA decay of the credit (0.9)                      */
  float beta;       /* weight of the current mass in the mix (0.9)        */
  float eps;        /* mass floor (1e-6)                                  */
  float softmax_scale; /* 0 => 1/sqrt(head_dim)                           */
  int seg_fixed;    /* ablation: > 0 = fixed-length segments               */
  int quota_by_len; /* ablation: 1 = quotas by segment length, not mass    */
  int global_topk;  /* ablation: 1 = one segment over all valid slots      */
  float redundancy_sigma; /* > 0: select on the redundancy-mixed score    */
} kvc_ref_config;

/* ---- per-unit steps, fp64 (for the pins) -------------------------------- */

/* Step 1: attention usage of the cache by the W most recent queries of the
 * GQA group, summed over queries and heads, unseen suffix entries filled with
 * the window max.  q: [G*W*d] (query j of head h at q[(h*W+j)*d]), k: [T*d].
 * a: [T] (0 on padding).  *fill_out receives the fill value (window max p). */
void kvc_ref_usage(const double* q, const double* k, int G, int W, int d,
                   int T, int pad, double scale, double* a, double* fill_out);

/* Step 1 (score): s = max-pool of a over valid neighbours within kernel/2;
 * padding slots get -inf. */
void kvc_ref_maxpool(const double* a, int T, int pad, int kernel, double* s);

/* Step 2 (pool): u = average pool of a over the valid range, zero outside it,
 * always divided by the kernel size.  Padding slots get 0. */
void kvc_ref_avgpool(const double* a, int T, int pad, int kernel, double* u);

/* Step 2 (mass): m_i = (max(u_i,0)+eps) / sum_v (max(u_v,0)+eps) over valid
 * slots; 0 on padding. */
void kvc_ref_mass_normalize(const double* u, int T, int pad, double eps,
                            double* m);

/* Step 2 (credit): slots [pad+n_carry, T) are new and take c_in := m.
 * c = lambda*c_in + (1-lambda)*m;  m_used = normalize(beta*m +
 * (1-beta)*normalize(c)).  c_out and m_used are 0 on padding. */
void kvc_ref_credit(const double* m, const double* c_in, int T, int pad,
                    int n_carry, double lambda, double beta, double* c_out,
                    double* m_used);

/* Step 3 (boundaries before split/merge): the fixed-point thresholds and
 * b_k = min{t in [1,n] : C(t) >= tau_k}.  Writes up to *n_b boundaries
 * (k = 1..K) to b[]; returns K. */
int kvc_ref_boundaries(const float* m_used, int T, int pad, float delta,
                       int64_t* b, uint64_t* total_out);

/* Step 3 (segments): raw segments from the boundaries, empty ones dropped,
 * merge of short ones, split of long ones.  Starts are valid offsets
 * (0 = first valid slot).  Returns the number of segments. */
int kvc_ref_segments(const float* m_used, int T, int pad, float delta,
                     int seg_min, int seg_max, int32_t* seg_start,
                     int32_t* seg_len, uint64_t* seg_mass);

/* Ablations of [AMS] (Experiments, ablation table): fixed-length segments
 * (seg_fixed > 0) or one segment over all valid slots (global != 0), with the
 * masses recounted as in kvc_ref_segments.  Returns the segment count. */
int kvc_ref_segments_ablation(const float* m_used, int T, int pad, int seg_fixed,
                              int global, int32_t* seg_start, int32_t* seg_len,
                              uint64_t* seg_mass);

/* Step 4 (quotas): exact-integer quotas summing to min(budget, n). */
void kvc_ref_quotas(const int32_t* seg_len, const uint64_t* seg_mass,
                    int n_seg, int budget_eff, int q_min, int32_t* quota);

/* Step 5 (selection): kept absolute slots, ascending; returns n_kept. */
int kvc_ref_select_unit(const float* score, int T, int pad,
                        const int32_t* seg_start, const int32_t* seg_len,
                        const int32_t* quota, int n_seg, int budget,
                        int n_sink, int n_recent, int32_t* kept);

/* ---- batched mirrors of the library entry points (compact [U,...]) ------ */

/* Largest segment count a cache of T slots can produce: max(1, T/seg_min). */
int kvc_ref_s_max(const kvc_ref_config* cfg, int T);

/* Steps 1-2 for U units.  q: [U,G,W,d] bf16 bits; k: [U,T,d] bf16 bits;
 * credit_in: [U,T]; pad, n_carry: [U].  Outputs [U,T] fp32 (rounded from
 * fp64): m_used, score, post-EMA credit. */
int kvc_ref_mass(const kvc_ref_config* cfg, int U, int T, const uint16_t* q,
                 const uint16_t* k, const float* credit_in,
                 const int32_t* pad, const int32_t* n_carry, float* mass,
                 float* score, float* credit_post);

/* Steps 3-4 for U units on the fp32 mass.  Outputs [U,S_max]: starts as
 * ABSOLUTE slots, lengths, quotas; n_seg [U]. */
int kvc_ref_segment_quota(const kvc_ref_config* cfg, int U, int T,
                          const float* mass, const int32_t* pad,
                          int32_t* seg_start, int32_t* seg_len,
                          int32_t* quota, int32_t* n_seg);

/* Step 5 for U units on the fp32 score.  kept_idx: [U,budget], -1 past
 * n_kept; n_kept: [U]. */
int kvc_ref_select(const kvc_ref_config* cfg, int U, int T, const float* score,
                   const int32_t* pad, const int32_t* seg_start,
                   const int32_t* seg_len, const int32_t* quota,
                   const int32_t* n_seg, int32_t* kept_idx, int32_t* n_kept);

/* Step 6 for U units: rows of k, v ([U,T,d] bf16 bits) and credit ([U,T]) at
 * the kept slots; slots past n_kept are zero. */
int kvc_ref_compact(const kvc_ref_config* cfg, int U, int T, const uint16_t* k,
                    const uint16_t* v, const float* credit_post,
                    const int32_t* kept_idx, const int32_t* n_kept,
                    uint16_t* k_out, uint16_t* v_out, float* credit_out);

/* [SKV] token redundancy (after R-KV): for each row i in rows[0..n_rows),
 * r_i = mean over the other valid slots j != i of cos(k_i, k_j); k [T][d]
 * bf16 bits, valid slots [pad, T); a zero key has cosine 0 with every key;
 * r_i = 0 when fewer than two slots are valid. */
void kvc_ref_mean_cosine_rows(const uint16_t* k, int T, int d, int pad, const int32_t* rows,
                              int n_rows, double* r_out);

/* [SKV] redundancy-mixed eviction score of one unit: score [T] (the max-pooled
 * usage, >= 0 on valid slots).  r_out[T] = r (above), R_out[T] = softmax of r
 * over the valid slots, f_out[T] = sigma * s_i / sum_v s_v - (1 - sigma) * R_i;
 * padding slots get r = R = 0 and f = -inf.  Any output may be NULL. */
void kvc_ref_redundancy_score(const uint16_t* k, const float* score, int T, int d, int pad,
                              double sigma, double* r_out, double* R_out, double* f_out);

/* [AMS] Appendix E, paged layout: per-head compaction into newly allocated
 * blocks.  Pools k_pool, v_pool: [L][n_blocks][H][bs][d] bf16 bits (in/out);
 * block tables [B][max_blocks] shared by all layers (logical token t of
 * sequence b lives in block table[b][t / bs], row t % bs); seq_len [B] tokens
 * before the event; pad [B] converts the dense slots of kept_idx
 * ([L][B][H][budget], n_kept [L][B][H]) to logical positions (t = slot - pad).
 * free_list [n_blocks] with *free_top entries free, used as a stack: sequence
 * b takes ceil(n_kept_b / bs) blocks in sequence order from the top, the copy
 * follows, then the ceil(seq_len_b / bs) old blocks are pushed back in
 * sequence order.  table_new [B][max_blocks] gets the new blocks (-1 past
 * them).  Returns 0, or -1 (nothing changed) if the pool cannot supply the
 * blocks or an index is out of range. */
int kvc_ref_compact_paged(int L, int B, int H, int d, int bs, int n_blocks, int max_blocks,
                          int budget, uint16_t* k_pool, uint16_t* v_pool,
                          const int32_t* seq_len, const int32_t* pad,
                          const int32_t* kept_idx, const int32_t* n_kept,
                          const int32_t* table_old, int32_t* table_new,
                          int32_t* free_list, int32_t* free_top);

/* [RefreshKV] query-similarity trigger, per (layer, sequence) row of LB rows:
 * the current token's query averaged over the Hq query heads (q: [LB][Hq][d]
 * bf16 bits) against the reference query of the last full step (q_ref: [LB][d],
 * updated where a refresh is decided).  flag[r] = 1 where the cosine is below
 * `threshold` (or undefined), else 0; sim[r] = the cosine (-2 when undefined). */
void kvc_ref_refresh_decision(int LB, int Hq, int d, const uint16_t* q, double* q_ref,
                              double threshold, int32_t* flag, double* sim);

#ifdef __cplusplus
}
#endif
#endif
