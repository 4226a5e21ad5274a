/*
 * kvc_ref.c -- CPU oracle of the decode-time KV-cache compression event.
 *
 * TEST INFRASTRUCTURE ONLY (see kvc_ref.h).  Plain loops in fp64, one unit at
 * a time, in the order the method states its steps.  No blocking, no fusion,
 * no reordering beyond the definitions.  Where the pages leave a step open,
 * the reading taken is marked [R] and explained next to the code.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off -fPIC -shared kvc_ref.c -lm
 * (-ffp-contract=off: the segmentation thresholds are defined as separately
 * rounded double products.)
 */
#include "kvc_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* helpers                                                                    */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> double (exact: bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double config_scale(const kvc_ref_config* cfg) {
  if (cfg->softmax_scale > 0.0f) return (double)cfg->softmax_scale;
  return 1.0 / sqrt((double)cfg->head_dim);
}

/* ------------------------------------------------------------------------ */
/* Step 1: attention usage from the window queries                           */
/* ------------------------------------------------------------------------ */

/*
 * [AMS] Key design 1: the attention that the W most recent decode queries pay
 * to each cache position; entries a query cannot see because of the causal
 * mask are filled with the window's maximum score, so that new positions are
 * not penalised for having been observed fewer times.
 * [SKV] token importance: query window Q [H_q, alpha, d] against K [H_k, N', d];
 * query head i reads KV head g(i) = floor(i/n); M masks padding.
 *
 * Readings:
 *  [R] query j (0-based) of the window sits at slot T-W+j, so it sees slots
 *      [pad, T-W+j] (causal), the scale is the usual 1/sqrt(d);
 *  [R] a query whose slot lies in the padding is absent: it adds nothing;
 *  [R] "window max score" = the largest softmax probability observed over
 *      every (head, query, seen slot) of the unit;
 *  [R] usage is summed over the window queries and the group's heads.
 */
void kvc_ref_usage(const double* q, const double* k, int G, int W, int d,
                   int T, int pad, double scale, double* a, double* fill_out) {
  double* z = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  int* unseen_count = (int*)calloc((size_t)(T > 0 ? T : 1), sizeof(int));
  double p_max = 0.0;
  for (int i = 0; i < T; ++i) a[i] = 0.0;

  for (int h = 0; h < G; ++h) {
    for (int j = 0; j < W; ++j) {
      const int qpos = T - W + j;
      if (qpos < pad) continue; /* absent query */
      const double* qv = q + ((size_t)h * W + j) * d;
      double zmax = -INFINITY;
      for (int i = pad; i <= qpos; ++i) {
        const double* kv = k + (size_t)i * d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += qv[e] * kv[e];
        z[i] = scale * dot;
        if (z[i] > zmax) zmax = z[i];
      }
      double Z = 0.0;
      for (int i = pad; i <= qpos; ++i) Z += exp(z[i] - zmax);
      for (int i = pad; i <= qpos; ++i) {
        const double p = exp(z[i] - zmax) / Z;
        a[i] += p;
        if (p > p_max) p_max = p;
      }
      for (int i = qpos + 1; i < T; ++i) unseen_count[i] += 1;
    }
  }
  for (int i = pad; i < T; ++i) a[i] += p_max * (double)unseen_count[i];
  if (fill_out) *fill_out = p_max;
  free(z);
  free(unseen_count);
}

/*
 * Base score.  [RKV] A2: top-K is chosen on attention scores max-pooled over
 * neighbouring tokens (SnapKV); A6: kernel size 7.  [AMS] Key design 4: the
 * base scorer ranks candidates inside a segment, shape [B, H_kv, T].
 * [R] the pool runs over the valid slots only; padding gets -inf.
 */
void kvc_ref_maxpool(const double* a, int T, int pad, int kernel, double* s) {
  const int r = kernel / 2;
  for (int i = 0; i < T; ++i) {
    if (i < pad) {
      s[i] = -INFINITY;
      continue;
    }
    double best = -INFINITY;
    for (int t = i - r; t <= i + r; ++t) {
      if (t < pad || t >= T) continue;
      if (a[t] > best) best = a[t];
    }
    s[i] = best;
  }
}

/*
 * [AMS] Key design 1: a small 1-D average pool along the sequence damps local
 * noise.  [R] zero outside the valid range, always divided by the kernel size.
 */
void kvc_ref_avgpool(const double* a, int T, int pad, int kernel, double* u) {
  const int r = kernel / 2;
  for (int i = 0; i < T; ++i) {
    if (i < pad) {
      u[i] = 0.0;
      continue;
    }
    double sum = 0.0;
    for (int t = i - r; t <= i + r; ++t) {
      if (t < pad || t >= T) continue;
      sum += a[t];
    }
    u[i] = sum / (double)kernel;
  }
}

/*
 * [AMS] Key design 1, mass equation:
 *   m_i = (max(u_i,0) + eps) / sum_v (max(u_v,0) + eps),  eps > 0.
 */
void kvc_ref_mass_normalize(const double* u, int T, int pad, double eps,
                            double* m) {
  double total = 0.0;
  for (int i = pad; i < T; ++i) total += (u[i] > 0.0 ? u[i] : 0.0) + eps;
  for (int i = 0; i < T; ++i) {
    if (i < pad) {
      m[i] = 0.0;
      continue;
    }
    m[i] = ((u[i] > 0.0 ? u[i] : 0.0) + eps) / total;
  }
}

/*
 * [AMS] Key design 1, history smoothing:
 *   c <- lambda c + (1-lambda) m,   m_used = normalize(beta m + (1-beta) normalize(c)).
 * The credit must stay aligned with the cache slots; the pages do not spell
 * out the re-indexing, so the convention is: the credit is compacted with the
 * kept indices (step 6), and slots that are new since the last event start at
 * their current mass.  Slots [pad, pad+n_carry) carry credit.
 * [R] if sum(c) == 0, normalize(c) is taken as m (cannot happen once m > 0).
 */
void kvc_ref_credit(const double* m, const double* c_in, int T, int pad,
                    int n_carry, double lambda, double beta, double* c_out,
                    double* m_used) {
  const int n = T - pad;
  if (n_carry < 0) n_carry = 0;
  if (n_carry > n) n_carry = n;
  double c_total = 0.0;
  for (int i = 0; i < T; ++i) {
    if (i < pad) {
      c_out[i] = 0.0;
      continue;
    }
    const double prior = (i < pad + n_carry) ? c_in[i] : m[i];
    c_out[i] = lambda * prior + (1.0 - lambda) * m[i];
    c_total += c_out[i];
  }
  double mix_total = 0.0;
  for (int i = pad; i < T; ++i) {
    const double c_norm = (c_total > 0.0) ? c_out[i] / c_total : m[i];
    m_used[i] = beta * m[i] + (1.0 - beta) * c_norm;
    mix_total += m_used[i];
  }
  for (int i = 0; i < T; ++i) {
    if (i < pad) {
      m_used[i] = 0.0;
      continue;
    }
    m_used[i] = m_used[i] / mix_total;
  }
}

/* ------------------------------------------------------------------------ */
/* Step 3: cumulative-mass segmentation                                       */
/* ------------------------------------------------------------------------ */

/* Fixed-point mass: mu_i = trunc(m_i * 2^40).  Exact for fp32 m_i <= 1. */
static uint64_t fixed_mass(float m) {
  const double scaled = ldexp((double)m, 40);
  if (!(scaled > 0.0)) return 0;
  return (uint64_t)scaled; /* C truncates toward zero */
}

/*
 * [AMS] Key design 2: C(t) = sum_{u<=t} m_u,  b_k = min{ t | C(t) >= k*Delta }.
 * [R] To make the cut points reproducible bit for bit, masses are rounded to
 * fp32 (the interface type) and then to 40-bit fixed point; thresholds are
 * tau_k = ceil( fl( fl(k*Delta) * S ) ) with S the fixed-point total, for all
 * k >= 1 with fl(k*Delta) < 1.  t runs over 1..n (valid slots in order).
 */
int kvc_ref_boundaries(const float* m_used, int T, int pad, float delta,
                       int64_t* b, uint64_t* total_out) {
  const int n = T - pad;
  const double dd = (double)delta;
  uint64_t S = 0;
  for (int v = 0; v < n; ++v) S += fixed_mass(m_used[pad + v]);
  if (total_out) *total_out = S;
  if (n <= 0) return 0;
  int K = 0;
  for (int kk = 1;; ++kk) {
    const double frac = (double)kk * dd;
    if (!(frac < 1.0)) break;
    const double prod = frac * (double)S;
    const uint64_t tau = (uint64_t)ceil(prod);
    uint64_t C = 0;
    int64_t bk = n; /* C(n) = S >= tau always holds */
    for (int t = 1; t <= n; ++t) {
      C += fixed_mass(m_used[pad + t - 1]);
      if (C >= tau) {
        bk = t;
        break;
      }
    }
    b[K++] = bk;
  }
  return K;
}

int kvc_ref_s_max(const kvc_ref_config* cfg, int T) {
  const int s = T / cfg->seg_min;
  return s > 1 ? s : 1;
}

/*
 * [AMS] Key design 2, split/merge heuristic: segments longer than the maximum
 * are cut into near-equal parts, short adjacent segments are merged, and the
 * segment masses are recounted afterwards.  Lengths 16..256 by default.
 * Readings:
 *  [R] empty raw segments (repeated boundaries) are dropped;
 *  [R] merge first, left to right: a segment shorter than seg_min absorbs its
 *      successors until it reaches seg_min; a short last segment joins its
 *      predecessor;
 *  [R] then a segment of length L > seg_max becomes c = ceil(L/seg_max)
 *      parts, the first (L mod c) of length floor(L/c)+1, the rest floor(L/c).
 * Starts are valid offsets (0 = slot pad).
 */
int kvc_ref_segments(const float* m_used, int T, int pad, float delta,
                     int seg_min, int seg_max, int32_t* seg_start,
                     int32_t* seg_len, uint64_t* seg_mass) {
  const int n = T - pad;
  if (n <= 0) return 0;
  /* boundaries: at most 1/delta + 1 of them */
  int64_t* b = (int64_t*)malloc(sizeof(int64_t) * (size_t)(1.0 / (double)delta + 2.0));
  const int K = kvc_ref_boundaries(m_used, T, pad, delta, b, NULL);

  /* raw segments */
  int32_t* raw_start = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K + 1));
  int32_t* raw_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K + 1));
  int n_raw = 0;
  int64_t prev = 0;
  for (int kk = 0; kk < K; ++kk) {
    if (b[kk] > prev) {
      raw_start[n_raw] = (int32_t)prev;
      raw_len[n_raw] = (int32_t)(b[kk] - prev);
      ++n_raw;
      prev = b[kk];
    }
  }
  if (prev < n) {
    raw_start[n_raw] = (int32_t)prev;
    raw_len[n_raw] = (int32_t)(n - prev);
    ++n_raw;
  }

  /* merge */
  int32_t* mer_start = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_raw);
  int32_t* mer_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_raw);
  int n_mer = 0;
  int32_t cur_start = raw_start[0], cur_len = raw_len[0];
  for (int r = 1; r < n_raw; ++r) {
    if (cur_len < seg_min) {
      cur_len += raw_len[r];
    } else {
      mer_start[n_mer] = cur_start;
      mer_len[n_mer] = cur_len;
      ++n_mer;
      cur_start = raw_start[r];
      cur_len = raw_len[r];
    }
  }
  if (cur_len < seg_min && n_mer > 0) {
    mer_len[n_mer - 1] += cur_len;
  } else {
    mer_start[n_mer] = cur_start;
    mer_len[n_mer] = cur_len;
    ++n_mer;
  }

  /* split */
  int n_seg = 0;
  for (int r = 0; r < n_mer; ++r) {
    const int L = mer_len[r];
    if (L <= seg_max) {
      seg_start[n_seg] = mer_start[r];
      seg_len[n_seg] = L;
      ++n_seg;
      continue;
    }
    const int c = (L + seg_max - 1) / seg_max;
    const int base = L / c, extra = L % c;
    int s = mer_start[r];
    for (int part = 0; part < c; ++part) {
      const int len = base + (part < extra ? 1 : 0);
      seg_start[n_seg] = s;
      seg_len[n_seg] = len;
      ++n_seg;
      s += len;
    }
  }

  /* recount the segment masses */
  for (int s = 0; s < n_seg; ++s) {
    uint64_t M = 0;
    for (int v = seg_start[s]; v < seg_start[s] + seg_len[s]; ++v)
      M += fixed_mass(m_used[pad + v]);
    seg_mass[s] = M;
  }
  free(b);
  free(raw_start);
  free(raw_len);
  free(mer_start);
  free(mer_len);
  return n_seg;
}

/*
 * [AMS] Experiments, ablation table: the method without adaptive cut points
 * ("fixed-length segments"), without mass-weighted quotas, and as a global
 * head-only top-k ("no EMA credit" is beta = 1 in kvc_ref_credit).  The pages
 * name the ablations but not their details.
 * Readings:
 *  [R] fixed-length segments: consecutive runs of seg_fixed valid slots from
 *      the first valid slot; a shorter tail joins the segment before it (a
 *      single segment when n < seg_fixed); no merge or split;
 *  [R] global head-only top-k: one segment over all n valid slots, so its
 *      quota is the whole budget; must-keep and selection are unchanged;
 *  [R] no mass-weighted quota: kvc_ref_quotas with each segment's length in
 *      place of its mass (see kvc_ref_segment_quota).
 */
int kvc_ref_segments_ablation(const float* m_used, int T, int pad, int seg_fixed,
                              int global, int32_t* seg_start, int32_t* seg_len,
                              uint64_t* seg_mass) {
  const int n = T - pad;
  if (n <= 0) return 0;
  int n_seg = 1;
  if (global) {
    seg_start[0] = 0;
    seg_len[0] = n;
  } else {
    n_seg = n / seg_fixed;
    if (n_seg < 1) n_seg = 1;
    for (int s = 0; s < n_seg; ++s) {
      seg_start[s] = s * seg_fixed;
      seg_len[s] = (s + 1 < n_seg) ? seg_fixed : n - s * seg_fixed;
    }
  }
  for (int s = 0; s < n_seg; ++s) {
    uint64_t M = 0;
    for (int v = seg_start[s]; v < seg_start[s] + seg_len[s]; ++v)
      M += fixed_mass(m_used[pad + v]);
    seg_mass[s] = M;
  }
  return n_seg;
}

/* ------------------------------------------------------------------------ */
/* Step 4: quotas                                                             */
/* ------------------------------------------------------------------------ */

/*
 * [AMS] Key design 3:
 *   q_i^min = min(q_min, L_i),  T_rem = T_keep - sum_i q_i^min,
 *   q_i = q_i^min + round(T_rem * M_i / sum_j M_j),
 * then clipped to L_i and corrected so that the quotas sum to the budget.
 * The minimum quotas need a feasible budget.
 * Readings (all integer, so that the result is exact):
 *  [R] the budget is min(T_keep, n) (a short cache keeps everything);
 *  [R] infeasible minimums (sum q^min > budget): segments in descending mass
 *      order (ties: lower index first) receive their minimum while budget
 *      remains; the others get 0;
 *  [R] round = round half up: floor((2*T_rem*M_i + sum M) / (2 sum M));
 *  [R] correction one unit at a time on the exact remainder
 *      delta_i = (q_i^min sum M + T_rem M_i) - q_i sum M:
 *      short  -> +1 to the segment with q_i < L_i and the largest delta_i
 *                (ties: lower index);
 *      over   -> -1 to the segment with q_i > q_i^min and the smallest
 *                delta_i (ties: higher index).
 */
void kvc_ref_quotas(const int32_t* seg_len, const uint64_t* seg_mass,
                    int n_seg, int budget_eff, int q_min, int32_t* quota) {
  if (n_seg <= 0) return;
  int32_t* q_floor = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_seg);
  int64_t* rem = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_seg);
  uint64_t M_total = 0;
  int64_t floor_total = 0;
  for (int s = 0; s < n_seg; ++s) {
    q_floor[s] = q_min < seg_len[s] ? q_min : seg_len[s];
    floor_total += q_floor[s];
    M_total += seg_mass[s];
  }

  if (floor_total > budget_eff) {
    /* infeasible minimums: hand them out in descending mass order */
    char* done = (char*)calloc((size_t)n_seg, 1);
    int64_t left = budget_eff;
    for (int round_ = 0; round_ < n_seg; ++round_) {
      int best = -1;
      for (int s = 0; s < n_seg; ++s) {
        if (done[s]) continue;
        if (best < 0 || seg_mass[s] > seg_mass[best]) best = s;
      }
      done[best] = 1;
      const int64_t give = q_floor[best] < left ? q_floor[best] : left;
      q_floor[best] = (int32_t)give;
      left -= give;
    }
    free(done);
    floor_total = budget_eff;
  }

  const int64_t T_rem = (int64_t)budget_eff - floor_total;
  int64_t total = 0;
  for (int s = 0; s < n_seg; ++s) {
    int64_t share = 0;
    if (M_total > 0) {
      const uint64_t num = 2ull * (uint64_t)T_rem * seg_mass[s] + M_total;
      share = (int64_t)(num / (2ull * M_total));
    }
    int64_t qs = q_floor[s] + share;
    if (qs > seg_len[s]) qs = seg_len[s];
    quota[s] = (int32_t)qs;
    total += qs;
    rem[s] = ((int64_t)q_floor[s] * (int64_t)M_total +
              T_rem * (int64_t)seg_mass[s]) -
             qs * (int64_t)M_total;
  }

  while (total < budget_eff) {
    int best = -1;
    for (int s = 0; s < n_seg; ++s) {
      if (quota[s] >= seg_len[s]) continue;
      if (best < 0 || rem[s] > rem[best]) best = s;
    }
    if (best < 0) break; /* cannot happen: sum L_i = n >= budget */
    quota[best] += 1;
    rem[best] -= (int64_t)M_total;
    total += 1;
  }
  while (total > budget_eff) {
    int best = -1;
    for (int s = n_seg - 1; s >= 0; --s) {
      if (quota[s] <= q_floor[s]) continue;
      if (best < 0 || rem[s] < rem[best]) best = s;
    }
    if (best < 0) break; /* cannot happen: sum q_floor <= budget */
    quota[best] -= 1;
    rem[best] += (int64_t)M_total;
    total -= 1;
  }
  free(q_floor);
  free(rem);
}

/* ------------------------------------------------------------------------ */
/* Step 5: segment-local top-k, must-keep, budget fix-up                      */
/* ------------------------------------------------------------------------ */

typedef struct {
  float score;
  int32_t v;
} cand_t;

/* best first: score descending, ties -> lower slot first */
static int cand_best_first(const void* x, const void* y) {
  const cand_t* a = (const cand_t*)x;
  const cand_t* b = (const cand_t*)y;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  return (a->v < b->v) ? -1 : (a->v > b->v) ? 1 : 0;
}

/* worst first: the exact reverse order */
static int cand_worst_first(const void* x, const void* y) {
  return -cand_best_first(x, y);
}

/*
 * [AMS] Key design 3: must-keep positions (4 sinks, the recent suffix) are
 * inserted first; if the budget left is negative the recent suffix is
 * shortened and the sinks are protected.  The worked example counts the
 * must-keep start and end inside the first and last segments' quotas.
 * [AMS] Key design 4: top quota positions inside each segment, union with the
 * must-keep set, de-duplication; over budget -> drop low-score non-must-keep
 * positions; under budget -> add the best unselected; sort the kept indices.
 * Readings:
 *  [R] n_s = min(n_sink, B), n_r = min(n_recent, B - n_s), B = min(T_keep, n);
 *  [R] must-keep slots count inside their own segment's quota; each segment
 *      picks max(0, q_i - |MK in segment|) of its non-must-keep slots;
 *  [R] order: score descending, ties -> lower slot; removal in the exact
 *      reverse order.  Under budget cannot occur: |MK| + sum picks >= sum q.
 */
int kvc_ref_select_unit(const float* score, int T, int pad,
                        const int32_t* seg_start, const int32_t* seg_len,
                        const int32_t* quota, int n_seg, int budget,
                        int n_sink, int n_recent, int32_t* kept) {
  const int n = T - pad;
  if (n <= 0) return 0;
  const int B = budget < n ? budget : n;
  const int n_s = n_sink < B ? n_sink : B;
  const int n_r = n_recent < (B - n_s) ? n_recent : (B - n_s);

  char* must = (char*)calloc((size_t)n, 1);
  char* chosen = (char*)calloc((size_t)n, 1);
  for (int v = 0; v < n_s; ++v) must[v] = 1;
  for (int v = n - n_r; v < n; ++v) must[v] = 1;
  int size = n_s + n_r;

  cand_t* picks = (cand_t*)malloc(sizeof(cand_t) * (size_t)n);
  int n_picks = 0;
  cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)n);
  for (int s = 0; s < n_seg; ++s) {
    int mk = 0, n_cand = 0;
    for (int v = seg_start[s]; v < seg_start[s] + seg_len[s]; ++v) {
      if (must[v]) {
        ++mk;
      } else {
        cand[n_cand].score = score[pad + v];
        cand[n_cand].v = v;
        ++n_cand;
      }
    }
    int want = quota[s] - mk;
    if (want < 0) want = 0;
    if (want > n_cand) want = n_cand;
    qsort(cand, (size_t)n_cand, sizeof(cand_t), cand_best_first);
    for (int r = 0; r < want; ++r) {
      picks[n_picks++] = cand[r];
      chosen[cand[r].v] = 1;
    }
    size += want;
  }

  if (size > B) {
    qsort(picks, (size_t)n_picks, sizeof(cand_t), cand_worst_first);
    for (int r = 0; r < size - B; ++r) chosen[picks[r].v] = 0;
    size = B;
  }

  int n_kept = 0;
  for (int v = 0; v < n; ++v)
    if (must[v] || chosen[v]) kept[n_kept++] = pad + v;

  free(must);
  free(chosen);
  free(picks);
  free(cand);
  return n_kept;
}

/* ------------------------------------------------------------------------ */
/* Second base score: key redundancy                                          */
/* ------------------------------------------------------------------------ */

/*
 * [SKV] token redundancy score, after R-KV: per KV head, a redundancy value
 * for every cached token computed from the key states alone, with the
 * attention mask keeping padding out; the final eviction score trades the
 * token importance against it with sigma (0.1) and tokens are evicted in
 * ascending order of that score.  Both formulas are printed as images the
 * text does not reproduce, so the plainest reading of the text is taken:
 *  [R] cos(a, b) = a.b / (|a| |b|), and 0 when either key is the zero vector;
 *  [R] r_i = mean over the other valid slots j != i of cos(k_i, k_j): the
 *      pairwise definition, O(n^2 d) per unit, written out as is;
 *  [R] r_i = 0 when fewer than two slots are valid (no other key).
 */
static double key_norm(const double* x, int d) {
  double ss = 0.0;
  for (int e = 0; e < d; ++e) ss += x[e] * x[e];
  return sqrt(ss);
}

void kvc_ref_mean_cosine_rows(const uint16_t* k, int T, int d, int pad, const int32_t* rows,
                              int n_rows, double* r_out) {
  const int n = T - pad;
  double* ki = (double*)malloc(sizeof(double) * (size_t)d);
  double* kj = (double*)malloc(sizeof(double) * (size_t)d);
  for (int q = 0; q < n_rows; ++q) {
    const int i = rows[q];
    if (n < 2) {
      r_out[q] = 0.0;
      continue;
    }
    for (int e = 0; e < d; ++e) ki[e] = bf16_to_double(k[(size_t)i * d + e]);
    const double ni = key_norm(ki, d);
    double sum = 0.0;
    for (int j = pad; j < T; ++j) {
      if (j == i) continue;
      for (int e = 0; e < d; ++e) kj[e] = bf16_to_double(k[(size_t)j * d + e]);
      const double nj = key_norm(kj, d);
      if (ni == 0.0 || nj == 0.0) continue; /* cosine 0 */
      double dot = 0.0;
      for (int e = 0; e < d; ++e) dot += ki[e] * kj[e];
      sum += dot / (ni * nj);
    }
    r_out[q] = sum / (double)(n - 1);
  }
  free(ki);
  free(kj);
}

/*
 * [SKV] final eviction score without the sentence term (sentence similarity
 * needs text segmentation and hidden states, outside this path):
 *  [R] R = softmax of r over the valid slots (the redundancy is normalised
 *      like the importance, so the two are on one scale);
 *  [R] I_i = s_i / sum over valid v of s_v, s = the max-pooled attention
 *      usage: the importance normalised over the observation window; I = 0
 *      when that sum is 0;
 *  [R] f_i = sigma * I_i - (1 - sigma) * R_i: the more redundant a token,
 *      the earlier it is evicted.
 * f replaces the score in the segment-local selection only; segments and
 * quotas stay on the attention mass ([AMS] Method: the mass and the score
 * are separate inputs, and any base scorer can supply the score).
 */
void kvc_ref_redundancy_score(const uint16_t* k, const float* score, int T, int d, int pad,
                              double sigma, double* r_out, double* R_out, double* f_out) {
  const int n = T - pad;
  double* r = (double*)calloc((size_t)(T > 0 ? T : 1), sizeof(double));
  int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  for (int i = 0; i < n; ++i) rows[i] = pad + i;
  if (n > 0) kvc_ref_mean_cosine_rows(k, T, d, pad, rows, n, r + pad);
  double z = 0.0, s_sum = 0.0;
  for (int i = pad; i < T; ++i) {
    z += exp(r[i]);
    s_sum += (double)score[i];
  }
  for (int i = 0; i < T; ++i) {
    if (i < pad) {
      if (r_out) r_out[i] = 0.0;
      if (R_out) R_out[i] = 0.0;
      if (f_out) f_out[i] = -INFINITY;
      continue;
    }
    const double Ri = exp(r[i]) / z;
    const double Ii = s_sum > 0.0 ? (double)score[i] / s_sum : 0.0;
    if (r_out) r_out[i] = r[i];
    if (R_out) R_out[i] = Ri;
    if (f_out) f_out[i] = sigma * Ii - (1.0 - sigma) * Ri;
  }
  free(r);
  free(rows);
}

/* ------------------------------------------------------------------------ */
/* batched mirrors                                                            */
/* ------------------------------------------------------------------------ */

int kvc_ref_mass(const kvc_ref_config* cfg, int U, int T, const uint16_t* q,
                 const uint16_t* k, const float* credit_in,
                 const int32_t* pad, const int32_t* n_carry, float* mass,
                 float* score, float* credit_post) {
  const int G = cfg->group, W = cfg->window, d = cfg->head_dim;
  const double scale = config_scale(cfg);
  double* qd = (double*)malloc(sizeof(double) * (size_t)G * W * d);
  double* kd = (double*)malloc(sizeof(double) * (size_t)T * d);
  double* a = (double*)malloc(sizeof(double) * (size_t)T);
  double* s = (double*)malloc(sizeof(double) * (size_t)T);
  double* u = (double*)malloc(sizeof(double) * (size_t)T);
  double* m = (double*)malloc(sizeof(double) * (size_t)T);
  double* c_in = (double*)malloc(sizeof(double) * (size_t)T);
  double* c = (double*)malloc(sizeof(double) * (size_t)T);
  double* mu = (double*)malloc(sizeof(double) * (size_t)T);

  for (int unit = 0; unit < U; ++unit) {
    const int p = pad[unit];
    const uint16_t* qu = q + (size_t)unit * G * W * d;
    const uint16_t* ku = k + (size_t)unit * T * d;
    for (size_t e = 0; e < (size_t)G * W * d; ++e) qd[e] = bf16_to_double(qu[e]);
    for (size_t e = 0; e < (size_t)T * d; ++e) kd[e] = bf16_to_double(ku[e]);
    for (int i = 0; i < T; ++i) c_in[i] = (double)credit_in[(size_t)unit * T + i];

    float* mass_u = mass + (size_t)unit * T;
    float* score_u = score + (size_t)unit * T;
    float* cp_u = credit_post + (size_t)unit * T;
    if (T - p <= 0) {
      for (int i = 0; i < T; ++i) {
        mass_u[i] = 0.0f;
        score_u[i] = -INFINITY;
        cp_u[i] = 0.0f;
      }
      continue;
    }
    kvc_ref_usage(qd, kd, G, W, d, T, p, scale, a, NULL);
    kvc_ref_maxpool(a, T, p, cfg->max_pool, s);
    kvc_ref_avgpool(a, T, p, cfg->avg_pool, u);
    kvc_ref_mass_normalize(u, T, p, (double)cfg->eps, m);
    kvc_ref_credit(m, c_in, T, p, n_carry[unit], (double)cfg->lambda,
                   (double)cfg->beta, c, mu);
    for (int i = 0; i < T; ++i) {
      mass_u[i] = (float)mu[i];
      score_u[i] = (float)s[i];
      cp_u[i] = (float)c[i];
    }
  }
  free(qd);
  free(kd);
  free(a);
  free(s);
  free(u);
  free(m);
  free(c_in);
  free(c);
  free(mu);
  return 0;
}

int kvc_ref_segment_quota(const kvc_ref_config* cfg, int U, int T,
                          const float* mass, const int32_t* pad,
                          int32_t* seg_start, int32_t* seg_len,
                          int32_t* quota, int32_t* n_seg) {
  const int S_max = kvc_ref_s_max(cfg, T);
  uint64_t* M = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)S_max);
  for (int unit = 0; unit < U; ++unit) {
    const int p = pad[unit];
    int32_t* st = seg_start + (size_t)unit * S_max;
    int32_t* ln = seg_len + (size_t)unit * S_max;
    int32_t* qu = quota + (size_t)unit * S_max;
    for (int s = 0; s < S_max; ++s) {
      st[s] = 0;
      ln[s] = 0;
      qu[s] = 0;
    }
    const int ns = (cfg->global_topk || cfg->seg_fixed > 0)
                       ? kvc_ref_segments_ablation(mass + (size_t)unit * T, T, p,
                                                   cfg->seg_fixed, cfg->global_topk, st,
                                                   ln, M)
                       : kvc_ref_segments(mass + (size_t)unit * T, T, p, cfg->delta,
                                          cfg->seg_min, cfg->seg_max, st, ln, M);
    if (cfg->quota_by_len)
      for (int s = 0; s < ns; ++s) M[s] = (uint64_t)ln[s];
    const int n = T - p;
    const int budget_eff = cfg->budget < n ? cfg->budget : n;
    kvc_ref_quotas(ln, M, ns, budget_eff, cfg->q_min, qu);
    for (int s = 0; s < ns; ++s) st[s] += p; /* absolute slots */
    n_seg[unit] = ns;
  }
  free(M);
  return 0;
}

int kvc_ref_select(const kvc_ref_config* cfg, int U, int T, const float* score,
                   const int32_t* pad, const int32_t* seg_start,
                   const int32_t* seg_len, const int32_t* quota,
                   const int32_t* n_seg, int32_t* kept_idx, int32_t* n_kept) {
  const int S_max = kvc_ref_s_max(cfg, T);
  int32_t* st = (int32_t*)malloc(sizeof(int32_t) * (size_t)S_max);
  for (int unit = 0; unit < U; ++unit) {
    const int p = pad[unit];
    const int ns = n_seg[unit];
    for (int s = 0; s < ns; ++s) st[s] = seg_start[(size_t)unit * S_max + s] - p;
    int32_t* out = kept_idx + (size_t)unit * cfg->budget;
    const int nk = kvc_ref_select_unit(
        score + (size_t)unit * T, T, p, st, seg_len + (size_t)unit * S_max,
        quota + (size_t)unit * S_max, ns, cfg->budget, cfg->n_sink,
        cfg->n_recent, out);
    for (int r = nk; r < cfg->budget; ++r) out[r] = -1;
    n_kept[unit] = nk;
  }
  free(st);
  return 0;
}

/*
 * [AMS] Key design 4: the kept indices are sorted and the same indices
 * gather K and V into a fixed-length per-head cache -- a real copy, not a
 * mask.  The credit is gathered with the same indices (alignment rule of Key
 * design 1).  Rows past n_kept are zero.
 */
int kvc_ref_compact(const kvc_ref_config* cfg, int U, int T, const uint16_t* k,
                    const uint16_t* v, const float* credit_post,
                    const int32_t* kept_idx, const int32_t* n_kept,
                    uint16_t* k_out, uint16_t* v_out, float* credit_out) {
  const int d = cfg->head_dim, Bk = cfg->budget;
  for (int unit = 0; unit < U; ++unit) {
    for (int r = 0; r < Bk; ++r) {
      uint16_t* ko = k_out + ((size_t)unit * Bk + r) * d;
      uint16_t* vo = v_out + ((size_t)unit * Bk + r) * d;
      float* co = credit_out + (size_t)unit * Bk + r;
      if (r < n_kept[unit]) {
        const int32_t slot = kept_idx[(size_t)unit * Bk + r];
        const uint16_t* ki = k + ((size_t)unit * T + slot) * d;
        const uint16_t* vi = v + ((size_t)unit * T + slot) * d;
        for (int e = 0; e < d; ++e) {
          ko[e] = ki[e];
          vo[e] = vi[e];
        }
        *co = credit_post[(size_t)unit * T + slot];
      } else {
        for (int e = 0; e < d; ++e) {
          ko[e] = 0;
          vo[e] = 0;
        }
        *co = 0.0f;
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Query-similarity refresh trigger                                           */
/* ------------------------------------------------------------------------ */

/*
 * [RefreshKV] "Deciding when to decode with full cache" / "Dynamic scheduling":
 * every S-th decode step, for each layer, the cosine similarity between the
 * query of the current token averaged over all query heads and the averaged
 * query of the layer's most recent full-attention step decides: above the
 * threshold s the partial cache is used, otherwise the layer takes a full
 * step (and that step's averaged query becomes the new reference).
 * Readings:
 *  [R] one decision per (layer, sequence of the batch);
 *  [R] a zero reference (no full step yet) or a zero current query (cosine
 *      undefined) decides a refresh; sim = -2 marks the undefined cosine;
 *  [R] "below the threshold" is strict: sim < s refreshes.
 */
void kvc_ref_refresh_decision(int LB, int Hq, int d, const uint16_t* q, double* q_ref,
                              double threshold, int32_t* flag, double* sim) {
  double* mean = (double*)malloc(sizeof(double) * (size_t)d);
  for (int r = 0; r < LB; ++r) {
    for (int i = 0; i < d; ++i) mean[i] = 0.0;
    for (int h = 0; h < Hq; ++h)
      for (int i = 0; i < d; ++i)
        mean[i] += bf16_to_double(q[((size_t)r * Hq + h) * d + i]);
    for (int i = 0; i < d; ++i) mean[i] /= (double)Hq;
    double dot = 0.0, nq = 0.0, nr = 0.0;
    double* ref = q_ref + (size_t)r * d;
    for (int i = 0; i < d; ++i) {
      dot += mean[i] * ref[i];
      nq += mean[i] * mean[i];
      nr += ref[i] * ref[i];
    }
    const int defined = nq > 0.0 && nr > 0.0;
    const double c = defined ? dot / (sqrt(nq) * sqrt(nr)) : -2.0;
    sim[r] = c;
    flag[r] = (!defined || c < threshold) ? 1 : 0;
    if (flag[r])
      for (int i = 0; i < d; ++i) ref[i] = mean[i];
  }
  free(mean);
}

/* ------------------------------------------------------------------------ */
/* Paged compaction                                                           */
/* ------------------------------------------------------------------------ */

/*
 * [AMS] Appendix E: the selection is separated from the paged storage layout.
 * The method outputs the kept indices per head; the runtime allocates new
 * blocks, copies each head's KV from its original positions into the new
 * physical slots, replaces the request's block table and frees the old
 * blocks.  The same compacted slot may hold different original positions in
 * different heads.
 * Readings (the page gives the steps, not the data structures):
 *  [R] pools [L][n_blocks][H][bs][d]; one block table per sequence, shared by
 *      all layers (every layer and head of a sequence keeps the same count);
 *  [R] the free blocks form a stack; allocation for all sequences happens
 *      before any copy (old and new blocks coexist during the copy), in
 *      sequence order from the top of the stack; the old blocks are pushed
 *      back afterwards, in sequence order;
 *  [R] kept slot j of head h goes to block table_new[b][j / bs], row j % bs.
 */
int kvc_ref_compact_paged(int L, int B, int H, int d, int bs, int n_blocks, int max_blocks,
                          int budget, uint16_t* k_pool, uint16_t* v_pool,
                          const int32_t* seq_len, const int32_t* pad,
                          const int32_t* kept_idx, const int32_t* n_kept,
                          const int32_t* table_old, int32_t* table_new,
                          int32_t* free_list, int32_t* free_top) {
  /* blocks needed after compaction, per sequence (same count in every head) */
  int64_t need_total = 0;
  for (int b = 0; b < B; ++b) {
    const int nk = n_kept[(size_t)b * H];  /* layer 0, head 0 */
    if (nk < 0 || nk > budget || (nk + bs - 1) / bs > max_blocks) return -1;
    for (int l = 0; l < L; ++l)
      for (int h = 0; h < H; ++h)
        if (n_kept[((size_t)l * B + b) * H + h] != nk) return -1;
    need_total += (nk + bs - 1) / bs;
  }
  if (need_total > *free_top) return -1;
  /* check every source position before changing anything */
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h) {
        const size_t u = ((size_t)l * B + b) * H + h;
        for (int j = 0; j < n_kept[u]; ++j) {
          const int t = kept_idx[u * budget + j] - pad[b];
          if (t < 0 || t >= seq_len[b]) return -1;
          const int blk = table_old[(size_t)b * max_blocks + t / bs];
          if (blk < 0 || blk >= n_blocks) return -1;
        }
      }
  /* allocate: sequence b takes the next blocks from the top of the stack */
  int64_t pos = *free_top - need_total;
  for (int b = 0; b < B; ++b) {
    const int nk = n_kept[(size_t)b * H];
    const int nb = (nk + bs - 1) / bs;
    for (int i = 0; i < max_blocks; ++i)
      table_new[(size_t)b * max_blocks + i] = i < nb ? free_list[pos + i] : -1;
    pos += nb;
  }
  *free_top -= (int32_t)need_total;
  /* copy each head's kept rows into the new blocks */
  const size_t row = (size_t)d;
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h) {
        const size_t u = ((size_t)l * B + b) * H + h;
        for (int j = 0; j < n_kept[u]; ++j) {
          const int t = kept_idx[u * budget + j] - pad[b];
          const int src_blk = table_old[(size_t)b * max_blocks + t / bs];
          const int dst_blk = table_new[(size_t)b * max_blocks + j / bs];
          const size_t src = ((((size_t)l * n_blocks + src_blk) * H + h) * bs + t % bs) * row;
          const size_t dst = ((((size_t)l * n_blocks + dst_blk) * H + h) * bs + j % bs) * row;
          for (int i = 0; i < d; ++i) {
            k_pool[dst + i] = k_pool[src + i];
            v_pool[dst + i] = v_pool[src + i];
          }
        }
      }
  /* free the old blocks, in sequence order */
  for (int b = 0; b < B; ++b) {
    const int nb_old = (seq_len[b] + bs - 1) / bs;
    for (int i = 0; i < nb_old; ++i) free_list[(*free_top)++] = table_old[(size_t)b * max_blocks + i];
  }
  return 0;
}
