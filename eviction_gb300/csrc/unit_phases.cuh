// unit_phases.cuh -- the three per-unit steps after the attention usage, as
// CTA-wide device functions: mass (pool, normalise, credit EMA, mix), the
// cumulative-mass segmentation with its quotas, and the segment-local top-k.
//
// "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Method,
// Key designs 1-4 (each function names its own passage).  One CTA handles one
// unit (a layer's KV head of one sequence).  The stand-alone kernels
// (mass_post.cu, segment_quota.cu, select.cu) and the fused per-unit kernel
// (unit_post.cu) all run these functions, so that a step computes the same
// bits whichever kernel runs it: the fused kernel only moves the mass, the
// score and the segments from global to shared memory between the steps.
#pragma once

#include <climits>
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace unit {

// ---------------------------------------------------------------- reductions

// Three block sums in one pass: per-warp butterfly sums, then the warps' sums
// in a fixed order (repeated runs give identical bits).  red holds
// 3 * (NT/32 + 1) floats.
template <int NT>
__device__ __forceinline__ float3 block_sum3(float3 v, float* red) {
  constexpr int W = NT / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) {
    red[warp] = v.x;
    red[W + 1 + warp] = v.y;
    red[2 * (W + 1) + warp] = v.z;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    float3 t = make_float3(0.f, 0.f, 0.f);
    if (lane < W) t = make_float3(red[lane], red[W + 1 + lane], red[2 * (W + 1) + lane]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      t.x += __shfl_xor_sync(0xffffffffu, t.x, o);
      t.y += __shfl_xor_sync(0xffffffffu, t.y, o);
      t.z += __shfl_xor_sync(0xffffffffu, t.z, o);
    }
    if (lane == 0) {
      red[W] = t.x;
      red[2 * W + 1] = t.y;
      red[3 * W + 2] = t.z;
    }
  }
  __syncthreads();
  return make_float3(red[W], red[2 * W + 1], red[3 * W + 2]);
}

template <int NT>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = (lane < NT / 32) ? red[lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (lane == 0) red[NT / 32] = t;
  }
  __syncthreads();
  return red[NT / 32];
}

template <int NT>
__device__ __forceinline__ int block_count(int v, int* red) {
  constexpr int kWarps = NT / 32;
  v = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(v)));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += red[w];
  return t;
}

// ---------------------------------------------------------------- step 2: mass

struct PostParams {
  int T, R, W, G, B, H;
  int avg_pool, max_pool;
  float eps, lambda, beta;
  int Rp;
  const float* pmax;  // [U][Rp] largest probability of each row (0 if absent)
  float* usage;       // [U][T] raw usage, filled in place
  const int32_t* pad;
  const int32_t* n_carry;
  const float* credit_in;
  float* credit_post;
  float* mass;
  float* score;
};

// The CTA shape of the mass step for units of up to kSmemT slots: threads and
// slots per thread.  The step's fp32 sums follow this shape, so the
// stand-alone mass kernel and the fused per-unit kernel take it from here.
// 128-thread CTAs up to 2048 slots: each unit is a chain of short dependent
// steps, and 16 such CTAs share an SM (0.122 -> 0.118 ms on the 28-layer
// batch-32 event, 0.451 -> 0.414 ms on the ragged batch, against 8 CTAs of 256
// threads).
constexpr int kSmemT = 4096;
__host__ __device__ inline void mass_shape(int T, int* nt, int* ept) {
  *nt = T <= 2048 ? 128 : 256;
  const int e = (T + *nt - 1) / *nt;
  *ept = e <= 4 ? 4 : e <= 6 ? 6 : e <= 8 ? 8 : e <= 12 ? 12 : 16;
}

// Key design 1 (and RefreshKV A2/A6 for the score), for a unit of at most
// kEpt * NT slots:
//   * entries a window query cannot see (causal suffix) are filled with the
//     window's maximum score, the largest softmax probability of the unit
//     (max_r 1/Z'_r, from pass 1 of the attention kernel);
//   * u = average pool (zero outside the valid slots, divided by the kernel
//     size);  m_i = (max(u_i,0)+eps) / sum_v (max(u_v,0)+eps);
//   * c = lambda*c_in + (1-lambda)*m with c_in := m on slots new since the last
//     event;  m_used = normalize(beta*m + (1-beta)*normalize(c));
//   * score = the filled usage max-pooled over valid neighbours.
// Thread t owns slots t + k*NT (coalesced global reads and writes).  The
// unit's filled usage sits in `a` (shared, kEpt * NT floats) and the pooling
// windows read it there: with the default pools (average over 5, max over 7)
// an interior slot's window is seven unrolled loads, other slots loop over
// their valid neighbours; either way in ascending slot order, the same sums.
// Each thread keeps its slots' values in registers; every sum is a per-thread
// pass over its slots in order, then one fixed-order block reduction, so
// repeated runs give identical bits.  Score, mass and credit go
// to global memory, and also to mass_sm / score_sm (shared, indexed by slot)
// when given; mass_sm may be `a` itself (it is written after a's last read).
template <int kEpt, int NT>
__device__ __forceinline__ void mass_phase(const PostParams& p, int u, float* a, float* red,
                                           float* mass_sm, float* score_sm) {
  const int b = (u / p.H) % p.B;
  const int T = p.T;
  const int pad = min(max(p.pad[b], 0), T);
  const size_t base = static_cast<size_t>(u) * T;
  float* mass = p.mass + base;
  float* score = p.score + base;
  float* cpost = p.credit_post + base;
  const float* cin = p.credit_in + base;
  const float* usage = p.usage + base;

  if (pad >= T) {
    for (int i = threadIdx.x; i < T; i += NT) {
      mass[i] = 0.f;
      score[i] = -INFINITY;
      cpost[i] = 0.f;
      if (mass_sm) mass_sm[i] = 0.f;
      if (score_sm) score_sm[i] = -INFINITY;
    }
    return;
  }
  const int n_carry = min(max(p.n_carry[b], 0), T - pad);
  const int tid = static_cast<int>(threadIdx.x);

  // this thread's raw usage, loaded together with the row statistics
  float use[kEpt];
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = tid + k * NT;
    use[k] = (i >= pad && i < T) ? usage[i] : 0.f;
  }
  float pm = 0.f;
  for (int r = tid; r < p.R; r += NT) pm = fmaxf(pm, p.pmax[static_cast<size_t>(u) * p.Rp + r]);
  const float fill = block_max<NT>(pm, red);

  const int j_lo = max(0, pad - (T - p.W));
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = tid + k * NT;
    if (i < T) {
      const int unseen = max(0, min(p.W, i - T + p.W) - j_lo) * p.G;
      a[i] = i >= pad ? use[k] + fill * static_cast<float>(unseen) : 0.f;
    }
  }
  __syncthreads();

  const int ra = p.avg_pool / 2, rm = p.max_pool / 2;
  const bool pools75 = ra == 2 && rm == 3;
  const float inv_k = 1.0f / static_cast<float>(p.avg_pool);
  float up[kEpt];  // max(avg pool, 0) + eps
  float tot = 0.f;
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = tid + k * NT;
    up[k] = 0.f;
    if (i >= T) continue;
    if (i < pad) {
      score[i] = -INFINITY;
      if (score_sm) score_sm[i] = -INFINITY;
      continue;
    }
    float mx, sm;
    if (pools75 && i - 3 >= pad && i + 3 < T) {
      const float w0 = a[i - 3], w1 = a[i - 2], w2 = a[i - 1], w3 = a[i], w4 = a[i + 1],
                  w5 = a[i + 2], w6 = a[i + 3];
      mx = fmaxf(fmaxf(fmaxf(w0, w1), fmaxf(w2, w3)), fmaxf(fmaxf(w4, w5), w6));
      sm = (((w1 + w2) + w3) + w4) + w5;
    } else {
      mx = -INFINITY;
      sm = 0.f;
      for (int t = max(pad, i - rm); t <= min(T - 1, i + rm); ++t) mx = fmaxf(mx, a[t]);
      for (int t = max(pad, i - ra); t <= min(T - 1, i + ra); ++t) sm += a[t];
    }
    score[i] = mx;
    if (score_sm) score_sm[i] = mx;
    up[k] = fmaxf(sm * inv_k, 0.f) + p.eps;
    tot += up[k];
  }
  // One reduction gives the three totals the rest needs.  With
  // m_i = up_i / U (U = sum up), sum_i m_i = 1, so the credit total is
  //   sum_i c_i = 1 + lambda * (sum_carried c_in - sum_carried m)
  // (c_i = m_i on slots new since the last event), and
  //   beta*m + (1-beta)*c/sum(c) already sums to 1: the final normalisation
  // of m_used divides by one, and is left out.
  float cin_c = 0.f, up_c = 0.f;  // carried slots: credit-in, up
  float cprior[kEpt];
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = tid + k * NT;
    const bool carried = i >= pad && i < pad + n_carry;
    cprior[k] = carried ? cin[i] : 0.f;
    cin_c += cprior[k];
    up_c += carried ? up[k] : 0.f;
  }
  const float3 tt = block_sum3<NT>(make_float3(tot, cin_c, up_c), red);
  const float total1 = tt.x;
  const float lam = p.lambda, beta = p.beta;
  const float c_total = 1.0f + lam * (tt.y - tt.z / total1);
  // the two normalisations as products with reciprocals taken once per unit
  // (an IEEE division per slot costs about ten instructions; the product is
  // within an ulp of the quotient)
  const float inv_total = 1.0f / total1;
  const float inv_ct = c_total > 0.f ? 1.0f / c_total : 0.f;
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = tid + k * NT;
    if (i >= T) continue;
    float mu = 0.f, c = 0.f;
    if (i >= pad) {
      const float m = up[k] * inv_total;
      c = (i < pad + n_carry) ? lam * cprior[k] + (1.0f - lam) * m : m;
      const float cn = (c_total > 0.f) ? c * inv_ct : m;
      mu = beta * m + (1.0f - beta) * cn;
    }
    mass[i] = mu;
    cpost[i] = c;
    if (mass_sm) mass_sm[i] = mu;
  }
}

// ---------------------------------------------------------------- step 3: segments, quotas

constexpr int kMaxK = 1024;     // thresholds: delta >= 1/1024

struct SegParams {
  int T, B, H, S_max, S_cap;
  int budget, q_min, seg_min, seg_max;
  int seg_fixed, quota_by_len, global_topk;  // ablation switches (0 = the method)
  uint64_t delta_m;  // Delta = delta_m * 2^delta_e, delta_m odd (the fp32 Delta's significand)
  int delta_e;
  int K;  // number of thresholds
  const float* mass;
  const int32_t* pad;
  int32_t* seg_start;
  int32_t* seg_len;
  int32_t* quota;
  int32_t* n_seg;
};

// Shared memory of the segmentation.  mass, rem, start, len, q and floor hold
// S_cap entries; b K entries; part NT/32; pre NT; sub NT*kSub when
// segment_phase runs with kSub > 1 (else unused).  After segment_phase returns,
// start (valid offsets), len and q hold the unit's segments and *nseg their
// number; mass, rem, floor, b and part are free again.
struct SegSmem {
  uint64_t* mass;
  int64_t* rem;
  int32_t* start;
  int32_t* len;
  int32_t* q;
  int32_t* floor;
  int32_t* b;
  uint64_t* part;
  uint64_t* pre;  // [NT] fixed-point mass before each thread's range
  uint64_t* sub;  // [NT][kSub] the same before each of its kSub sub-ranges
  uint64_t* total;
  int* nseg;
};

__device__ __forceinline__ uint64_t fixed_mass(float m) {
  // m * 2^40 is exact in fp32 (an exponent shift); truncation toward zero.
  const float scaled = m * 1099511627776.0f;
  return scaled > 0.f ? __float2ull_rz(scaled) : 0ull;
}

// x rounded to 53 significant bits (IEEE round to nearest, ties to even) as
// q * 2^r, q <= 2^53; x < 2^88 given as hi:lo, so r <= 35.
__device__ __forceinline__ uint64_t round53(uint64_t lo, uint64_t hi, int* r_out) {
  const int nb = hi ? 128 - __clzll(hi) : 64 - __clzll(lo);
  if (nb <= 53) {
    *r_out = 0;
    return lo;
  }
  const int r = nb - 53;
  uint64_t q = (lo >> r) | (hi << (64 - r));
  const bool g = (lo >> (r - 1)) & 1ull;                               // the first bit dropped
  const bool sticky = r > 1 && (lo & ((1ull << (r - 1)) - 1ull)) != 0ull;  // any bit below it
  if (g && (sticky || (q & 1ull))) ++q;
  *r_out = r;
  return q;
}

// ceil(fl(fl(A * 2^eA) * fl(S))) in IEEE double for A < 2^35 and
// A * 2^eA < 1: fl(A * 2^eA) is exact, fl(S) is S rounded to 53 significant
// bits, and the product of the two significands (below 2^88) is rounded to 53
// bits once; the ceiling of the result.  Integers only, and bit for bit the
// double computation (double arithmetic is a slow path on this GPU).
__device__ __forceinline__ uint64_t ceil_scaled_product(uint64_t A, int eA, uint64_t S) {
  if (A == 0ull || S == 0ull) return 0ull;
  int ts, r;
  const uint64_t qs = round53(S, 0ull, &ts);
  const uint64_t q = round53(A * qs, __umul64hi(A, qs), &r);
  const int t = eA + ts + r;  // the rounded product is q * 2^t
  if (t >= 0) return q << t;  // (below S: A * 2^eA < 1)
  const int s = -t;
  if (s >= 64) return 1ull;
  return (q >> s) + ((q & ((1ull << s) - 1ull)) ? 1ull : 0ull);
}

__device__ __forceinline__ uint64_t warp_incl_scan(uint64_t v) {
  const int lane = threadIdx.x % 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// x as an fp32 estimate (relative error below 2^-22) from two 32-bit
// conversions: 64-bit conversions are far slower on this GPU.
__device__ __forceinline__ float u64_to_f32_est(uint64_t x) {
  return __fmaf_rn(__uint2float_rn(static_cast<uint32_t>(x >> 32)), 4294967296.0f,
                   __uint2float_rn(static_cast<uint32_t>(x)));
}

// floor(num / den) for 0 <= num, 0 < den, with num / den < 2^24: an fp32
// estimate (off by a few units at most) corrected by exact integer
// multiplication (products below 2^63).
__device__ __forceinline__ uint64_t udiv_small(uint64_t num, uint64_t den) {
  uint64_t q = __float2uint_rz(
      fminf(16777216.f, fmaxf(0.f, __fdividef(u64_to_f32_est(num), u64_to_f32_est(den)))));
  while (q > 0 && q * den > num) --q;
  while ((q + 1) * den <= num) ++q;
  return q;
}

// floor(num / den) for 0 < den, |num / den| < 2^24, likewise.
__device__ __forceinline__ int64_t sdiv_floor_small(int64_t num, int64_t den) {
  const uint64_t a = num < 0 ? static_cast<uint64_t>(-num) : static_cast<uint64_t>(num);
  const float e = fminf(16777216.f, __fdividef(u64_to_f32_est(a),
                                               u64_to_f32_est(static_cast<uint64_t>(den))));
  const int64_t m = static_cast<int64_t>(__float2uint_rz(e));
  int64_t q = num < 0 ? -m : m;
  while (q * den > num) --q;
  while ((q + 1) * den <= num) ++q;
  return q;
}

// The correction steps of the quota rule, in bulk.  Each step gives (or takes)
// one unit to the segment with the best current remainder, and a segment's
// remainder moves by the mass total M per unit, so the steps taken are exactly
// the D best "bids" b_s(k) = b0_s - k*M over k < cap_s, ordered by value and
// then by segment index:
//   short (negate = false): b0_s = rem_s,  cap_s = len_s - q_s;   q_s += taken
//   over  (negate = true):  b0_s = -rem_s, cap_s = q_s - floor_s; q_s -= taken
// Levels: with h = floor(M/2), the bids of level l lie in [l*M - h, l*M - h + M),
// so every bid of level l beats every bid of level l-1.  Segment s has the
// levels j_s - k, k < cap_s, with j_s = floor((b0_s + h) / M) its first bid's.
// The D best bids are all bids above the level L at which the count from the
// top reaches D (a binary search on small integers), plus the D' best bids of
// level L in (value, index) order.  A segment's bid at level L is
// (L*M - h) + w_s with w_s = (b0_s + h) - j_s*M in [0, M), the remainder of
// its level division, so level L's bids order as their w: a bitwise search
// finds the D'-th largest w among the segments with a bid there, and the ties
// at it go in index order.  One small division per segment; counts are 32-bit
// (they are at most the unit's slot count).  `scratch` holds 2*ns int32: the
// segments' first levels, then the units taken; `rem` is overwritten with w.
__device__ __forceinline__ void take_best_bids(int64_t* rem, const int32_t* ref, int32_t* q,
                                               int ns, int64_t M, int D, bool negate,
                                               bool low_first, int lane, int32_t* scratch) {
  int32_t* lev = scratch;
  int32_t* take = scratch + ns;
  auto b0_of = [&](int s) { return negate ? -rem[s] : rem[s]; };
  auto cap_of = [&](int s) { return negate ? q[s] - ref[s] : ref[s] - q[s]; };
  if (M <= 0) {
    // all remainders equal and unchanging: the segments fill in index order
    // (lower first when short, higher first when over)
    int before = 0;
    const int n_chunks = (ns + 31) / 32;
    for (int cc = 0; cc < n_chunks; ++cc) {
      const int chunk = low_first ? cc : n_chunks - 1 - cc;
      const int s = chunk * 32 + lane;
      const int cap = s < ns ? max(cap_of(s), 0) : 0;
      int incl = cap;  // inclusive scan in fill order
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = low_first ? __shfl_up_sync(0xffffffffu, incl, o)
                                : __shfl_down_sync(0xffffffffu, incl, o);
        if (low_first ? lane >= o : lane + o < 32) incl += t;
      }
      if (s < ns) take[s] = min(cap, max(0, D - (before + incl - cap)));
      before += __shfl_sync(0xffffffffu, incl, low_first ? 31 : 0);
    }
  } else {
    const int64_t h = M >> 1;
    int lo = INT_MAX, hi = INT_MIN;
    for (int s = lane; s < ns; s += 32) {
      const int cap = cap_of(s);
      int j = 0;
      int64_t w = 0;
      if (cap > 0) {
        const int64_t num = b0_of(s) + h;
        j = static_cast<int>(sdiv_floor_small(num, M));
        w = num - static_cast<int64_t>(j) * M;
        lo = min(lo, j - cap + 1);
        hi = max(hi, j);
      }
      lev[s] = j;
      rem[s] = w;  // b0 is not needed again
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lo > hi) lo = hi = 0;  // no capacity anywhere (cannot happen: sum L_i >= budget)
    __syncwarp();
    auto count_ge = [&](int l) {  // bids of level >= l
      int c = 0;
      for (int s = lane; s < ns; s += 32) {
        const int cap = cap_of(s);
        if (cap > 0) c += max(0, min(cap, lev[s] - l + 1));
      }
      return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
    };
    // L = the largest level with count_ge(L) >= D (count_ge(lo) is every bid)
    int L = lo, L_hi = hi;
    while (L < L_hi) {
      const int mid = L + (L_hi - L + 1) / 2;
      if (count_ge(mid) >= D) L = mid; else L_hi = mid - 1;
    }
    const int d_at_L = D - count_ge(L + 1);  // bids taken at level L
    auto at_L = [&](int s) {  // segment s has a bid at level L
      const int cap = cap_of(s);
      return cap > 0 && lev[s] - cap < L && L <= lev[s];
    };
    for (int s = lane; s < ns; s += 32) {
      const int cap = cap_of(s);
      take[s] = cap > 0 ? max(0, min(cap, lev[s] - L)) : 0;  // bids above level L
    }
    if (d_at_L > 0) {  // warp-uniform
      // x = the d_at_L-th largest w at level L: the largest x with
      // #(w >= x) >= d_at_L
      uint64_t x = 0;
      for (int bit = 63 - __clzll(static_cast<uint64_t>(M)); bit >= 0; --bit) {  // w < M
        const uint64_t t = x | (1ull << bit);
        int c = 0;
        for (int s = lane; s < ns; s += 32)
          c += (at_L(s) && static_cast<uint64_t>(rem[s]) >= t) ? 1 : 0;
        if (static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c))) >= d_at_L)
          x = t;
      }
      int gt = 0;
      for (int s = lane; s < ns; s += 32)
        gt += (at_L(s) && static_cast<uint64_t>(rem[s]) > x) ? 1 : 0;
      int ties_left = d_at_L - static_cast<int>(__reduce_add_sync(0xffffffffu,
                                                                   static_cast<unsigned>(gt)));
      // every bid above x, then the ties at x in index order (lower first when
      // short, higher first when over), 32 segments at a time
      const int n_chunks = (ns + 31) / 32;
      const uint32_t ahead = low_first ? ((1u << lane) - 1u)
                                       : (lane == 31 ? 0u : (0xffffffffu << (lane + 1)));
      for (int cc = 0; cc < n_chunks; ++cc) {
        const int s = (low_first ? cc : n_chunks - 1 - cc) * 32 + lane;
        const bool in = s < ns && at_L(s);
        const uint64_t w = in ? static_cast<uint64_t>(rem[s]) : 0ull;
        const bool tie = in && w == x;
        const uint32_t ball = __ballot_sync(0xffffffffu, tie);
        if ((in && w > x) || (tie && static_cast<int>(__popc(ball & ahead)) < ties_left))
          take[s] += 1;
        ties_left -= __popc(ball);
      }
    }
  }
  __syncwarp();
  for (int s = lane; s < ns; s += 32) q[s] = negate ? q[s] - take[s] : q[s] + take[s];
  __syncwarp();
}

__device__ __forceinline__ int64_t shfl64_down(int64_t v) {  // lane + 1's value (lane 31: its own)
  const int lo = __shfl_down_sync(0xffffffffu, static_cast<int>(v & 0xffffffff), 1);
  const int hi = __shfl_down_sync(0xffffffffu, static_cast<int>(v >> 32), 1);
  return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

__device__ __forceinline__ int64_t shfl64(int64_t v, int src) {
  const int lo = __shfl_sync(0xffffffffu, static_cast<int>(v & 0xffffffff), src);
  const int hi = __shfl_sync(0xffffffffu, static_cast<int>(v >> 32), src);
  return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

// take_best_bids for at most 32 segments, one per lane, in registers: this
// lane's first bid b0 and capacity cap (<= 0 or an idle lane: no bids); returns
// the units this lane's segment takes.  Same levels and order as above.
__device__ __forceinline__ int best_bids_lane(int64_t b0, int cap, int64_t M, int D,
                                              bool low_first, int lane) {
  if (M <= 0) {  // equal, unchanging remainders: fill in index order
    const int c = max(cap, 0);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = low_first ? __shfl_up_sync(0xffffffffu, incl, o)
                              : __shfl_down_sync(0xffffffffu, incl, o);
      if (low_first ? lane >= o : lane + o < 32) incl += t;
    }
    return min(c, max(0, D - (incl - c)));
  }
  int lev = 0, lo = INT_MAX, hi = INT_MIN;
  if (cap > 0) {
    lev = static_cast<int>(sdiv_floor_small(b0 + (M >> 1), M));
    lo = lev - cap + 1;
    hi = lev;
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lo > hi) return 0;
  auto count_ge = [&](int l) {
    const int c = cap > 0 ? max(0, min(cap, lev - l + 1)) : 0;
    return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
  };
  int L = lo, L_hi = hi;
  while (L < L_hi) {
    const int mid = L + (L_hi - L + 1) / 2;
    if (count_ge(mid) >= D) L = mid; else L_hi = mid - 1;
  }
  const int d_at_L = D - count_ge(L + 1);
  int t = cap > 0 ? max(0, min(cap, lev - L)) : 0;
  const bool member = cap > 0 && lev - cap < L && L <= lev;
  if (d_at_L > 0 && __any_sync(0xffffffffu, member)) {
    const int64_t v = b0 - static_cast<int64_t>(lev - L) * M;
    int rank = 0;
    for (int j = 0; j < 32; ++j) {
      const int64_t vj = shfl64(v, j);
      const bool mj = __shfl_sync(0xffffffffu, member, j);
      rank += (mj && j != lane && (vj > v || (vj == v && (low_first ? j < lane : j > lane))))
                  ? 1 : 0;
    }
    if (member && rank < d_at_L) ++t;
  }
  return t;
}

// Key design 3 for at most 32 segments (lane s = segment s), in registers: the
// rule of the general path in segment_phase step 5, with the same integers.
template <class SP>
__device__ __forceinline__ void quotas_warp(const SP& p, int ns, int budget,
                                            const int32_t* s_len, const uint64_t* s_mass,
                                            int32_t* s_q, int lane) {
  const bool act = lane < ns;
  const int len = act ? s_len[lane] : 0;
  const uint64_t ms = act ? s_mass[lane] : 0ull;
  int fl = act ? min(p.q_min, len) : 0;
  // sum of the masses (each at most the unit's total, below 2^41): exact from
  // two 32-bit reductions
  const uint64_t Mt =
      (static_cast<uint64_t>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(ms >> 20)))
       << 20) +
      __reduce_add_sync(0xffffffffu, static_cast<unsigned>(ms & 0xfffffu));
  int floor_tot = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(fl)));
  if (floor_tot > budget) {
    // heaviest segments first (ties: lower index) while budget remains
    int64_t before_s = 0;
    for (int j = 0; j < 32; ++j) {
      const uint64_t mj = static_cast<uint64_t>(shfl64(static_cast<int64_t>(ms), j));
      const int fj = __shfl_sync(0xffffffffu, fl, j);
      before_s += (j < ns && (mj > ms || (mj == ms && j < lane))) ? fj : 0;
    }
    const int64_t left = budget - before_s;
    fl = act ? static_cast<int>(left <= 0 ? 0 : (left < fl ? left : fl)) : 0;
    floor_tot = budget;
  }
  const int64_t t_rem = budget - floor_tot;
  int64_t share = 0;
  if (Mt > 0 && act)
    share = static_cast<int64_t>(
        udiv_small(2ull * static_cast<uint64_t>(t_rem) * ms + Mt, 2ull * Mt));
  int q = static_cast<int>(fl + share > len ? len : fl + share);
  const int64_t rem = (static_cast<int64_t>(fl) * static_cast<int64_t>(Mt) +
                       t_rem * static_cast<int64_t>(ms)) -
                      static_cast<int64_t>(q) * static_cast<int64_t>(Mt);
  const int qtot = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(q)));
  if (qtot < budget) {
    // +1 to the largest remainder among q < L (ties: lower index), in bulk
    q += best_bids_lane(rem, act ? len - q : 0, static_cast<int64_t>(Mt), budget - qtot, true,
                        lane);
  } else if (qtot > budget) {
    // -1 to the smallest remainder among q > q_min (ties: higher index), in bulk
    q -= best_bids_lane(-rem, act ? q - fl : 0, static_cast<int64_t>(Mt), qtot - budget, false,
                        lane);
  }
  if (act) s_q[lane] = q;
  __syncwarp();
}

// Key design 2: C(t) = sum_{u<=t} m_u, b_k = min{t | C(t) >= k*Delta}; segments
// longer than the maximum are split into near-equal parts, short adjacent ones
// merged, masses recounted.  Key design 3: q_i^min = min(q_min, L_i),
// T_rem = T_keep - sum q_i^min, q_i = q_i^min + round(T_rem M_i / sum M),
// clipped to L_i and corrected to the exact budget.
//
// Exactness: the fp32 mass becomes 40-bit fixed point (mu = trunc(m * 2^40),
// exact), prefix sums are uint64, the thresholds are
// tau_k = ceil(fl(fl(k*Delta) * S)) in IEEE double with round-to-nearest and no
// fused operations (evaluated exactly so in integers by ceil_scaled_product),
// the split/merge and quota rules are integer only.  The same definitions with
// the same tie rules give the same bits on any machine and for any NT.
//   * empty raw segments are dropped; merge left to right until >= seg_min,
//     a short tail joins its predecessor; then split L > seg_max into
//     c = ceil(L/seg_max) parts, the first L mod c one longer;
//   * budget = min(T_keep, n); infeasible minimums go to the heaviest segments
//     (ties: lower index); round = half up; correction one unit at a time on the
//     exact remainder (short: largest remainder among q < L, ties lower index;
//     over: smallest remainder among q > q^min, ties higher index).
// `m` points at the unit's first valid slot (n = T - pad of them), in global or
// shared memory.  With `write_out` the segments (absolute starts), lengths,
// quotas and count go to the global arrays, zero past the count.  kSub > 1
// keeps the prefix at kSub sub-ranges of every thread's range too (sm.sub), so
// that the warp's later scans of `m` (long units: in global memory) cover one
// sub-range at most.
template <int NT, int kSub = 1>
__device__ __forceinline__ void segment_phase(const SegParams& p, int u, const float* m, int pad,
                                              int n, const SegSmem& sm, bool write_out) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int32_t* o_start = p.seg_start + static_cast<size_t>(u) * p.S_max;
  int32_t* o_len = p.seg_len + static_cast<size_t>(u) * p.S_max;
  int32_t* o_q = p.quota + static_cast<size_t>(u) * p.S_max;

  if (n <= 0) {
    if (write_out) {
      for (int s = threadIdx.x; s < p.S_max; s += NT) {
        o_start[s] = 0;
        o_len[s] = 0;
        o_q[s] = 0;
      }
      if (threadIdx.x == 0) p.n_seg[u] = 0;
    }
    if (threadIdx.x == 0) *sm.nseg = 0;
    __syncthreads();
    return;
  }

  // ---- 1. prefix sums of the fixed-point mass over contiguous thread ranges
  // (and, with kSub > 1, over kSub sub-ranges of g slots in each)
  const int per = (n + NT - 1) / NT;
  const int g = (per + kSub - 1) / kSub;
  const int lo = min(n, static_cast<int>(threadIdx.x) * per), hi = min(n, lo + per);
  uint64_t local = 0;
  if constexpr (kSub > 1) {
    for (int j = 0; j < kSub; ++j) {
      sm.sub[threadIdx.x * kSub + j] = local;  // relative to the range's start for now
      const int e = min(hi, lo + (j + 1) * g);
      for (int v = min(hi, lo + j * g); v < e; ++v) local += fixed_mass(m[v]);
    }
  } else {
    for (int v = lo; v < hi; ++v) local += fixed_mass(m[v]);
  }
  const uint64_t incl = warp_incl_scan(local);
  if (lane == 31) sm.part[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t run = 0;
    for (int w = 0; w < NT / 32; ++w) {
      const uint64_t t = sm.part[w];
      sm.part[w] = run;
      run += t;
    }
    *sm.total = run;
  }
  __syncthreads();
  const uint64_t before = sm.part[warp] + incl - local;  // prefix before `lo`
  const uint64_t S = *sm.total;
  sm.pre[threadIdx.x] = before;  // C at the start of each thread's range
  if constexpr (kSub > 1) {
#pragma unroll
    for (int j = 0; j < kSub; ++j) sm.sub[threadIdx.x * kSub + j] += before;
  }
  __syncthreads();
  // Steps 2-6 are one short chain per unit: warp 0 runs them alone, with warp
  // barriers only; the other warps are done.
  if (warp != 0) return;

  // ---- 2. cut points: b_k = min{t in [1,n] : C(t) >= tau_k}, lane k: the
  // threshold (the double computation, in integers), then the range (thread
  // range, or sub-range with kSub > 1) whose end first reaches it (a binary
  // search over the range prefixes) and the slot inside that range; n if no
  // prefix reaches it
  constexpr int kRanges = NT * kSub;
  const uint64_t* range_pre = kSub > 1 ? sm.sub : sm.pre;
  for (int k = lane; k < p.K; k += 32) {
    const uint64_t tau =
        ceil_scaled_product(static_cast<uint64_t>(k + 1) * p.delta_m, p.delta_e, S);
    int bk = 1;
    if (tau > 0) {
      int j = 0, j_hi = kRanges - 1;  // the first range j with C(end of j) >= tau (C(n) = S >= tau)
      while (j < j_hi) {
        const int mid = (j + j_hi) >> 1;
        const uint64_t end = mid + 1 < kRanges ? range_pre[mid + 1] : S;
        if (end >= tau) j_hi = mid; else j = mid + 1;
      }
      uint64_t c = range_pre[j];
      const int t_lo = min(n, (j / kSub) * per), t_hi = min(n, t_lo + per);
      int v = min(t_hi, t_lo + (j % kSub) * g);
      const int v_end = kSub > 1 ? min(t_hi, t_lo + (j % kSub + 1) * g) : t_hi;
      for (; v < v_end; ++v) {
        c += fixed_mass(m[v]);
        if (c >= tau) break;
      }
      bk = min(v + 1, n);
    }
    sm.b[k] = bk;
  }
  __syncwarp();

  // ---- 3. raw segments, merge, split (at most K+1 raw segments)
  int32_t* s_start = sm.start;
  int32_t* s_len = sm.len;
  // (each branch condition is uniform; warp 0 runs the shuffles whole)
  const bool ablation = p.global_topk || p.seg_fixed > 0;
  if (ablation && lane == 0) {
    // ablations: one segment over everything, or fixed-length segments whose
    // shorter tail joins the segment before it
    int ns_ab = 1;
    if (p.global_topk) {
      s_start[0] = 0;
      s_len[0] = n;
    } else {
      ns_ab = max(1, n / p.seg_fixed);
      for (int s = 0; s < ns_ab; ++s) {
        s_start[s] = s * p.seg_fixed;
        s_len[s] = (s + 1 < ns_ab) ? p.seg_fixed : n - s * p.seg_fixed;
      }
    }
    *sm.nseg = ns_ab;
  } else if (!ablation && p.K < 32) {
    // at most 32 raw segments: the same three rules, across warp 0.
    // Raw segments: the ends b_0 <= ... <= b_{K-1}, n; a segment where the end
    // grows (the empty ones dropped).
    const int e = lane < p.K ? sm.b[lane] : (lane == p.K ? n : INT_MAX);
    const int e_up = __shfl_up_sync(0xffffffffu, e, 1);
    const int pe = lane == 0 ? 0 : e_up;
    const bool raw = lane <= p.K && e > pe;
    const uint32_t rb = __ballot_sync(0xffffffffu, raw);
    const int n_raw = __popc(rb);
    if (raw) {
      const int r = __popc(rb & ((1u << lane) - 1u));
      s_start[r] = pe;
      s_len[r] = e - pe;
    }
    __syncwarp();
    const int rs = lane < n_raw ? s_start[lane] : 0;
    const int rl = lane < n_raw ? s_len[lane] : 0;
    // merge left to right until >= seg_min (every lane follows the same
    // sequence); bit r of gs: raw segment r starts a merged one
    uint32_t gs = 1u;
    int cur_l = __shfl_sync(0xffffffffu, rl, 0);
    for (int r = 1; r < n_raw; ++r) {
      const int lr = __shfl_sync(0xffffffffu, rl, r);
      if (cur_l < p.seg_min) {
        cur_l += lr;
      } else {
        gs |= 1u << r;
        cur_l = lr;
      }
    }
    const int last = 31 - __clz(gs);
    if (cur_l < p.seg_min && last > 0) gs &= ~(1u << last);  // a short tail joins its predecessor
    // merged segment of this lane (if it starts one): to the next start or n
    const bool head = lane < n_raw && ((gs >> lane) & 1u);
    const uint32_t after = lane == 31 ? 0u : (gs & ~((2u << lane) - 1u));
    const int end = after ? s_start[__ffs(after) - 1] : n;
    const int L = end - rs;
    // split L > seg_max into c = ceil(L/seg_max) parts, the first L mod c one longer
    const int c = head ? (L <= p.seg_max ? 1 : (L + p.seg_max - 1) / p.seg_max) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    __syncwarp();  // every raw start read before the merged ones overwrite them
    if (head) {
      const int base = L / c, extra = L % c;
      for (int j = 0; j < c; ++j) {
        s_start[incl - c + j] = rs + j * base + min(j, extra);
        s_len[incl - c + j] = base + (j < extra ? 1 : 0);
      }
    }
    if (lane == 31) *sm.nseg = incl;
  } else if (!ablation && p.K >= 32 && lane == 0) {
    // raw segments into s_start/s_len (drop empty)
    int n_raw = 0, prev = 0;
    for (int k = 0; k < p.K; ++k) {
      const int bk = sm.b[k];
      if (bk > prev) {
        s_start[n_raw] = prev;
        s_len[n_raw] = bk - prev;
        ++n_raw;
        prev = bk;
      }
    }
    if (prev < n) {
      s_start[n_raw] = prev;
      s_len[n_raw] = n - prev;
      ++n_raw;
    }
    // merge in place
    int n_mer = 0;
    int cur_s = s_start[0], cur_l = s_len[0];
    for (int r = 1; r < n_raw; ++r) {
      if (cur_l < p.seg_min) {
        cur_l += s_len[r];
      } else {
        s_start[n_mer] = cur_s;
        s_len[n_mer] = cur_l;
        ++n_mer;
        cur_s = s_start[r];
        cur_l = s_len[r];
      }
    }
    if (cur_l < p.seg_min && n_mer > 0) {
      s_len[n_mer - 1] += cur_l;
    } else {
      s_start[n_mer] = cur_s;
      s_len[n_mer] = cur_l;
      ++n_mer;
    }
    // split, back to front so that the merged list is read before overwritten
    int n_out = 0;
    for (int r = 0; r < n_mer; ++r) {
      const int L = s_len[r];
      n_out += (L <= p.seg_max) ? 1 : (L + p.seg_max - 1) / p.seg_max;
    }
    int w = n_out;
    for (int r = n_mer - 1; r >= 0; --r) {
      const int L = s_len[r], st = s_start[r];
      if (L <= p.seg_max) {
        --w;
        s_start[w] = st;
        s_len[w] = L;
        continue;
      }
      const int c = (L + p.seg_max - 1) / p.seg_max;
      const int base = L / c, extra = L % c;
      // part j starts at st + j*base + min(j, extra)
      for (int j = c - 1; j >= 0; --j) {
        --w;
        s_start[w] = st + j * base + min(j, extra);
        s_len[w] = base + (j < extra ? 1 : 0);
      }
    }
    *sm.nseg = n_out;
  }
  __syncwarp();
  const int ns = *sm.nseg;

  // ---- 4. segment masses: M_s = C(end) - C(start), with C(pos) the fixed-point
  // mass of the first pos valid slots from the range prefixes of step 1 (the
  // same integer sums, in another order: exact).  The segments tile [0, n), so
  // a segment ends where the next starts: C is taken once per start.
  auto prefix_at = [&](int pos) -> uint64_t {
    if (pos >= n) return S;
    const int t = pos / per;
    int v = t * per;
    uint64_t c;
    if constexpr (kSub > 1) {
      const int j = (pos - v) / g;
      c = sm.sub[t * kSub + j];
      v += j * g;
    } else {
      c = sm.pre[t];
    }
    for (; v < pos; ++v) c += fixed_mass(m[v]);
    return c;
  };
  if (p.quota_by_len) {  // ablation: lengths for masses
    for (int s = lane; s < ns; s += 32) sm.mass[s] = static_cast<uint64_t>(s_len[s]);
  } else if (ns <= 32) {  // one segment per lane
    const uint64_t c0 = lane < ns ? prefix_at(s_start[lane]) : 0ull;
    const uint64_t c1 = static_cast<uint64_t>(shfl64_down(static_cast<int64_t>(c0)));
    if (lane < ns) sm.mass[lane] = (lane + 1 < ns ? c1 : S) - c0;
  } else {  // C at every start into rem (free until step 5), then the differences
    for (int s = lane; s < ns; s += 32) sm.rem[s] = static_cast<int64_t>(prefix_at(s_start[s]));
    __syncwarp();
    for (int s = lane; s < ns; s += 32)
      sm.mass[s] = (s + 1 < ns ? static_cast<uint64_t>(sm.rem[s + 1]) : S) -
                   static_cast<uint64_t>(sm.rem[s]);
  }
  __syncwarp();

  // ---- 5. quotas
  if (ns <= 32) {
    quotas_warp(p, ns, min(p.budget, n), s_len, sm.mass, sm.q, lane);
  } else {
    int32_t* s_q = sm.q;
    int32_t* s_floor = sm.floor;
    const int budget = min(p.budget, n);
    uint64_t Mt = 0;
    int64_t floor_tot = 0;
    for (int s = lane; s < ns; s += 32) {
      s_floor[s] = min(p.q_min, s_len[s]);
      Mt += sm.mass[s];
      floor_tot += s_floor[s];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Mt += __shfl_xor_sync(0xffffffffu, Mt, o);
      floor_tot += __shfl_xor_sync(0xffffffffu, floor_tot, o);
    }
    __syncwarp();
    if (floor_tot > budget) {
      // heaviest segments first (ties: lower index) while budget remains
      for (int s = lane; s < ns; s += 32) {
        int64_t before_s = 0;
        for (int j = 0; j < ns; ++j) {
          const bool ahead = (sm.mass[j] > sm.mass[s]) || (sm.mass[j] == sm.mass[s] && j < s);
          if (ahead) before_s += s_floor[j];
        }
        const int64_t left = budget - before_s;
        s_q[s] = static_cast<int32_t>(left <= 0 ? 0 : (left < s_floor[s] ? left : s_floor[s]));
      }
      __syncwarp();
      for (int s = lane; s < ns; s += 32) s_floor[s] = s_q[s];
      __syncwarp();
      floor_tot = budget;
    }
    const int64_t t_rem = budget - floor_tot;
    int64_t qtot = 0;
    for (int s = lane; s < ns; s += 32) {
      int64_t share = 0;
      if (Mt > 0) {
        const uint64_t num = 2ull * static_cast<uint64_t>(t_rem) * sm.mass[s] + Mt;
        share = static_cast<int64_t>(udiv_small(num, 2ull * Mt));
      }
      int64_t q = s_floor[s] + share;
      if (q > s_len[s]) q = s_len[s];
      s_q[s] = static_cast<int32_t>(q);
      sm.rem[s] = (static_cast<int64_t>(s_floor[s]) * static_cast<int64_t>(Mt) +
                   t_rem * static_cast<int64_t>(sm.mass[s])) -
                  q * static_cast<int64_t>(Mt);
      qtot += q;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qtot += __shfl_xor_sync(0xffffffffu, qtot, o);
    __syncwarp();
    // correction to the exact budget (bulk form of the one-unit-at-a-time rule)
    if (qtot < budget) {
      // segment s bids rem_s - k*Mt for k < L_s - q_s; take the D largest,
      // ties between segments -> lower index first.
      take_best_bids(sm.rem, s_len, s_q, ns, static_cast<int64_t>(Mt),
                     static_cast<int>(budget - qtot),
                     /*negate=*/false, /*low_first=*/true, lane,
                     reinterpret_cast<int32_t*>(sm.mass));
    } else if (qtot > budget) {
      // segment s bids rem_s + k*Mt for k < q_s - floor_s; take the D smallest,
      // ties -> higher index first (the negated bids, largest first).
      take_best_bids(sm.rem, s_floor, s_q, ns, static_cast<int64_t>(Mt),
                     static_cast<int>(qtot - budget),
                     /*negate=*/true, /*low_first=*/false, lane,
                     reinterpret_cast<int32_t*>(sm.mass));
    }
  }
  __syncwarp();

  // ---- 6. outputs (absolute starts), zero past n_seg
  if (write_out) {
    for (int s = lane; s < p.S_max; s += 32) {
      if (s < ns) {
        o_start[s] = pad + s_start[s];
        o_len[s] = s_len[s];
        o_q[s] = sm.q[s];
      } else {
        o_start[s] = 0;
        o_len[s] = 0;
        o_q[s] = 0;
      }
    }
    if (lane == 0) p.n_seg[u] = ns;
  }
}

// ---------------------------------------------------------------- step 4: selection

// slots per thread up to which the excess search keeps keys in registers
constexpr int kRegPer = 8;
constexpr int kKeyPer = 16;  // longer units: gathered pick keys per thread held in registers

enum : uint8_t { kOut = 0, kMust = 1, kPick = 2 };

struct SelParams {
  int T, B, H, S_max, budget, n_sink, n_recent;
  const float* score;
  const int32_t* pad;
  const int32_t* seg_start;
  const int32_t* seg_len;
  const int32_t* quota;
  const int32_t* n_seg;
  int32_t* kept_idx;
  int32_t* n_kept;
};

// Scores are compared through an order-preserving 32-bit key; kLdg reads them
// from global memory through the read-only path, otherwise with plain loads
// (shared memory).
template <bool kLdg>
__device__ __forceinline__ uint32_t score_key(const float* sc, int v) {
  if constexpr (kLdg) return float_order_key(__ldg(sc + v));
  return float_order_key(sc[v]);
}

// One warp: mark the `want` best candidates (flag == kOut) of [st, en).
template <bool kLdg>
__device__ __forceinline__ void pick_segment(const float* sc, uint8_t* flag, int st, int en,
                                             int want, int lane) {
  // largest x with #(candidates with key >= x) >= want: the want-th largest key
  uint32_t x = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t t = x | (1u << bit);
    unsigned cnt = 0;
    for (int v = st + lane; v < en; v += 32)
      cnt += (flag[v] == kOut && score_key<kLdg>(sc, v) >= t) ? 1u : 0u;
    if (static_cast<int>(__reduce_add_sync(0xffffffffu, cnt)) >= want) x = t;
  }
  unsigned gt = 0;
  for (int v = st + lane; v < en; v += 32)
    gt += (flag[v] == kOut && score_key<kLdg>(sc, v) > x) ? 1u : 0u;
  int ties_left = want - static_cast<int>(__reduce_add_sync(0xffffffffu, gt));
  const uint32_t below = (1u << lane) - 1u;
  for (int base = st; base < en; base += 32) {
    const int v = base + lane;
    const bool cand = v < en && flag[v] == kOut;
    const uint32_t k = cand ? score_key<kLdg>(sc, v) : 0u;
    const bool tie = cand && k == x;
    const uint32_t ball = __ballot_sync(0xffffffffu, tie);
    const bool take = (cand && k > x) ||
                      (tie && static_cast<int>(__popc(ball & below)) < ties_left);
    ties_left -= __popc(ball);
    __syncwarp();
    if (take) flag[v] = kPick;
  }
}

// As pick_segment for segments of at most 256 slots (8 per lane), with the
// want-th largest candidate key found by a most-significant-digit radix
// select instead of 32 one-bit steps: the bits above the highest bit in which
// the candidates' smallest and largest keys differ are common to all of them;
// below it, each pass counts the candidates that share the bits fixed so far
// by their next 8-bit digit (a 256-bin histogram in this warp's `hist`, 16-byte
// aligned) and fixes the digit at which the count from the top reaches the
// rank still wanted.  The key found, and so every pick, is the one-bit
// search's.
template <bool kLdg>
__device__ __forceinline__ void pick_segment_radix(const float* sc, uint8_t* flag, int st,
                                                   int en, int want, int lane, int* hist) {
  constexpr int PER = 8;
  uint32_t key[PER];
  bool cand[PER];
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int v = st + lane + 32 * i;
    cand[i] = v < en && flag[v] == kOut;
    key[i] = cand[i] ? score_key<kLdg>(sc, v) : 0u;
    kmin = cand[i] ? min(kmin, key[i]) : kmin;
    kmax = cand[i] ? max(kmax, key[i]) : kmax;
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  int top = (kmin >= kmax) ? 0 : 32 - __clz(kmin ^ kmax);  // bits still open: [0, top)
  uint32_t x = top >= 32 ? 0u : (kmax & (0xffffffffu << top));
  int need = want;  // rank, from the top, among the candidates sharing x's fixed bits
  int4* h4 = reinterpret_cast<int4*>(hist);
  while (top > 0) {  // warp-uniform
    const int shift = top > 8 ? top - 8 : 0;
    const uint32_t fixed = top >= 32 ? 0u : (0xffffffffu << top);
    h4[2 * lane] = make_int4(0, 0, 0, 0);
    h4[2 * lane + 1] = make_int4(0, 0, 0, 0);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (cand[i] && (key[i] & fixed) == x) atomicAdd(&hist[(key[i] >> shift) & 255u], 1);
    __syncwarp();
    // lane L takes bins 255-8L down to 248-8L
    const int4 hi4 = h4[2 * (31 - lane) + 1], lo4 = h4[2 * (31 - lane)];
    const int c[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};
    int s8 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s8 += c[j];
    int incl = s8;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - s8, digit = 0, before = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool hit = run < need && run + c[j] >= need;
      digit = hit ? 255 - 8 * lane - j : digit;
      before = hit ? run : before;
      run += c[j];
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, incl - s8 < need && need <= incl)) - 1;
    digit = __shfl_sync(0xffffffffu, digit, src);
    before = __shfl_sync(0xffffffffu, before, src);
    need -= before;
    x |= static_cast<uint32_t>(digit) << shift;
    top = shift;
    __syncwarp();  // the histogram is cleared again by the next pass
  }
  unsigned gt = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) gt += (cand[i] && key[i] > x) ? 1u : 0u;
  int ties_left = want - static_cast<int>(__reduce_add_sync(0xffffffffu, gt));
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < PER; ++i) {  // 32-slot groups in slot order
    const bool tie = cand[i] && key[i] == x;
    const uint32_t ball = __ballot_sync(0xffffffffu, tie);
    const bool take = (cand[i] && key[i] > x) ||
                      (tie && static_cast<int>(__popc(ball & below)) < ties_left);
    ties_left -= __popc(ball);
    if (take) flag[st + lane + 32 * i] = kPick;
  }
  __syncwarp();
}

// The k-th smallest (1-based, k <= n) of key[0, n) in shared memory, by all NT
// threads of the CTA (barriers inside): a most-significant-digit radix select
// over four 8-bit digits.  Each pass counts the keys that share the digits
// fixed so far by their next digit (a 256-bin histogram in `hist`), and one
// warp fixes the digit at which the count from the bottom reaches the rank
// still wanted; hist[256], hist[257] pass the digit and the count below it to
// every thread.
template <int NT>
__device__ __forceinline__ uint32_t cta_kth_smallest(const uint32_t* key, int n, int k,
                                                     int* hist) {
  uint32_t x = 0;
  int need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
    __syncthreads();  // (also: every thread has read the last pass's digit)
    const uint32_t above = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
    for (int j = threadIdx.x; j < n; j += NT) {
      const uint32_t kj = key[j];
      if ((kj & above) == x) atomicAdd(&hist[(kj >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      // lane L takes bins 8L .. 8L+7, ascending
      const int4 a = reinterpret_cast<const int4*>(hist)[2 * lane];
      const int4 b = reinterpret_cast<const int4*>(hist)[2 * lane + 1];
      const int c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      int s8 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) s8 += c[j];
      int incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int run = incl - s8, digit = 0, below = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool hit = run < need && run + c[j] >= need;
        digit = hit ? 8 * lane + j : digit;
        below = hit ? run : below;
        run += c[j];
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, incl - s8 < need && need <= incl)) - 1;
      digit = __shfl_sync(0xffffffffu, digit, src);
      below = __shfl_sync(0xffffffffu, below, src);
      if (lane == 0) {
        hist[256] = digit;
        hist[257] = below;
      }
    }
    __syncthreads();
    x |= static_cast<uint32_t>(hist[256]) << shift;
    need -= hist[257];
  }
  return x;
}

// Where the selection reads the unit's segments: the global arrays written by
// segment_phase (absolute starts) or its shared arrays (valid offsets).
struct SegsGlobal {
  const int32_t* start;
  const int32_t* len;
  const int32_t* quota;
  int pad;
  __device__ int st(int s) const { return start[s] - pad; }
  __device__ int L(int s) const { return len[s]; }
  __device__ int q(int s) const { return quota[s]; }
};
struct SegsShared {
  const int32_t* start;
  const int32_t* len;
  const int32_t* quota;
  __device__ int st(int s) const { return start[s]; }
  __device__ int L(int s) const { return len[s]; }
  __device__ int q(int s) const { return quota[s]; }
};

// Shared memory of the selection: start and want hold ns entries, flag n, key
// the budget (units with more than kRegPer * NT slots only), hist 256 per warp;
// red, red2 and scan NT/32, 2*NT/32 and NT/32.
struct SelSmem {
  int32_t* start;
  int32_t* want;
  uint8_t* flag;
  uint32_t* key;
  int* hist;  // [NT/32][256], 16-byte aligned: one radix histogram per warp
  int* xhist;  // [256 + 4], 16-byte aligned: the excess search of 1024-thread CTAs
  int* red;
  int* red2;
  int* scan;
};

// Key design 3: must-keep = 4 sinks and the recent suffix, inserted first; if
// the budget left is negative the suffix is shortened, sinks protected (the
// worked example counts the must-keep start and end inside the first and last
// segments' quotas).  Key design 4: top-q_i inside each segment on the base
// score, union with the must-keep set, over budget -> drop low-score
// non-must-keep picks; the kept indices are sorted.
// Rules (shared with any exact implementation of the same reading):
//   * B = min(T_keep, n); n_s = min(n_sink, B); n_r = min(n_recent, B - n_s);
//   * segment i picks max(0, q_i - |MK in i|) of its non-must-keep slots;
//   * order: score descending, ties -> lower slot; removal of the excess picks
//     in the exact reverse order (score ascending, ties -> higher slot).
// Each warp takes whole segments: a radix select (segments of up to 256 slots)
// or a bitwise search finds the want-th largest key among the segment's
// candidates, then one ordered ballot pass takes the ties at that key lowest
// slot first.  The global excess is removed the same
// way across the CTA (bitwise search for the excess-th smallest pick key, ties
// highest slot first).  `sc` points at the unit's first valid slot.  The
// selection compares keys only, so the result is the same for any NT.
template <int NT, bool kLdg, class Segs>
__device__ __forceinline__ void select_phase(const SelParams& p, int u, const float* sc, int pad,
                                             int n, int ns, const Segs& segs,
                                             const SelSmem& sm) {
  constexpr int kWarps = NT / 32;
  int32_t* out = p.kept_idx + static_cast<size_t>(u) * p.budget;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  uint8_t* flag = sm.flag;

  const int Bk = min(p.budget, max(n, 0));
  const int n_s = min(p.n_sink, Bk);
  const int n_r = min(p.n_recent, Bk - n_s);

  // segment starts (valid offsets) and picks wanted per segment
  int want_sum = 0;
  for (int s = threadIdx.x; s < ns; s += NT) {
    const int st = min(max(segs.st(s), 0), n);
    const int L = segs.L(s);
    const int q = segs.q(s);
    const int mk = max(0, min(st + L, n_s) - st) + max(0, st + L - max(st, n - n_r));
    const int want = max(0, min(q - mk, L - mk));
    sm.start[s] = st;
    sm.want[s] = want;
    want_sum += want;
  }
  for (int v = threadIdx.x; v < n; v += NT)
    flag[v] = (v < n_s || v >= n - n_r) ? kMust : kOut;
  const int total_picks = block_count<NT>(want_sum, sm.red);  // (also orders the writes above)

  // segment-local picks, one warp per segment
  for (int s = warp; s < ns; s += kWarps) {
    const int st = sm.start[s];
    const int en = (s + 1 < ns) ? max(st, sm.start[s + 1]) : n;
    const int want = sm.want[s];
    if (want <= 0) continue;
    // a quota that covers the whole segment takes every candidate: no search
    const int mk = max(0, min(en, n_s) - st) + max(0, en - max(st, n - n_r));
    if (want >= en - st - mk) {
      for (int v = st + lane; v < en; v += 32)
        if (flag[v] == kOut) flag[v] = kPick;
      __syncwarp();
      continue;
    }
    if (en - st <= 32 * 8)
      pick_segment_radix<kLdg>(sc, flag, st, en, want, lane, sm.hist + 256 * warp);
    else
      pick_segment<kLdg>(sc, flag, st, en, want, lane);
  }
  __syncthreads();

  // over budget: drop the `excess` worst picks (score ascending, ties: higher slot)
  const int excess = n_s + n_r + total_picks - Bk;
  const int per = (n + NT - 1) / NT;
  const int lo = min(n, static_cast<int>(threadIdx.x) * per);
  const int hi = min(n, lo + per);
  if (excess > 0) {
    // x = the excess-th smallest pick key: largest x with #(pick key < x) < excess
    uint32_t x = 0;
    // CTA-uniform: every thread takes the same branch (barriers inside)
    if (NT < 1024 && per <= kRegPer) {
      uint32_t key[kRegPer];
      bool pk[kRegPer];
#pragma unroll
      for (int i = 0; i < kRegPer; ++i) {
        const int v = lo + i;
        pk[i] = v < hi && flag[v] == kPick;
        key[i] = pk[i] ? score_key<kLdg>(sc, v) : 0u;
      }
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t t = x | (1u << bit);
        unsigned cnt = 0;
#pragma unroll
        for (int i = 0; i < kRegPer; ++i) cnt += (pk[i] && key[i] < t) ? 1u : 0u;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        // alternate buffers: one barrier per step
        int* rb = sm.red2 + (bit & 1) * kWarps;
        if (lane == 0) rb[warp] = static_cast<int>(cnt);
        __syncthreads();
        int total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) total += rb[w];
        if (total < excess) x = t;
      }
    } else {
      // long units: the picks' keys (at most the budget) gathered once into
      // shared memory in slot order, then searched there -- in registers when
      // there are at most kKeyPer per thread -- instead of every step
      // re-reading all of this thread's slots
      int cnt = 0;
      for (int v = lo; v < hi; ++v) cnt += flag[v] == kPick ? 1 : 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) sm.scan[warp] = incl;
      __syncthreads();
      int pos = incl - cnt;
      for (int w = 0; w < warp; ++w) pos += sm.scan[w];
      int n_pick = 0;
      for (int w = 0; w < kWarps; ++w) n_pick += sm.scan[w];
      for (int v = lo; v < hi; ++v)
        if (flag[v] == kPick) sm.key[pos++] = score_key<kLdg>(sc, v);
      __syncthreads();
      if constexpr (NT >= 1024) {
        // many warps: four radix passes instead of 32 bitwise steps, each with
        // a barrier across the CTA
        x = cta_kth_smallest<NT>(sm.key, n_pick, excess, sm.xhist);
      } else if (n_pick <= kKeyPer * NT) {  // CTA-uniform
        uint32_t key[kKeyPer];
#pragma unroll
        for (int i = 0; i < kKeyPer; ++i) {
          const int j = threadIdx.x + i * NT;
          key[i] = j < n_pick ? sm.key[j] : 0xffffffffu;  // never below a threshold
        }
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t t = x | (1u << bit);
          unsigned c2 = 0;
#pragma unroll
          for (int i = 0; i < kKeyPer; ++i) c2 += key[i] < t ? 1u : 0u;
          c2 = __reduce_add_sync(0xffffffffu, c2);
          int* rb = sm.red2 + (bit & 1) * kWarps;
          if (lane == 0) rb[warp] = static_cast<int>(c2);
          __syncthreads();
          int total = 0;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) total += rb[w];
          if (total < excess) x = t;
        }
      } else {
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t t = x | (1u << bit);
          int c2 = 0;
          for (int j = threadIdx.x; j < n_pick; j += NT) c2 += sm.key[j] < t ? 1 : 0;
          if (block_count<NT>(c2, sm.red) < excess) x = t;
        }
      }
      __syncthreads();  // scan is reused below
    }
    int lt = 0, ties = 0;
    for (int v = lo; v < hi; ++v) {
      if (flag[v] != kPick) continue;
      const uint32_t k = score_key<kLdg>(sc, v);
      lt += (k < x) ? 1 : 0;
      ties += (k == x) ? 1 : 0;
    }
    const int drop_ties = excess - block_count<NT>(lt, sm.red);
    // ties above this thread's range (higher slots are dropped first)
    int incl = ties;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += t;
    }
    if (lane == 0) sm.scan[warp] = incl;
    __syncthreads();
    int after = incl - ties;  // ties in higher lanes of this warp
    for (int w = warp + 1; w < kWarps; ++w) after += sm.scan[w];
    for (int v = hi - 1; v >= lo; --v) {
      if (flag[v] != kPick) continue;
      const uint32_t k = score_key<kLdg>(sc, v);
      if (k < x) {
        flag[v] = kOut;
      } else if (k == x) {
        if (after < drop_ties) flag[v] = kOut;
        ++after;
      }
    }
    __syncthreads();
  }

  if constexpr (NT >= 1024) {
    // ordered write-out, coalesced: each warp takes a run of whole 32-slot
    // groups, and a ballot places its kept slots, consecutive lanes at
    // consecutive positions (one thread's run of positions would scatter a
    // warp's stores over 32 places)
    const int gpw = ((n + 31) / 32 + kWarps - 1) / kWarps;  // groups per warp
    const int w_lo = min(n, warp * gpw * 32), w_hi = min(n, w_lo + gpw * 32);
    int cnt = 0;
    for (int b = w_lo; b < w_hi; b += 32) {
      const int v = b + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, v < w_hi && flag[v] != kOut));
    }
    __syncthreads();  // scan may still be read by the excess pass
    if (lane == 0) sm.scan[warp] = cnt;
    __syncthreads();
    int pos = 0, total = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = sm.scan[w];
      pos += w < warp ? c : 0;
      total += c;
    }
    const uint32_t lower = (1u << lane) - 1u;
    for (int b = w_lo; b < w_hi; b += 32) {
      const int v = b + lane;
      const bool keep = v < w_hi && flag[v] != kOut;
      const uint32_t ball = __ballot_sync(0xffffffffu, keep);
      const int at = pos + __popc(ball & lower);
      if (keep && at < p.budget) out[at] = pad + v;
      pos += __popc(ball);
    }
    for (int r = total + threadIdx.x; r < p.budget; r += NT) out[r] = -1;
    if (threadIdx.x == 0) p.n_kept[u] = min(total, p.budget);
  } else {
    // ordered write-out: contiguous ranges per thread + block exclusive scan
    int cnt = 0;
    for (int v = lo; v < hi; ++v) cnt += flag[v] != kOut ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    __syncthreads();  // scan may still be read by the excess pass
    if (lane == 31) sm.scan[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += sm.scan[w];
    int pos = wbase + incl - cnt;
    for (int v = lo; v < hi; ++v)
      if (flag[v] != kOut && pos < p.budget) out[pos++] = pad + v;
    int total = 0;
    for (int w = 0; w < kWarps; ++w) total += sm.scan[w];
    for (int r = total + threadIdx.x; r < p.budget; r += NT) out[r] = -1;
    if (threadIdx.x == 0) p.n_kept[u] = min(total, p.budget);
  }
}

}  // namespace unit
}  // namespace kvc
